"""Python binding of the C ABI in include/moe.h (libcrs_moe.so).

Argument marshalling only: every function takes torch tensors (device memory
owned by the caller), passes their data pointers and the current CUDA stream
to the C entry point of the same name, and raises MoeError on a non-OK status.
All computation happens in the CUDA kernels of the library; there is no CPU
fallback, and loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# CRS_MOE_CHECKED=1 selects the bounds-checked build (build.build(checked=True)),
# CRS_MOE_OBSERVER=1 the flag-observer test build (build.build(observer=True)),
# CRS_MOE_PHASE=1 the phase-time test build (build.build(phase=True))
LIB_PATH = os.path.join(_HERE, "_build", *(["checked"] if os.environ.get("CRS_MOE_CHECKED") == "1" else
                                           ["observer"] if os.environ.get("CRS_MOE_OBSERVER") == "1" else
                                           ["phase"] if os.environ.get("CRS_MOE_PHASE") == "1" else []),
                        "libcrs_moe.so")

MOE_OK = 0
STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "BAD_EXPERT_ID",
          5: "MASK_ORDER", 6: "TIMEOUT", 7: "CUDA", 8: "CAPACITY", 9: "BAD_ASSIST", 10: "OUT_OF_BOUNDS"}

MOE_I32, MOE_F16, MOE_BF16 = 0, 1, 2
DTYPE_CODE = {torch.int32: MOE_I32, torch.float16: MOE_F16, torch.bfloat16: MOE_BF16}
PLANE_RULE, PLANE_STORES_ONLY, PLANE_BULK_ALL = 0, 1, 2
COMBINE_GATHER, COMBINE_TWO_PHASE, COMBINE_PUT_ONLY = 0, 1, 2
Y_DEFAULT, Y_FP8_E4M3, Y_FP8_E5M2, Y_FP4_E2M1 = 0, 1, 2, 3
Y_CODE = {"": Y_DEFAULT, "int8": Y_DEFAULT, "fp8_e4m3": Y_FP8_E4M3, "fp8_e5m2": Y_FP8_E5M2, "fp4_e2m1": Y_FP4_E2M1}
SCALES_NONE, SCALES_SCALAR, SCALES_CHANNEL, SCALES_EXPERT = 0, 1, 2, 3
BULK_MIN_BYTES = 2 * 1024 * 1024

# Every symbol include/moe.h declares.
EXPORTS = ("moe_get_workspace_size", "moe_workspace_init", "moe_dispatch", "moe_combine",
           "moe_dispatch_ffn_combine", "moe_combine_noalloc", "moe_get_device_status", "moe_status_string")
NOALLOC_MAX_PICKS = 262144


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code
        self.name = STATUS.get(code, str(code))


class MoeConfig(ctypes.Structure):
    """moe_config_t."""
    _fields_ = [
        ("ep_world_size", ctypes.c_int32), ("bs", ctypes.c_int32), ("h", ctypes.c_int32),
        ("topk", ctypes.c_int32), ("moe_expert_num", ctypes.c_int32),
        ("zero_expert_num", ctypes.c_int32), ("copy_expert_num", ctypes.c_int32),
        ("const_expert_num", ctypes.c_int32), ("quant_mode", ctypes.c_int32),
        ("mask_kind", ctypes.c_int32), ("x_dtype", ctypes.c_int32),
        ("plane_policy", ctypes.c_int32), ("bulk_min_bytes", ctypes.c_int64),
        ("combine_mode", ctypes.c_int32), ("wait_timeout_us", ctypes.c_int32),
        ("ffn_intermediate", ctypes.c_int32), ("expand_dtype", ctypes.c_int32),
        ("prof_events", ctypes.c_void_p), ("seg_ready", ctypes.c_void_p),
        ("seg_ready_ticket", ctypes.c_uint32), ("scales_kind", ctypes.c_int32),
        ("performance_info", ctypes.c_void_p),
    ]


def config(ep_world_size: int, bs: int, h: int, topk: int, moe_expert_num: int, x_dtype,
           zero_expert_num: int = 0, copy_expert_num: int = 0, quant_mode: int = 0, mask_kind: int = 0,
           plane_policy: int = PLANE_RULE, bulk_min_bytes: int = BULK_MIN_BYTES,
           combine_mode: int = COMBINE_GATHER, wait_timeout_us: int = 2_000_000,
           ffn_intermediate: int = 0, expand_dtype=Y_DEFAULT, scales_kind: int = SCALES_NONE) -> MoeConfig:
    """moe_config_t; expand_dtype is a MOE_Y_* code or one of the names in Y_CODE."""
    dt = DTYPE_CODE[x_dtype] if isinstance(x_dtype, torch.dtype) else int(x_dtype)
    yd = Y_CODE[expand_dtype] if isinstance(expand_dtype, str) else int(expand_dtype)
    return MoeConfig(ep_world_size, bs, h, topk, moe_expert_num, zero_expert_num, copy_expert_num, 0,
                     quant_mode, mask_kind, dt, plane_policy, bulk_min_bytes, combine_mode, wait_timeout_us,
                     ffn_intermediate, yd, None, None, 0, scales_kind, None)


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with combine_route_scan_gb300.build.build() "
                               "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, C = ctypes.c_void_p, ctypes.POINTER(MoeConfig)
        L.moe_get_workspace_size.argtypes = [C, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_int64)]
        L.moe_workspace_init.argtypes = [C, P, ctypes.c_size_t, P]
        L.moe_dispatch.argtypes = [C, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.moe_combine.argtypes = [C, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.moe_dispatch_ffn_combine.argtypes = [C, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.moe_combine_noalloc.argtypes = [C, P, P, P, P, P, P, P, P, P, P]
        L.moe_get_device_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
        L.moe_status_string.argtypes = [ctypes.c_int32]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_launch_count.argtypes = []
        L.moe_launch_count.restype = ctypes.c_uint64
        for f in ("moe_get_workspace_size", "moe_workspace_init", "moe_dispatch", "moe_combine",
                  "moe_dispatch_ffn_combine", "moe_combine_noalloc", "moe_get_device_status"):
            getattr(L, f).restype = ctypes.c_int32
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    """The tensor's device address as an int (ctypes passes it as void*)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(code: int, what: str):
    if code != MOE_OK:
        raise MoeError(code, what)


class ProfEvents:
    """A {start, stop} pair of CUDA events the library records around the main
    kernel of a call (set on a config with ``attach``)."""

    def __init__(self):
        self.start = torch.cuda.Event(enable_timing=True)
        self.stop = torch.cuda.Event(enable_timing=True)
        # torch creates its events on first record; record once so the handles
        # exist (the library's later records replace these)
        self.start.record()
        self.stop.record()
        self._arr = (ctypes.c_void_p * 2)(self.start.cuda_event, self.stop.cuda_event)

    def attach(self, cfg: MoeConfig) -> MoeConfig:
        c = MoeConfig.from_buffer_copy(cfg)
        c.prof_events = ctypes.cast(self._arr, ctypes.c_void_p)
        return c

    def elapsed_ms(self) -> float:
        return self.start.elapsed_time(self.stop)


def with_seg_ready(cfg: MoeConfig, seg_ready: torch.Tensor, ticket: int) -> MoeConfig:
    """A copy of cfg whose dispatch stores `ticket` into seg_ready[d][le*W+s]
    once segment (le, s) of rank d is complete (uint32 CUDA tensor [W, L*W])."""
    c = MoeConfig.from_buffer_copy(cfg)
    c.seg_ready = _ptr(seg_ready)
    c.seg_ready_ticket = ticket
    return c


def with_performance_info(cfg: MoeConfig, perf: torch.Tensor) -> MoeConfig:
    """A copy of cfg whose dispatch adds each rank's communication time (ns)
    to perf (int64 CUDA tensor [W])."""
    c = MoeConfig.from_buffer_copy(cfg)
    c.performance_info = _ptr(perf)
    return c


def workspace_size(cfg: MoeConfig):
    """(workspace bytes, rows per rank A)."""
    n = ctypes.c_size_t(0)
    a = ctypes.c_int64(0)
    _check(lib().moe_get_workspace_size(ctypes.byref(cfg), ctypes.byref(n), ctypes.byref(a)),
           "moe_get_workspace_size")
    return int(n.value), int(a.value)


def workspace_init(cfg: MoeConfig, ws: torch.Tensor, stream=None):
    _check(lib().moe_workspace_init(ctypes.byref(cfg), _ptr(ws), ws.numel() * ws.element_size(),
                                    _stream(stream)), "moe_workspace_init")


def dispatch(cfg: MoeConfig, x, expert_ids, active_mask, expert_scales, expand_x, dynamic_scales,
             assist_info, ep_recv_count, expand_scales=None, seg_plane=None, ws=None, stream=None, scales=None):
    """moe_dispatch; `scales` is the fp32 coefficient / smoothing input that
    cfg.scales_kind describes (None when it is SCALES_NONE)."""
    _check(lib().moe_dispatch(ctypes.byref(cfg), _ptr(x), _ptr(expert_ids), _ptr(active_mask),
                              _ptr(expert_scales), _ptr(scales), _ptr(expand_x), _ptr(dynamic_scales),
                              _ptr(assist_info),
                              _ptr(ep_recv_count), _ptr(expand_scales), _ptr(seg_plane), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "moe_dispatch")


def combine(cfg: MoeConfig, expert_out, assist_info, ep_recv_count, expert_ids, expert_scales, active_mask,
            x, x_out, seg_plane=None, ws=None, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), _ptr(expert_out), _ptr(assist_info), _ptr(ep_recv_count),
                             _ptr(expert_ids), _ptr(expert_scales), _ptr(active_mask), _ptr(x), _ptr(x_out),
                             _ptr(seg_plane), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_combine")


def dispatch_ffn_combine(cfg: MoeConfig, x, expert_ids, active_mask, expert_scales, w_gate, w_up, w_down, x_out,
                         ws=None, stream=None):
    _check(lib().moe_dispatch_ffn_combine(ctypes.byref(cfg), _ptr(x), _ptr(expert_ids), _ptr(active_mask),
                                          _ptr(expert_scales), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                          _ptr(x_out), _ptr(ws), ws.numel() * ws.element_size(),
                                          _stream(stream)), "moe_dispatch_ffn_combine")


def combine_noalloc(cfg: MoeConfig, expert_out, assist_info, ep_recv_count, expert_ids, expert_scales,
                    active_mask, x, x_out, status, stream=None):
    """moe_combine_noalloc: the gather combine for callers that cannot
    allocate; `status` is a one-element int32 CUDA tensor that receives the
    first device-side error."""
    _check(lib().moe_combine_noalloc(ctypes.byref(cfg), _ptr(expert_out), _ptr(assist_info), _ptr(ep_recv_count),
                                     _ptr(expert_ids), _ptr(expert_scales), _ptr(active_mask), _ptr(x),
                                     _ptr(x_out), _ptr(status), _stream(stream)), "moe_combine_noalloc")


def get_device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream; returns and clears the first device-side error."""
    v = ctypes.c_int32(0)
    _check(lib().moe_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(v)), "moe_get_device_status")
    return int(v.value)


def status_string(code: int) -> str:
    return lib().moe_status_string(code).decode()


def launch_count() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(lib().moe_launch_count())


# ------------------------------------------------------------ allocation
# Device memory is torch's job; these helpers only size the tensors the C ABI
# expects.

def alloc_workspace(cfg: MoeConfig, device="cuda", stream=None) -> torch.Tensor:
    n, _ = workspace_size(cfg)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    workspace_init(cfg, ws, stream)
    return ws


def alloc_dispatch_outputs(cfg: MoeConfig, x_dtype: torch.dtype, device="cuda", expand_scales: bool = True,
                           seg_plane: bool = False) -> dict:
    """expand_x is x's type (quant_mode 0), int8 (1, 2) or uint8 codes (3, 4;
    [W, A, h/2] for packed FP4); dynamic_scales [W, A] fp32 (2), [W, A,
    ceil(h/128)] fp32 (3), [W, A, ceil(h/32)] uint8 E8M0 (4), else None."""
    _, A = workspace_size(cfg)
    W, h = cfg.ep_world_size, cfg.h
    L = cfg.moe_expert_num // W
    qm = cfg.quant_mode
    sdt = torch.int32 if x_dtype == torch.int32 else torch.float32
    if qm == 0:
        ex = torch.empty((W, A, h), dtype=x_dtype, device=device)
    elif qm in (1, 2):
        ex = torch.empty((W, A, h), dtype=torch.int8, device=device)
    else:
        ex = torch.empty((W, A, h // 2 if cfg.expand_dtype == Y_FP4_E2M1 else h), dtype=torch.uint8, device=device)
    dyn = None
    if qm == 2:
        dyn = torch.empty((W, A), dtype=torch.float32, device=device)
    elif qm == 3:
        dyn = torch.empty((W, A, (h + 127) // 128), dtype=torch.float32, device=device)
    elif qm == 4:
        dyn = torch.empty((W, A, (h + 31) // 32), dtype=torch.uint8, device=device)
    return {
        "expand_x": ex,
        "dynamic_scales": dyn,
        "assist_info": torch.empty((W, A, 3), dtype=torch.int32, device=device),
        "ep_recv_count": torch.empty((W, L * W), dtype=torch.int32, device=device),
        "expand_scales": torch.empty((W, A), dtype=sdt, device=device) if expand_scales else None,
        "seg_plane": torch.empty((W, L * W), dtype=torch.uint8, device=device) if seg_plane else None,
    }
