"""ctypes wrapper around the C oracle (oracle/moe_oracle.c). Test infrastructure.

Every function takes numpy arrays laid out as workloads.make_inputs returns
them and hands back numpy arrays. Nothing here does any of the method's
arithmetic: it only allocates outputs and calls the C functions.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import numpy as np

from . import build as _build

X_KIND = {"int32": 0, "float16": 1, "bfloat16": 2}
Y_KIND = {"": 0, "int8": 0, "fp8_e4m3": 1, "fp8_e5m2": 2, "fp4_e2m1": 3}
DEFAULT_BULK_MIN_BYTES = 2 * 1024 * 1024  # "2MB" in the plane rule, read as 2 MiB

STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 4: "BAD_EXPERT_ID",
                5: "MASK_ORDER", 8: "CAPACITY", 9: "BAD_ASSIST"}


class OrcCfg(ctypes.Structure):
    _fields_ = [
        ("W", ctypes.c_int32), ("bs", ctypes.c_int32), ("h", ctypes.c_int32),
        ("K", ctypes.c_int32), ("E", ctypes.c_int32), ("Z", ctypes.c_int32),
        ("C", ctypes.c_int32), ("quant_mode", ctypes.c_int32),
        ("mask_kind", ctypes.c_int32), ("x_kind", ctypes.c_int32),
        ("bulk_min_bytes", ctypes.c_int64),
        ("y_kind", ctypes.c_int32), ("scales_kind", ctypes.c_int32),
    ]


_lib = None
_lib_path_override = None
_lib_lock = threading.Lock()


def use_library(path: Optional[str]) -> None:
    """Point the wrapper at another build of moe_oracle.c (the mutation tests
    load deliberately broken copies); None goes back to the default build."""
    global _lib, _lib_path_override
    _lib_path_override = path
    _lib = None


def lib():
    global _lib
    if _lib is None:
        with _lib_lock:  # the tests call the oracle from thread pools
            if _lib is None:
                _lib = _load()
    return _lib


def _load():
    path = _lib_path_override or _build.build()
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    C = ctypes.POINTER(OrcCfg)
    L.orc_check_cfg.argtypes = [C]
    L.orc_capacity.argtypes = [C]
    L.orc_capacity.restype = ctypes.c_int64
    L.orc_dispatch.argtypes = [C, P, P, P, P, P, P, P, P, P, P]
    L.orc_combine.argtypes = [C, P, P, P, P, P, P, P, P]
    L.orc_combine_plane.argtypes = [C, P, P]
    L.orc_dispatch_plane.argtypes = [C, P, P]
    L.orc_swiglu_rows.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                  P, P, P, P, P, P]
    L.orc_moe_ffn_tokens.argtypes = [C, ctypes.c_int, ctypes.c_int64, P, P, P, P, P, P, P, P, P]
    L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    L.orc_f32_to_bf16.restype = ctypes.c_uint16
    L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_bf16_to_f32.restype = ctypes.c_float
    L.orc_f32_to_fp16.argtypes = [ctypes.c_float]
    L.orc_f32_to_fp16.restype = ctypes.c_uint16
    L.orc_fp16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_fp16_to_f32.restype = ctypes.c_float
    L.orc_quantize_row.argtypes = [C, P, P]
    L.orc_quantize_row.restype = ctypes.c_float
    L.orc_f32_to_minifloat.argtypes = [ctypes.c_float, ctypes.c_int]
    L.orc_f32_to_minifloat.restype = ctypes.c_uint8
    L.orc_quantize_pick.argtypes = [C, P, ctypes.c_int32, P, P, P]
    return L


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what}: status {code} ({STATUS_NAMES.get(code, '?')})")
        self.code = code
        self.name = STATUS_NAMES.get(code, "?")


def make_cfg(wl, bulk_min_bytes: int = DEFAULT_BULK_MIN_BYTES, quant_mode: Optional[int] = None) -> OrcCfg:
    q = wl.quant_mode if quant_mode is None else quant_mode
    return OrcCfg(wl.ep_world_size, wl.bs, wl.h, wl.topk, wl.moe_expert_num,
                  wl.zero_expert_num, wl.copy_expert_num, q,
                  wl.mask_kind, X_KIND[wl.x_dtype], bulk_min_bytes,
                  Y_KIND[wl.y_dtype] if q else 0, wl.scales_kind if q else 0)


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def capacity(wl) -> int:
    cfg = make_cfg(wl)
    return int(lib().orc_capacity(ctypes.byref(cfg)))


def _x_np_dtype(wl):
    return {"int32": np.int32, "float16": np.float16, "bfloat16": np.uint16}[wl.x_dtype]


def dispatch(wl, inp: dict, with_expand_scales: bool = True, raise_on_error: bool = True) -> dict:
    """Run the oracle dispatch. Rows beyond the received count stay zero.

    expand_x is x's type unquantised, int8 for quantMode 1 and 2, uint8 codes
    (fp8, or two packed fp4 per byte) for quantMode 3 and 4; dynamic_scales is
    [W, A] fp32 (mode 2), [W, A, ceil(h/128)] fp32 (mode 3), [W, A, ceil(h/32)]
    uint8 E8M0 (mode 4), else None."""
    cfg = make_cfg(wl)
    W, h, K = wl.ep_world_size, wl.h, wl.topk
    L = wl.moe_expert_num // W
    A = capacity(wl)
    qm = wl.quant_mode
    if qm == 0:
        ex = np.zeros((W, A, h), dtype=_x_np_dtype(wl))
    elif qm in (1, 2):
        ex = np.zeros((W, A, h), dtype=np.int8)
    else:
        ex = np.zeros((W, A, h // 2 if wl.y_dtype == "fp4_e2m1" else h), dtype=np.uint8)
    dyn = {2: lambda: np.zeros((W, A), dtype=np.float32),
           3: lambda: np.zeros((W, A, (h + 127) // 128), dtype=np.float32),
           4: lambda: np.zeros((W, A, (h + 31) // 32), dtype=np.uint8)}.get(qm, lambda: None)()
    out = {
        "expand_x": ex,
        "dynamic_scales": dyn,
        "assist_info": np.zeros((W, A, 3), dtype=np.int32),
        "ep_recv_count": np.zeros((W, L * W), dtype=np.int32),
        "expand_scales": (np.zeros((W, A), dtype=np.int32 if wl.x_dtype == "int32" else np.float32)
                          if with_expand_scales else None),
    }
    st = lib().orc_dispatch(ctypes.byref(cfg), _p(inp["x"]), _p(inp["expert_ids"]),
                            _p(inp.get("active_mask")), _p(inp["expert_scales"]), _p(inp.get("quant_scales")),
                            _p(out["expand_x"]), _p(out["dynamic_scales"]), _p(out["assist_info"]),
                            _p(out["ep_recv_count"]), _p(out["expand_scales"]))
    out["status"] = int(st)
    if st and raise_on_error:
        raise OracleError(st, "dispatch")
    return out


def combine(wl, expert_out: np.ndarray, assist_info: np.ndarray, ep_recv_count: np.ndarray,
            inp: dict, raise_on_error: bool = True):
    """Run the oracle combine; returns x_out [W, bs, h] (or (x_out, status))."""
    cfg = make_cfg(wl, quant_mode=0)
    x_out = np.zeros((wl.ep_world_size, wl.bs, wl.h), dtype=_x_np_dtype(wl))
    st = lib().orc_combine(ctypes.byref(cfg), _p(expert_out), _p(assist_info), _p(ep_recv_count),
                           _p(inp["expert_ids"]), _p(inp["expert_scales"]),
                           _p(inp.get("active_mask")), _p(inp["x"]), _p(x_out))
    if st and raise_on_error:
        raise OracleError(st, "combine")
    return x_out if raise_on_error else (x_out, int(st))


def dispatch_plane(wl, ep_recv_count: np.ndarray, bulk_min_bytes: int = DEFAULT_BULK_MIN_BYTES) -> np.ndarray:
    cfg = make_cfg(wl, bulk_min_bytes)
    plane = np.zeros(ep_recv_count.shape, dtype=np.uint8)
    st = lib().orc_dispatch_plane(ctypes.byref(cfg), _p(np.ascontiguousarray(ep_recv_count)), _p(plane))
    if st:
        raise OracleError(st, "dispatch_plane")
    return plane


def combine_plane(wl, ep_recv_count: np.ndarray, bulk_min_bytes: int = DEFAULT_BULK_MIN_BYTES) -> np.ndarray:
    cfg = make_cfg(wl, bulk_min_bytes, quant_mode=0)
    plane = np.zeros(ep_recv_count.shape, dtype=np.uint8)
    st = lib().orc_combine_plane(ctypes.byref(cfg), _p(np.ascontiguousarray(ep_recv_count)), _p(plane))
    if st:
        raise OracleError(st, "combine_plane")
    return plane


def swiglu_rows(x_rows: np.ndarray, expert: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray,
                w_down: np.ndarray) -> np.ndarray:
    """fp64 SwiGLU expert FFN of bf16 rows; x_rows [n, h] uint16 bits, expert [n];
    w_gate, w_up [E, I, h], w_down [E, h, I] (out-major)."""
    E, I, h = w_gate.shape
    x_rows = np.ascontiguousarray(x_rows, dtype=np.uint16)
    expert = np.ascontiguousarray(expert, dtype=np.int32)
    n = x_rows.shape[0]
    y = np.zeros((n, h), dtype=np.float64)
    st = lib().orc_swiglu_rows(h, I, E, n, _p(x_rows), _p(expert), _p(w_gate), _p(w_up), _p(w_down), _p(y))
    if st:
        raise OracleError(st, "swiglu_rows")
    return y


def moe_ffn_tokens(wl, inp: dict, tokens: np.ndarray) -> np.ndarray:
    """fp64 dispatch -> SwiGLU expert -> combine for the given flat token indices."""
    cfg = make_cfg(wl, quant_mode=0)
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    out = np.zeros((tokens.shape[0], wl.h), dtype=np.float64)
    st = lib().orc_moe_ffn_tokens(ctypes.byref(cfg), wl.ffn_intermediate, tokens.shape[0], _p(tokens),
                                  _p(inp["x"]), _p(inp["expert_ids"]), _p(inp.get("active_mask")),
                                  _p(inp["expert_scales"]), _p(inp["w_gate"]), _p(inp["w_up"]),
                                  _p(inp["w_down"]), _p(out))
    if st:
        raise OracleError(st, "moe_ffn_tokens")
    return out


def quantize_row(x_row: np.ndarray, x_dtype: str = "float16"):
    """quantMode 2 on one row: returns (q int8 [h], scale float)."""
    from workloads import Workload
    h = x_row.shape[0]
    wl = Workload("q", 2, 1, h, 1, 2, x_dtype, quant_mode=2)
    cfg = make_cfg(wl)
    x_row = np.ascontiguousarray(x_row)
    q = np.zeros(h, dtype=np.int8)
    scale = lib().orc_quantize_row(ctypes.byref(cfg), _p(x_row), _p(q))
    return q, float(scale)


def f32_to_minifloat(values, y_dtype: str) -> np.ndarray:
    """fp32 values -> codes of the small float format (uint8 each)."""
    L = lib()
    k = Y_KIND[y_dtype]
    return np.array([L.orc_f32_to_minifloat(float(v), k) for v in np.asarray(values, dtype=np.float32)],
                    dtype=np.uint8)


def quantize_pick(x_row: np.ndarray, quant_mode: int, x_dtype: str = "bfloat16", y_dtype: str = "",
                  expert: int = 0, quant_scales: Optional[np.ndarray] = None, scales_kind: int = 0,
                  moe_expert_num: int = 2):
    """quantMode 1..4 on one row for a pick of `expert`: returns (q bytes, dyn)."""
    from workloads import Workload
    h = x_row.shape[0]
    wl = Workload("q", 2, 1, h, 1, moe_expert_num, x_dtype, quant_mode=quant_mode, y_dtype=y_dtype,
                  scales_kind=scales_kind)
    cfg = make_cfg(wl)
    x_row = np.ascontiguousarray(x_row)
    q = np.zeros(h // 2 if y_dtype == "fp4_e2m1" and quant_mode == 4 else h, dtype=np.uint8)
    dyn = {1: None, 2: np.zeros(1, dtype=np.float32), 3: np.zeros((h + 127) // 128, dtype=np.float32),
           4: np.zeros((h + 31) // 32, dtype=np.uint8)}[quant_mode]
    qs = None if quant_scales is None else np.ascontiguousarray(quant_scales, dtype=np.float32)
    st = lib().orc_quantize_pick(ctypes.byref(cfg), _p(x_row), int(expert), _p(qs), _p(q), _p(dyn))
    if st:
        raise OracleError(st, "quantize_pick")
    return q, dyn


def identity_expert(disp: dict) -> np.ndarray:
    """The identity expert of the combine example: its output is expand_x."""
    return disp["expand_x"]
