"""ctypes wrapper around the C oracle (oracle/moe_oracle.c). Test infrastructure.

Every function takes numpy arrays laid out as workloads.make_inputs returns
them and hands back numpy arrays. Nothing here does any of the method's
arithmetic: it only allocates outputs and calls the C functions.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

X_KIND = {"int32": 0, "float16": 1, "bfloat16": 2}
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
    ]


_lib = None
_lib_path_override = None


def use_library(path: Optional[str]) -> None:
    """Point the wrapper at another build of moe_oracle.c (the mutation tests
    load deliberately broken copies); None goes back to the default build."""
    global _lib, _lib_path_override
    _lib_path_override = path
    _lib = None


def lib():
    global _lib
    if _lib is None:
        path = _lib_path_override or _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        C = ctypes.POINTER(OrcCfg)
        L.orc_check_cfg.argtypes = [C]
        L.orc_capacity.argtypes = [C]
        L.orc_capacity.restype = ctypes.c_int64
        L.orc_dispatch.argtypes = [C, P, P, P, P, P, P, P, P, P]
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
        _lib = L
    return _lib


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what}: status {code} ({STATUS_NAMES.get(code, '?')})")
        self.code = code
        self.name = STATUS_NAMES.get(code, "?")


def make_cfg(wl, bulk_min_bytes: int = DEFAULT_BULK_MIN_BYTES, quant_mode: Optional[int] = None) -> OrcCfg:
    return OrcCfg(wl.ep_world_size, wl.bs, wl.h, wl.topk, wl.moe_expert_num,
                  wl.zero_expert_num, wl.copy_expert_num,
                  wl.quant_mode if quant_mode is None else quant_mode,
                  wl.mask_kind, X_KIND[wl.x_dtype], bulk_min_bytes)


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
    """Run the oracle dispatch. Rows beyond the received count stay zero."""
    cfg = make_cfg(wl)
    W, h, K = wl.ep_world_size, wl.h, wl.topk
    L = wl.moe_expert_num // W
    A = capacity(wl)
    q = wl.quant_mode == 2
    out = {
        "expand_x": np.zeros((W, A, h), dtype=np.int8 if q else _x_np_dtype(wl)),
        "dynamic_scales": np.zeros((W, A), dtype=np.float32) if q else None,
        "assist_info": np.zeros((W, A, 3), dtype=np.int32),
        "ep_recv_count": np.zeros((W, L * W), dtype=np.int32),
        "expand_scales": (np.zeros((W, A), dtype=np.int32 if wl.x_dtype == "int32" else np.float32)
                          if with_expand_scales else None),
    }
    st = lib().orc_dispatch(ctypes.byref(cfg), _p(inp["x"]), _p(inp["expert_ids"]),
                            _p(inp.get("active_mask")), _p(inp["expert_scales"]),
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


def identity_expert(disp: dict) -> np.ndarray:
    """The identity expert of the combine example: its output is expand_x."""
    return disp["expand_x"]
