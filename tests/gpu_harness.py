"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
CUDA library through its C ABI, bring results back, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import workloads as WL
from combine_route_scan_gb300 import moe as M

TORCH_DT = {WL.X_INT32: torch.int32, WL.X_FP16: torch.float16, WL.X_BF16: torch.bfloat16}


def to_dev(a: np.ndarray, kind: str = "") -> torch.Tensor:
    if a is None:
        return None
    if kind == WL.X_BF16 or (a.dtype == np.uint16 and kind == "bf16"):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    if t is None:
        return None
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def device_inputs(wl: WL.Workload, inp: dict) -> dict:
    return {
        "x": to_dev(inp["x"], wl.x_dtype),
        "expert_ids": to_dev(inp["expert_ids"]),
        "active_mask": to_dev(inp.get("active_mask")),
        "expert_scales": to_dev(inp["expert_scales"]),
        "quant_scales": to_dev(inp.get("quant_scales")),
    }


def make_cfg(wl: WL.Workload, **kw) -> M.MoeConfig:
    q = kw.pop("quant_mode", wl.quant_mode)
    return M.config(wl.ep_world_size, wl.bs, wl.h, wl.topk, wl.moe_expert_num, TORCH_DT[wl.x_dtype],
                    zero_expert_num=wl.zero_expert_num, copy_expert_num=wl.copy_expert_num,
                    quant_mode=q, mask_kind=wl.mask_kind, expand_dtype=wl.y_dtype if q else "",
                    scales_kind=wl.scales_kind if q else 0, **kw)


def gpu_dispatch(wl: WL.Workload, dev: dict, plane_policy: int = M.PLANE_RULE,
                 bulk_min_bytes: int = M.BULK_MIN_BYTES, ws=None, out=None, check_status=True):
    cfg = make_cfg(wl, plane_policy=plane_policy, bulk_min_bytes=bulk_min_bytes)
    if ws is None:
        ws = M.alloc_workspace(cfg)
    if out is None:
        out = M.alloc_dispatch_outputs(cfg, TORCH_DT[wl.x_dtype], seg_plane=True)
        # poison the outputs so rows the kernels fail to write show up
        for k, t in out.items():
            if t is not None:
                t.view(torch.uint8).fill_(0xA5)
    M.dispatch(cfg, dev["x"], dev["expert_ids"], dev["active_mask"], dev["expert_scales"], out["expand_x"],
               out["dynamic_scales"], out["assist_info"], out["ep_recv_count"], out["expand_scales"],
               out["seg_plane"], ws, scales=dev.get("quant_scales"))
    st = M.get_device_status(ws)
    if check_status:
        assert st == 0, f"device status {M.STATUS.get(st, st)}"
    return out, ws, st


def gpu_combine(wl: WL.Workload, dev: dict, expert_out, assist_info, ep_recv_count, combine_mode=M.COMBINE_GATHER,
                plane_policy: int = M.PLANE_RULE, ws=None, check_status=True, seg_plane=False,
                bulk_min_bytes: int = M.BULK_MIN_BYTES):
    cfg = make_cfg(wl, quant_mode=0, combine_mode=combine_mode, plane_policy=plane_policy,
                   bulk_min_bytes=bulk_min_bytes)
    if ws is None:
        ws = M.alloc_workspace(cfg)
    x_out = torch.empty((wl.ep_world_size, wl.bs, wl.h), dtype=TORCH_DT[wl.x_dtype], device="cuda")
    x_out.view(torch.uint8).fill_(0x5A)
    sp = None
    if seg_plane:
        L = wl.moe_expert_num // wl.ep_world_size
        sp = torch.empty((wl.ep_world_size, L * wl.ep_world_size), dtype=torch.uint8, device="cuda")
    M.combine(cfg, expert_out, assist_info, ep_recv_count, dev["expert_ids"], dev["expert_scales"],
              dev["active_mask"], dev["x"], x_out, sp, ws)
    st = M.get_device_status(ws)
    if check_status:
        assert st == 0, f"device status {M.STATUS.get(st, st)}"
    return x_out, st, sp


def compare_dispatch(wl: WL.Workload, got: dict, ref: dict, plane_ref=None):
    """Bit-exact on every written row, counts, metadata and plane choice."""
    ep = to_host(got["ep_recv_count"])
    assert np.array_equal(ep, ref["ep_recv_count"]), "ep_recv_count"
    ex, ai = to_host(got["expand_x"]), to_host(got["assist_info"])
    es = to_host(got["expand_scales"]) if got.get("expand_scales") is not None else None
    ds = to_host(got["dynamic_scales"]) if got.get("dynamic_scales") is not None else None
    for d in range(wl.ep_world_size):
        n = int(ep[d, -1])
        assert np.array_equal(ai[d, :n], ref["assist_info"][d, :n]), f"assist_info rank {d}"
        assert np.array_equal(ex[d, :n].view(np.uint8), ref["expand_x"][d, :n].view(np.uint8)), f"expand_x rank {d}"
        if es is not None:
            assert np.array_equal(es[d, :n].view(np.uint32), ref["expand_scales"][d, :n].view(np.uint32)), \
                f"expand_scales rank {d}"
        if ds is not None:
            assert np.array_equal(ds[d, :n].view(np.uint8), ref["dynamic_scales"][d, :n].view(np.uint8)), \
                f"dynamic_scales rank {d}"
    if plane_ref is not None and got.get("seg_plane") is not None:
        assert np.array_equal(to_host(got["seg_plane"]), plane_ref), "segment planes"


def float_view(wl: WL.Workload, a: np.ndarray) -> np.ndarray:
    if wl.x_dtype == WL.X_BF16:
        return WL.bf16_bits_to_fp32(a).astype(np.float64)
    return a.astype(np.float64)


def compare_combine(wl: WL.Workload, got: np.ndarray, ref: np.ndarray, tol_rel: float = 1e-3):
    """int32: exact. Floats: max |gpu - oracle| <= tol_rel * max |oracle| (the
    stated tolerance); returns the max abs error."""
    if wl.x_dtype == WL.X_INT32:
        assert np.array_equal(got, ref), "int32 combine must be exact"
        return 0.0
    g, r = float_view(wl, got), float_view(wl, ref)
    scale = max(np.abs(r).max(), 1e-30)
    err = float(np.abs(g - r).max()) if g.size else 0.0
    assert err <= tol_rel * scale, f"max abs err {err} > {tol_rel} * {scale}"
    return err
