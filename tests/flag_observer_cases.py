"""Cases for the flag-observer test build (run by test_flag_order_gpu.py in a
child process with CRS_MOE_OBSERVER=1; collected only when named on the
command line).

The dispatch payload grid's last CTA watches every segment's ready flag and
copies the segment's rows, assist_info entries and dynamic scales the moment
the flag shows the call's ticket (the combine_doubleplane README, 实现逻辑:
a segment's status is written only after its payload is visible). Every copy
must equal the final output, which itself equals the oracle: a flag that
became visible before its rows would leave poisoned bytes in the copy."""
import ctypes
import os

import numpy as np
import pytest
import torch

import workloads as WL
from oracle import oracle as O

pytestmark = pytest.mark.gpu

if os.environ.get("CRS_MOE_OBSERVER") != "1":
    pytest.skip("needs the flag-observer build (CRS_MOE_OBSERVER=1)", allow_module_level=True)

import gpu_harness as H  # noqa: E402
from combine_route_scan_gb300 import moe as M  # noqa: E402

TICKET = 7


def observed_dispatch(wl, policy, bulk_min_bytes):
    inp = WL.make_inputs(wl)
    ref = O.dispatch(wl, inp)
    dev = H.device_inputs(wl, inp)
    W, L = wl.ep_world_size, wl.moe_expert_num // wl.ep_world_size
    cfg = H.make_cfg(wl, plane_policy=policy, bulk_min_bytes=bulk_min_bytes)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_dispatch_outputs(cfg, H.TORCH_DT[wl.x_dtype], seg_plane=True)
    for t in out.values():
        if t is not None:
            t.view(torch.uint8).fill_(0xA5)
    snap_rows = torch.empty_like(out["expand_x"])
    snap_rows.view(torch.uint8).fill_(0x5A)
    snap_assist = torch.full_like(out["assist_info"], -7)
    snap_dyn = None
    if out["dynamic_scales"] is not None:
        snap_dyn = torch.empty_like(out["dynamic_scales"])
        snap_dyn.view(torch.uint8).fill_(0x5A)
    nseg = wl.moe_expert_num * W
    seen = torch.zeros(nseg, dtype=torch.int64, device="cuda")
    prod_end = torch.zeros(1, dtype=torch.int64, device="cuda")
    n_seen = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = torch.zeros((W, L * W), dtype=torch.int32, device="cuda")
    lib = M.lib()
    lib.moe_test_set_flag_observer.argtypes = [ctypes.c_void_p] * 6
    lib.moe_test_set_flag_observer.restype = ctypes.c_int32
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert lib.moe_test_set_flag_observer(p(snap_rows), p(snap_assist), p(snap_dyn), p(seen), p(prod_end),
                                          p(n_seen)) == 0
    try:
        c = M.with_seg_ready(cfg, flags, TICKET)
        M.dispatch(c, dev["x"], dev["expert_ids"], dev["active_mask"], dev["expert_scales"], out["expand_x"],
                   out["dynamic_scales"], out["assist_info"], out["ep_recv_count"], out["expand_scales"],
                   out["seg_plane"], ws, scales=dev.get("quant_scales"))
        st = M.get_device_status(ws)
    finally:
        lib.moe_test_set_flag_observer(None, None, None, None, None, None)
    assert st == 0, M.STATUS.get(st, st)
    assert bool((flags == TICKET).all())
    assert int(n_seen.item()) == nseg, (int(n_seen.item()), nseg)
    H.compare_dispatch(wl, out, ref)
    # every copy taken at flag time equals the final rows
    ep = H.to_host(out["ep_recv_count"])
    for d in range(W):
        n = int(ep[d, -1])
        assert torch.equal(snap_rows[d, :n], out["expand_x"][d, :n]), f"rows of rank {d} seen before they landed"
        assert torch.equal(snap_assist[d, :n], out["assist_info"][d, :n]), f"assist_info of rank {d}"
        if snap_dyn is not None:
            assert torch.equal(snap_dyn[d, :n], out["dynamic_scales"][d, :n]), f"dynamic scales of rank {d}"
    # the copies were taken while other CTAs were still storing
    cnt = np.diff(np.concatenate([np.zeros((W, 1), np.int64), ep.astype(np.int64)], axis=1), axis=1)
    nonempty = cnt.reshape(-1) > 0  # index d*L*W + le*W + s == e*W + s
    early = (H.to_host(seen) < int(prod_end.item())) & nonempty
    planes = H.to_host(out["seg_plane"]).reshape(-1)
    print(f"{wl.name} policy {policy}: {int(nonempty.sum())} non-empty segments, {int(early.sum())} copied complete "
          f"before the last storing CTA ended ({int((early & (planes == 1)).sum())} of them on the bulk plane)")
    assert early.sum() >= 1
    return early, planes, nonempty


ZIPF = WL.Workload("flags_zipf", 8, 256, 4096, 8, 64, WL.X_BF16, zero_expert_num=2, copy_expert_num=2,
                   mask_kind=2, ids="zipf", special_p=0.05, mask_false_p=0.1, seed=71)


def test_flags_follow_rows_zipf_two_planes():
    """Zipf routing under the page's plane rule (size threshold 0: the
    above-mean remote segments go by bulk copies, the rest by stores); both
    planes' flags were seen early and their copies are complete."""
    early, planes, nonempty = observed_dispatch(ZIPF, M.PLANE_RULE, 0)
    assert (planes[nonempty] == 1).any() and (planes[nonempty] == 0).any()


def test_flags_follow_rows_every_remote_segment_bulk():
    observed_dispatch(ZIPF.with_(seed=72), M.PLANE_BULK_ALL, M.BULK_MIN_BYTES)


# 32768 tokens of short rows: dozens of tokens per storing CTA, so the source
# ranks' segments complete one after another while the grid keeps storing
WAVES = WL.Workload("flags_waves", 16, 2048, 256, 4, 64, WL.X_BF16, zero_expert_num=1, copy_expert_num=1,
                    mask_kind=2, ids="zipf", special_p=0.05, mask_false_p=0.1, seed=74)


@pytest.mark.parametrize("policy", ["rule", "bulk"])
def test_flags_seen_while_the_grid_stores(policy):
    """The source ranks' segments complete one after another; dozens of them
    are copied complete, store-plane and bulk-plane ones, while the grid is
    still storing (one observing CTA cannot copy all 57 MB that fast: the
    copies are a sample, taken in the order the flags appear)."""
    early, planes, nonempty = (observed_dispatch(WAVES, M.PLANE_RULE, 0) if policy == "rule" else
                               observed_dispatch(WAVES, M.PLANE_BULK_ALL, M.BULK_MIN_BYTES))
    assert early.sum() >= 32
    assert (early & (planes == 1)).sum() >= 4 and (early & (planes == 0) & nonempty).sum() >= 4


@pytest.mark.parametrize("q,y", [(2, ""), (4, "fp8_e4m3")])
def test_flags_seen_while_the_quantising_grid_stores(q, y):
    early, planes, nonempty = observed_dispatch(WAVES.with_(quant_mode=q, y_dtype=y, seed=75), M.PLANE_RULE, 0)
    assert early.sum() >= 32


@pytest.mark.parametrize("q,y", [(2, ""), (4, "fp8_e4m3")])
def test_flags_follow_rows_quantised(q, y):
    """The quantising scatter (per-token int8; MX FP8): rows, assist_info and
    dynamic scales complete when the flag is seen."""
    observed_dispatch(ZIPF.with_(quant_mode=q, y_dtype=y, seed=73), M.PLANE_RULE, 0)
