"""CUDA dispatch / combine against the CPU oracle, element by element.

Integer, index, count and int8 outputs must match bit for bit; float combine
outputs within max |gpu - oracle| <= 1e-3 * max |oracle|. The kernels fix the
fp32 accumulation order (k ascending, fused multiply-add), so the float
outputs are also checked for bit equality.
"""
import time

import numpy as np
import pytest
import torch

import workloads as WL
from oracle import oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gpu_harness as H
    from combine_route_scan_gb300 import moe as M
    from combine_route_scan_gb300 import build as B
    B.build()

SMALL = ["w2_bs8_h16_k2_e4_i32", "w8_bs8_h16_k2_e64_i32", "w8_bs8_h16_k2_e64_f16", "w2_bs8_h256_k2_e4_i32"]
FULL = ["w8_bs32_h7168_k8_e64_f16", "w8_bs32_h7168_k8_e64_f16_q2", "w8_bs32_h7168_k8_e64_i32",
        "w16_bs256_h7168_k8_e256_bf16_zipf", "w8_bs64_h2048_k8_e128_bf16_ffn"]


def run_and_compare(wl, inp=None, plane_policy=0, bulk_min_bytes=O.DEFAULT_BULK_MIN_BYTES, exact_float=True):
    inp = WL.make_inputs(wl) if inp is None else inp
    ref = O.dispatch(wl, inp)
    dev = H.device_inputs(wl, inp)
    got, ws, _ = H.gpu_dispatch(wl, dev, plane_policy=plane_policy, bulk_min_bytes=bulk_min_bytes)
    plane_ref = O.dispatch_plane(wl, ref["ep_recv_count"], bulk_min_bytes) if plane_policy == 0 else None
    if plane_policy == 0 and not _tma_rows(wl):
        plane_ref = np.zeros_like(ref["ep_recv_count"], dtype=np.uint8)
    H.compare_dispatch(wl, got, ref, plane_ref)
    err = None
    if wl.quant_mode == 0:
        x_out, _, _ = H.gpu_combine(wl, dev, got["expand_x"], got["assist_info"], got["ep_recv_count"])
        x_ref = O.combine(wl, ref["expand_x"], ref["assist_info"], ref["ep_recv_count"], inp)
        got_out = H.to_host(x_out)
        err = H.compare_combine(wl, got_out, x_ref)
        if exact_float:
            assert np.array_equal(got_out.view(np.uint8), x_ref.view(np.uint8)), "combine bytes"
    return got, ref, err


def _tma_rows(wl):
    """Rows in and out are 16-byte multiples (x's row; int8 / fp8 codes take h
    bytes, packed fp4 h / 2)."""
    out = wl.h * wl.es if wl.quant_mode == 0 else (wl.h // 2 if wl.y_dtype == "fp4_e2m1" else wl.h)
    return wl.h * wl.es % 16 == 0 and out % 16 == 0


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("plane_policy", [0, 1, 2])
def test_small_workloads(name, plane_policy):
    run_and_compare(WL.WORKLOADS[name], plane_policy=plane_policy)


@pytest.mark.parametrize("seed", range(24))
def test_random_small(seed):
    rng = np.random.default_rng(500 + seed)
    dt = [WL.X_INT32, WL.X_FP16, WL.X_BF16][seed % 3]
    wl = WL.small_random_workload(rng, x_dtype=dt, max_w=6, max_bs=12)
    run_and_compare(wl, plane_policy=seed % 3, bulk_min_bytes=0 if seed % 2 else O.DEFAULT_BULK_MIN_BYTES)


@pytest.mark.parametrize("seed", range(6))
def test_random_many_tokens_per_scatter_cta(seed):
    """Medium random problems with short rows: far more tokens than the TMA
    scatter's resident CTAs hold in their rings, so most tokens go out by the
    workspace's ticket counter; Zipf or uniform routing, masks and specials;
    dispatch and gather combine on the same workspace (the map the scatter
    wrote) against the oracle."""
    rng = np.random.default_rng(900 + seed)
    W = int(rng.choice([2, 4, 8, 16]))
    L = int(rng.choice([1, 2, 4, 8]))
    K = int(rng.integers(1, min(W * L, 8) + 1))
    h = int(rng.choice([8, 64, 256]))
    dt = [WL.X_FP16, WL.X_BF16, WL.X_INT32][seed % 3]
    bs = int(rng.integers(8192, 16385)) // W  # > 4 ring slots x 1216 CTAs (short rows: 8 CTAs a SM)
    Z, C = int(rng.integers(0, 3)), int(rng.integers(0, 3))
    wl = WL.Workload(f"rand_many_w{W}_l{L}_k{K}_bs{bs}_h{h}", W, bs, h, K, W * L, dt, zero_expert_num=Z,
                     copy_expert_num=C, mask_kind=int(rng.integers(0, 3)), special_p=0.1 if Z + C else 0.0,
                     mask_false_p=0.1, ids="zipf" if seed % 2 else "uniform", x_range=100, seed=seed + 77)
    inp = WL.make_inputs(wl)
    ref = O.dispatch(wl, inp)
    x_ref = O.combine(wl, ref["expand_x"], ref["assist_info"], ref["ep_recv_count"], inp)
    dev = H.device_inputs(wl, inp)
    got, ws, _ = H.gpu_dispatch(wl, dev)
    H.compare_dispatch(wl, got, ref, O.dispatch_plane(wl, ref["ep_recv_count"], O.DEFAULT_BULK_MIN_BYTES))
    x_out, st = _combine_same_ws(wl, dev, got, ws)
    assert st == 0, M.STATUS.get(st, st)
    assert np.array_equal(H.to_host(x_out).view(np.uint8), x_ref.view(np.uint8))


@pytest.mark.parametrize("h,dt,q", [(12, WL.X_FP16, 0), (20, WL.X_BF16, 0), (3, WL.X_INT32, 0),
                                    (24, WL.X_FP16, 2), (40, WL.X_BF16, 2), (5, WL.X_BF16, 2)])
def test_rows_not_multiple_of_16_bytes(h, dt, q):
    wl = WL.Workload(f"ragged_h{h}", 4, 9, h, 3, 8, dt, zero_expert_num=1, copy_expert_num=1, mask_kind=2,
                     special_p=0.2, mask_false_p=0.2, quant_mode=q, seed=h)
    run_and_compare(wl)


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads(name):
    got, ref, err = run_and_compare(WL.WORKLOADS[name])
    if name.endswith("_zipf"):
        # the skewed routing really sends some segments by the bulk plane
        assert H.to_host(got["seg_plane"]).sum() > 0


def test_planes_give_identical_bytes():
    """The page requires the two-plane version to give the same outputs as the
    single-plane one: rule, stores only and bulk for all remote segments."""
    wl = WL.WORKLOADS["w16_bs256_h7168_k8_e256_bf16_zipf"]
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    outs = []
    for pol in (0, 1, 2):
        got, _, _ = H.gpu_dispatch(wl, dev, plane_policy=pol)
        outs.append(got)
    ep = H.to_host(outs[0]["ep_recv_count"])
    for other in outs[1:]:
        assert np.array_equal(H.to_host(other["ep_recv_count"]), ep)
        for d in range(wl.ep_world_size):
            n = int(ep[d, -1])
            assert torch.equal(other["expand_x"][d, :n], outs[0]["expand_x"][d, :n])
            assert torch.equal(other["assist_info"][d, :n], outs[0]["assist_info"][d, :n])
    assert H.to_host(outs[1]["seg_plane"]).sum() == 0
    assert H.to_host(outs[2]["seg_plane"]).sum() > H.to_host(outs[0]["seg_plane"]).sum() > 0


def test_quant_q2_small_with_ties():
    """quantMode 2 on rows built to hit exact .5 ties (amax 127, scale 1)."""
    wl = WL.Workload("q2_ties", 2, 16, 64, 2, 4, WL.X_FP16, quant_mode=2, seed=3)
    inp = WL.make_inputs(wl)
    rng = np.random.default_rng(4)
    x = (rng.integers(-254, 255, size=inp["x"].shape) / 2.0).astype(np.float16)
    x[..., 0] = 127.0
    x[0, 3] = 0.0  # an all-zero token: scale 0, q 0
    inp["x"] = x
    run_and_compare(wl, inp)


def test_determinism_same_bytes():
    wl = WL.WORKLOADS["w16_bs256_h7168_k8_e256_bf16_zipf"]
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    a, ws, _ = H.gpu_dispatch(wl, dev)
    b, _, _ = H.gpu_dispatch(wl, dev, ws=ws)
    ep = H.to_host(a["ep_recv_count"])
    assert np.array_equal(ep, H.to_host(b["ep_recv_count"]))
    for d in range(wl.ep_world_size):
        n = int(ep[d, -1])
        assert torch.equal(a["expand_x"][d, :n], b["expand_x"][d, :n])
    xa, _, _ = H.gpu_combine(wl, dev, a["expand_x"], a["assist_info"], a["ep_recv_count"])
    xb, _, _ = H.gpu_combine(wl, dev, a["expand_x"], a["assist_info"], a["ep_recv_count"])
    assert torch.equal(xa, xb)


def test_empty_batch():
    wl = WL.Workload("empty", 4, 0, 64, 2, 8, WL.X_FP16)
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    got, _, _ = H.gpu_dispatch(wl, dev)
    assert H.to_host(got["ep_recv_count"]).sum() == 0
    x_out, _, _ = H.gpu_combine(wl, dev, got["expand_x"], got["assist_info"], got["ep_recv_count"])
    assert x_out.numel() == 0


def test_all_masked_and_all_special():
    wl = WL.Workload("masked", 4, 8, 32, 2, 8, WL.X_INT32, mask_kind=2, mask_false_p=1.0, seed=1)
    got, ref, _ = run_and_compare(wl)
    assert H.to_host(got["ep_recv_count"]).sum() == 0
    wl = WL.Workload("special", 4, 8, 32, 2, 8, WL.X_BF16, zero_expert_num=1, copy_expert_num=2,
                     special_p=1.0, seed=2)
    got, ref, _ = run_and_compare(wl)
    assert H.to_host(got["ep_recv_count"]).sum() == 0


def test_one_expert_takes_everything():
    """Every token routes to expert 0 (plus distinct others): one segment per
    source holds the whole batch."""
    wl = WL.Workload("hot", 8, 64, 1024, 2, 16, WL.X_FP16, seed=6)
    inp = WL.make_inputs(wl)
    ids = inp["expert_ids"]
    ids[..., 0] = 0
    ids[..., 1] = np.where(ids[..., 1] == 0, 1, ids[..., 1])
    run_and_compare(wl, inp, bulk_min_bytes=64 * 1024)


@pytest.mark.parametrize("W,E,bs,K,h", [(64, 1024, 16, 8, 64), (768, 768, 2, 1, 16), (32, 256, 40, 16, 128),
                                        (8, 1024, 16, 8, 64), (16, 512, 8, 4, 32), (4, 64, 300, 4, 128),
                                        (8, 256, 12, 32, 64), (2, 64, 9, 32, 256)])
def test_wide_configurations(W, E, bs, K, h):
    wl = WL.Workload(f"wide_w{W}", W, bs, h, K, E, WL.X_BF16, zero_expert_num=2, copy_expert_num=2,
                     mask_kind=1, special_p=0.1, seed=W)
    run_and_compare(wl)


def test_one_dimensional_mask():
    wl = WL.Workload("mask1d", 8, 32, 256, 4, 32, WL.X_FP16, mask_kind=1, copy_expert_num=2, special_p=0.1, seed=8)
    run_and_compare(wl)


# ----------------------------------------------------------------- errors

def _status_of_dispatch(wl, inp):
    dev = H.device_inputs(wl, inp)
    _, _, st = H.gpu_dispatch(wl, dev, check_status=False)
    return M.STATUS[st]


def test_device_errors_match_oracle():
    base = WL.Workload("err", 2, 4, 16, 2, 4, WL.X_INT32, zero_expert_num=1, copy_expert_num=1)
    inp = WL.make_inputs(base)
    bad = dict(inp, expert_ids=inp["expert_ids"].copy())
    bad["expert_ids"][1, 2, 1] = 6
    assert _status_of_dispatch(base, bad) == "BAD_EXPERT_ID" == O.STATUS_NAMES[O.dispatch(base, bad, raise_on_error=False)["status"]]
    bad["expert_ids"][1, 2, 1] = -3
    assert _status_of_dispatch(base, bad) == "BAD_EXPERT_ID"
    dup = dict(inp, expert_ids=inp["expert_ids"].copy())
    dup["expert_ids"][0, 0, :] = 3
    assert _status_of_dispatch(base, dup) == "BAD_EXPERT_ID"
    m1 = base.with_(mask_kind=1)
    badm = dict(inp, active_mask=np.array([[1, 0, 1, 0], [1, 1, 1, 1]], dtype=np.uint8))
    assert _status_of_dispatch(m1, badm) == "MASK_ORDER" == O.STATUS_NAMES[O.dispatch(m1, badm, raise_on_error=False)["status"]]
    # the status word is cleared by reading it: a good call afterwards is OK
    assert _status_of_dispatch(base, inp) == "OK"


def test_combine_detects_inconsistent_assist_info():
    wl = WL.WORKLOADS["w8_bs8_h16_k2_e64_i32"]
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    got, _, _ = H.gpu_dispatch(wl, dev)
    ai = got["assist_info"].clone()
    ep = H.to_host(got["ep_recv_count"])
    d = int(np.argmax(ep[:, -1]))
    ai[d, 0, 1] = (ai[d, 0, 1] + 1) % wl.bs  # row 0 of rank d now names another token
    _, st, _ = H.gpu_combine(wl, dev, got["expand_x"], ai, got["ep_recv_count"], check_status=False)
    assert M.STATUS[st] == "BAD_ASSIST"


def test_host_argument_errors():
    wl = WL.WORKLOADS["w2_bs8_h16_k2_e4_i32"]
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    cfg = H.make_cfg(wl)
    out = M.alloc_dispatch_outputs(cfg, torch.int32)
    ws = M.alloc_workspace(cfg)
    with pytest.raises(M.MoeError) as ei:
        M.dispatch(cfg, dev["x"], dev["expert_ids"], None, dev["expert_scales"], out["expand_x"], None,
                   out["assist_info"], out["ep_recv_count"], ws=ws[:64])
    assert ei.value.name == "WORKSPACE"
    with pytest.raises(M.MoeError) as ei:
        M.dispatch(cfg, dev["x"], dev["expert_ids"], None, None, out["expand_x"], None,
                   out["assist_info"], out["ep_recv_count"], expand_scales=out["expand_scales"], ws=ws)
    assert ei.value.name == "INVALID_ARG"


# ------------------------------------------------------- two-phase combine

@pytest.mark.parametrize("name", ["w2_bs8_h16_k2_e4_i32", "w8_bs8_h16_k2_e64_f16",
                                  "w8_bs32_h7168_k8_e64_i32", "w16_bs256_h7168_k8_e256_bf16_zipf"])
@pytest.mark.parametrize("plane_policy", [0, 1, 2])
def test_two_phase_matches_gather_and_oracle(name, plane_policy):
    """The page's write-back + status protocol gives the same bytes as the
    gather combine and the oracle, and picks the oracle's planes."""
    wl = WL.WORKLOADS[name]
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    got, _, _ = H.gpu_dispatch(wl, dev)
    ref = O.dispatch(wl, inp)
    x_ref = O.combine(wl, ref["expand_x"], ref["assist_info"], ref["ep_recv_count"], inp)
    xg, _, _ = H.gpu_combine(wl, dev, got["expand_x"], got["assist_info"], got["ep_recv_count"])
    xt, _, sp = H.gpu_combine(wl, dev, got["expand_x"], got["assist_info"], got["ep_recv_count"],
                              combine_mode=M.COMBINE_TWO_PHASE, plane_policy=plane_policy, seg_plane=True)
    assert torch.equal(xt, xg)
    H.compare_combine(wl, H.to_host(xt), x_ref)
    assert np.array_equal(H.to_host(xt).view(np.uint8), x_ref.view(np.uint8))
    if plane_policy == 0:
        assert np.array_equal(H.to_host(sp), O.combine_plane(wl, ref["ep_recv_count"]))
    elif plane_policy == 1:
        assert H.to_host(sp).sum() == 0


def test_two_phase_repeated_calls_and_put_only():
    wl = WL.WORKLOADS["w16_bs256_h7168_k8_e256_bf16_zipf"]
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    got, _, _ = H.gpu_dispatch(wl, dev)
    cfg = H.make_cfg(wl, combine_mode=M.COMBINE_TWO_PHASE)
    ws = M.alloc_workspace(cfg)
    xg, _, _ = H.gpu_combine(wl, dev, got["expand_x"], got["assist_info"], got["ep_recv_count"])
    cfg_put = H.make_cfg(wl, combine_mode=M.COMBINE_PUT_ONLY)
    for _ in range(3):
        x_out = torch.zeros_like(xg)
        M.combine(cfg, got["expand_x"], got["assist_info"], got["ep_recv_count"], dev["expert_ids"],
                  dev["expert_scales"], dev["active_mask"], dev["x"], x_out, None, ws)
        assert M.get_device_status(ws) == 0
        assert torch.equal(x_out, xg)
        # put only (the page's comm_only): x_out is not written, the epoch still advances
        untouched = torch.full_like(xg, 7)
        M.combine(cfg_put, got["expand_x"], got["assist_info"], got["ep_recv_count"], dev["expert_ids"],
                  dev["expert_scales"], dev["active_mask"], dev["x"], untouched, None, ws)
        assert M.get_device_status(ws) == 0
        assert bool((untouched == 7).all())


def test_two_phase_wait_times_out_on_a_missing_flag():
    """Withhold one row from the put phase (its rank claims one row less): the
    reduce's bounded wait on that pick's flag runs out and reports TIMEOUT."""
    wl = WL.WORKLOADS["w8_bs8_h16_k2_e64_f16"]
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    got, _, _ = H.gpu_dispatch(wl, dev)
    ep = got["ep_recv_count"].clone()
    d = int(torch.argmax(ep[:, -1]).item())
    ep[d, -1] -= 1
    cfg = H.make_cfg(wl, quant_mode=0, combine_mode=M.COMBINE_TWO_PHASE, wait_timeout_us=20000)
    ws = M.alloc_workspace(cfg)
    x_out = torch.empty_like(dev["x"])
    M.combine(cfg, got["expand_x"], got["assist_info"], ep, dev["expert_ids"], dev["expert_scales"],
              dev["active_mask"], dev["x"], x_out, None, ws)
    assert M.STATUS[M.get_device_status(ws)] == "TIMEOUT"
    # the workspace stays usable: a consistent call afterwards is clean
    M.combine(cfg, got["expand_x"], got["assist_info"], got["ep_recv_count"], dev["expert_ids"],
              dev["expert_scales"], dev["active_mask"], dev["x"], x_out, None, ws)
    assert M.get_device_status(ws) == 0


# ------------------------------------------------- dispatch ready flags

@pytest.mark.parametrize("name,policy", [("w16_bs256_h7168_k8_e256_bf16_zipf", 0),
                                         ("w16_bs256_h7168_k8_e256_bf16_zipf", 2),
                                         ("w8_bs32_h7168_k8_e64_f16_q2", 2),
                                         ("w8_bs8_h16_k2_e64_f16", 0),
                                         ("ragged_h12_f16", 0)])
def test_dispatch_ready_flags(name, policy):
    """seg_ready[d][le*W+s] carries the call's ticket once segment (le, s) of
    rank d is complete, for every segment (empty ones too); flags change no
    output."""
    if name == "ragged_h12_f16":
        wl = WL.Workload(name, 4, 9, 12, 3, 8, WL.X_FP16, mask_kind=2, mask_false_p=0.2, seed=12)
    else:
        wl = WL.WORKLOADS[name]
    inp = WL.make_inputs(wl)
    ref = O.dispatch(wl, inp)
    dev = H.device_inputs(wl, inp)
    L = wl.moe_expert_num // wl.ep_world_size
    cfg = H.make_cfg(wl, plane_policy=policy, bulk_min_bytes=0 if policy == 0 and wl.h < 1024 else M.BULK_MIN_BYTES)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_dispatch_outputs(cfg, H.TORCH_DT[wl.x_dtype])
    flags = torch.zeros((wl.ep_world_size, L * wl.ep_world_size), dtype=torch.int32, device="cuda")
    for ticket in (7, 8):
        c = M.with_seg_ready(cfg, flags, ticket)
        M.dispatch(c, dev["x"], dev["expert_ids"], dev["active_mask"], dev["expert_scales"], out["expand_x"],
                   out["dynamic_scales"], out["assist_info"], out["ep_recv_count"], out["expand_scales"], None, ws)
        assert M.get_device_status(ws) == 0
        assert bool((flags == ticket).all()), f"ticket {ticket}: {int((flags != ticket).sum())} segments not flagged"
        H.compare_dispatch(wl, out, ref)


# ------------------------------------------------- dispatch performance info

@pytest.mark.parametrize("name", ["w16_bs256_h7168_k8_e256_bf16_zipf", "w8_bs32_h7168_k8_e64_f16_q2",
                                  "ragged_h12_f16", "empty_batch"])
def test_dispatch_performance_info(name):
    """performance_info[s] gains rank s's communication time (ns) on every
    call: never negative, never longer than the host-timed calls, growing
    across calls, zero for an empty batch; outputs are unchanged."""
    if name == "ragged_h12_f16":
        wl = WL.Workload(name, 4, 9, 12, 3, 8, WL.X_FP16, mask_kind=2, mask_false_p=0.2, seed=12)
    elif name == "empty_batch":
        wl = WL.Workload(name, 4, 0, 256, 2, 8, WL.X_BF16, seed=13)
    else:
        wl = WL.WORKLOADS[name]
    inp = WL.make_inputs(wl)
    ref = O.dispatch(wl, inp)
    dev = H.device_inputs(wl, inp)
    cfg = H.make_cfg(wl)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_dispatch_outputs(cfg, H.TORCH_DT[wl.x_dtype])
    perf = torch.zeros(wl.ep_world_size, dtype=torch.int64, device="cuda")
    c = M.with_performance_info(cfg, perf)
    prev = np.zeros(wl.ep_world_size, dtype=np.int64)
    torch.cuda.synchronize()
    t0 = time.perf_counter_ns()
    for _ in range(3):
        M.dispatch(c, dev["x"], dev["expert_ids"], dev["active_mask"], dev["expert_scales"], out["expand_x"],
                   out["dynamic_scales"], out["assist_info"], out["ep_recv_count"], out["expand_scales"], None, ws)
        assert M.get_device_status(ws) == 0
        cur = perf.cpu().numpy()
        assert (cur >= prev).all(), (prev, cur)
        prev = cur
    elapsed = time.perf_counter_ns() - t0
    if wl.bs == 0:
        assert not prev.any()
        return
    H.compare_dispatch(wl, out, ref)
    assert prev.max() <= elapsed, (prev.max(), elapsed)
    if wl.ep_world_size * wl.bs >= 1024:
        # a multi-microsecond scatter: every rank's span is measurable
        assert (prev > 0).all(), prev


def test_dispatch_performance_info_alignment():
    wl = WL.Workload("perf_align", 2, 4, 64, 2, 4, WL.X_FP16, seed=14)
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    cfg = H.make_cfg(wl)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_dispatch_outputs(cfg, H.TORCH_DT[wl.x_dtype])
    buf = torch.zeros(8, dtype=torch.int32, device="cuda")
    c = M.with_performance_info(cfg, buf[1:])  # 4-byte aligned only
    with pytest.raises(M.MoeError) as ei:
        M.dispatch(c, dev["x"], dev["expert_ids"], dev["active_mask"], dev["expert_scales"], out["expand_x"],
                   out["dynamic_scales"], out["assist_info"], out["ep_recv_count"], out["expand_scales"], None, ws)
    assert ei.value.name == "INVALID_ARG"


# ------------------------------------- pick -> row map left by the dispatch

def _combine_same_ws(wl, dev, got, ws, assist=None, ep=None):
    cfg = H.make_cfg(wl, quant_mode=0)
    x_out = torch.empty((wl.ep_world_size, wl.bs, wl.h), dtype=H.TORCH_DT[wl.x_dtype], device="cuda")
    M.combine(cfg, got["expand_x"], got["assist_info"] if assist is None else assist,
              got["ep_recv_count"] if ep is None else ep, dev["expert_ids"], dev["expert_scales"],
              dev["active_mask"], dev["x"], x_out, None, ws)
    return x_out, M.get_device_status(ws)


@pytest.mark.parametrize("name", ["w16_bs256_h7168_k8_e256_bf16_zipf", "w8_bs8_h16_k2_e64_i32", "ragged_h12_f16"])
def test_combine_reuses_the_dispatch_row_map(name):
    """Dispatch and combine on one workspace: the combine takes the map the
    scatter wrote (no inverse pass) and matches the oracle byte for byte."""
    if name == "ragged_h12_f16":
        wl = WL.Workload(name, 4, 9, 12, 3, 8, WL.X_FP16, mask_kind=2, mask_false_p=0.2, zero_expert_num=1,
                         copy_expert_num=1, special_p=0.2, seed=41)
    else:
        wl = WL.WORKLOADS[name]
    inp = WL.make_inputs(wl)
    ref = O.dispatch(wl, inp)
    x_ref = O.combine(wl, ref["expand_x"], ref["assist_info"], ref["ep_recv_count"], inp)
    dev = H.device_inputs(wl, inp)
    got, ws, _ = H.gpu_dispatch(wl, dev)
    x_out, st = _combine_same_ws(wl, dev, got, ws)
    assert st == 0
    assert np.array_equal(H.to_host(x_out).view(np.uint8), x_ref.view(np.uint8))


def test_row_map_follows_the_buffers():
    """Two dispatches on one workspace into different output buffers: a
    combine of the first one's buffers rebuilds its map and is still right;
    an assist_info changed in place after the dispatch so that a pick has no
    row is reported."""
    wl = WL.WORKLOADS["w8_bs8_h16_k2_e64_i32"]
    inp_a = WL.make_inputs(wl)
    inp_b = WL.make_inputs(wl, seed=99)
    dev_a, dev_b = H.device_inputs(wl, inp_a), H.device_inputs(wl, inp_b)
    got_a, ws, _ = H.gpu_dispatch(wl, dev_a)
    got_b, _, _ = H.gpu_dispatch(wl, dev_b, ws=ws)
    ref_a = O.dispatch(wl, inp_a)
    x_ref = O.combine(wl, ref_a["expand_x"], ref_a["assist_info"], ref_a["ep_recv_count"], inp_a)
    x_out, st = _combine_same_ws(wl, dev_a, got_a, ws)
    assert st == 0 and np.array_equal(H.to_host(x_out), x_ref)
    # B's buffers are the ones the workspace's map belongs to; now break B's
    # assist_info in place (same pointer): the reduce's check must catch it
    got_b2, ws2, _ = H.gpu_dispatch(wl, dev_b)
    ep = H.to_host(got_b2["ep_recv_count"])
    d = int(np.argmax(ep[:, -1]))
    got_b2["assist_info"][d, 0, 1] = (got_b2["assist_info"][d, 0, 1] + 1) % wl.bs
    _, st = _combine_same_ws(wl, dev_b, got_b2, ws2)
    assert M.STATUS[st] == "BAD_ASSIST"


def _ragged_wl():
    return WL.Workload("ragged_h12_f16", 4, 9, 12, 3, 8, WL.X_FP16, mask_kind=2, mask_false_p=0.2, zero_expert_num=1,
                       copy_expert_num=1, special_p=0.2, seed=41)


@pytest.mark.parametrize("name", ["w16_bs256_h7168_k8_e256_bf16_zipf", "w8_bs32_h7168_k8_e64_f16", "ragged_h12_f16"])
def test_graph_replays_and_eager_calls_share_a_workspace(name):
    """A CUDA graph holding dispatch + combine of buffer set B and eager calls
    on set A share one workspace. A replay of the graph overwrites the
    workspace's row map unseen by the library, so an eager combine of A
    after it must not take that map for A's; the graph's own combine follows
    its dispatch on every replay. Both match the oracle byte for byte (ragged
    rows take the element-wise reduce)."""
    wl = _ragged_wl() if name == "ragged_h12_f16" else WL.WORKLOADS[name]
    inp_a, inp_b = WL.make_inputs(wl), WL.make_inputs(wl, seed=5)
    dev_a, dev_b = H.device_inputs(wl, inp_a), H.device_inputs(wl, inp_b)
    cfg = H.make_cfg(wl)
    ws = M.alloc_workspace(cfg)
    out_b = M.alloc_dispatch_outputs(cfg, H.TORCH_DT[wl.x_dtype])
    x_out_b = torch.empty((wl.ep_world_size, wl.bs, wl.h), dtype=H.TORCH_DT[wl.x_dtype], device="cuda")
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        M.dispatch(cfg, dev_b["x"], dev_b["expert_ids"], dev_b["active_mask"], dev_b["expert_scales"],
                   out_b["expand_x"], out_b["dynamic_scales"], out_b["assist_info"], out_b["ep_recv_count"],
                   out_b["expand_scales"], None, ws)
        M.combine(cfg, out_b["expand_x"], out_b["assist_info"], out_b["ep_recv_count"], dev_b["expert_ids"],
                  dev_b["expert_scales"], dev_b["active_mask"], dev_b["x"], x_out_b, None, ws)

    def ref(inp):
        r = O.dispatch(wl, inp)
        return O.combine(wl, r["expand_x"], r["assist_info"], r["ep_recv_count"], inp)

    got_a, _, _ = H.gpu_dispatch(wl, dev_a, ws=ws)
    graph.replay()  # B's map is now in the workspace
    x_out_a, st = _combine_same_ws(wl, dev_a, got_a, ws)
    assert st == 0, M.STATUS.get(st, st)
    assert np.array_equal(H.to_host(x_out_a).view(np.uint8), ref(inp_a).view(np.uint8))
    x_out_b.view(torch.uint8).fill_(0x5A)
    graph.replay()
    torch.cuda.synchronize()
    assert M.get_device_status(ws) == 0
    assert np.array_equal(H.to_host(x_out_b).view(np.uint8), ref(inp_b).view(np.uint8))


def test_launch_count_shows_the_skipped_inverse_pass():
    """The library's own launch count: dispatch = routing + scatter; a combine
    of the same buffers on the same workspace = the reduce alone; a combine
    of buffers the workspace's map was not written for adds the inverse-map
    kernel."""
    wl = WL.WORKLOADS["w8_bs32_h7168_k8_e64_f16"]
    inp_a, inp_b = WL.make_inputs(wl), WL.make_inputs(wl, seed=3)
    dev_a, dev_b = H.device_inputs(wl, inp_a), H.device_inputs(wl, inp_b)
    n0 = M.launch_count()
    got_a, ws, _ = H.gpu_dispatch(wl, dev_a)
    assert M.launch_count() - n0 == 2
    n0 = M.launch_count()
    _, st = _combine_same_ws(wl, dev_a, got_a, ws)
    assert st == 0 and M.launch_count() - n0 == 1
    got_b, _, _ = H.gpu_dispatch(wl, dev_b, ws=ws)
    n0 = M.launch_count()
    x_out, st = _combine_same_ws(wl, dev_a, got_a, ws)  # the map is B's now
    assert st == 0 and M.launch_count() - n0 == 2
    ref = O.dispatch(wl, inp_a)
    x_ref = O.combine(wl, ref["expand_x"], ref["assist_info"], ref["ep_recv_count"], inp_a)
    assert np.array_equal(H.to_host(x_out).view(np.uint8), x_ref.view(np.uint8))


def test_launch_limits_survive_smaller_shapes():
    """A kernel's dynamic shared-memory limit only ever rises: a large row
    shape, then a small one, then the large one again all launch and match."""
    for h in (7168, 256, 7168, 1024):
        wl = WL.Workload(f"lim_h{h}", 4, 8, h, 4, 16, WL.X_BF16, seed=61)
        run_and_compare(wl)
        wq = wl.with_(quant_mode=3, y_dtype="fp8_e4m3")
        inp = WL.make_inputs(wq)
        ref = O.dispatch(wq, inp)
        got, _, _ = H.gpu_dispatch(wq, H.device_inputs(wq, inp))
        H.compare_dispatch(wq, got, ref)
