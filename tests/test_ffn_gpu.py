"""moe_dispatch_ffn_combine (dispatch -> SwiGLU expert FFN on tcgen05 -> combine)
against the fp64 CPU oracle: max |gpu - oracle| <= 2e-2 * max |oracle| over
the compared tokens (bf16 operands, fp32 accumulation, bf16 intermediate and
expert output on the GPU)."""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import workloads as WL
from oracle import oracle as O

pytestmark = pytest.mark.gpu

TOL = 2e-2

if torch.cuda.is_available():
    import gpu_harness as H
    from combine_route_scan_gb300 import build as B
    from combine_route_scan_gb300 import moe as M
    B.build()


def run_ffn(wl, inp, ws=None):
    dev = H.device_inputs(wl, inp)
    w = {k: H.to_dev(inp[k], WL.X_BF16) for k in ("w_gate", "w_up", "w_down")}
    cfg = H.make_cfg(wl, ffn_intermediate=wl.ffn_intermediate)
    if ws is None:
        ws = M.alloc_workspace(cfg)
    x_out = torch.empty_like(dev["x"])
    x_out.view(torch.uint8).fill_(0x7F)
    M.dispatch_ffn_combine(cfg, dev["x"], dev["expert_ids"], dev["active_mask"], dev["expert_scales"],
                           w["w_gate"], w["w_up"], w["w_down"], x_out, ws)
    st = M.get_device_status(ws)
    assert st == 0, M.STATUS.get(st, st)
    return WL.bf16_bits_to_fp32(H.to_host(x_out)).astype(np.float64).reshape(-1, wl.h), ws


def oracle_tokens(wl, inp, tokens):
    """The unchanged fp64 oracle on slices of `tokens`, one slice a host thread
    (the C call lets go of the interpreter lock), concatenated in order."""
    n = max(1, min(len(tokens) // 16, os.cpu_count() or 1))
    parts = [p for p in np.array_split(np.asarray(tokens, dtype=np.int64), n) if len(p)]
    with cf.ThreadPoolExecutor(max_workers=len(parts)) as ex:
        outs = list(ex.map(lambda p: O.moe_ffn_tokens(wl, inp, p), parts))
    return np.concatenate(outs, axis=0)


def check(wl, inp, tokens):
    got, _ = run_ffn(wl, inp)
    ref = oracle_tokens(wl, inp, tokens)
    g = got[tokens]
    scale = max(float(np.abs(ref).max()), 1e-30)
    err = float(np.abs(g - ref).max())
    assert np.isfinite(g).all()
    assert err <= TOL * scale, f"max abs err {err} vs {TOL} * {scale}"
    return err / scale


def test_ffn_small_all_tokens():
    wl = WL.Workload("ffn_small", 4, 16, 256, 2, 8, WL.X_BF16, zero_expert_num=1, copy_expert_num=1,
                     mask_kind=2, special_p=0.15, mask_false_p=0.1, ffn_intermediate=128, seed=21)
    inp = WL.make_inputs(wl)
    check(wl, inp, np.arange(wl.ep_world_size * wl.bs))


def test_ffn_expert_with_several_token_passes():
    """One expert receives every token (192 rows): three 64-token MMA passes."""
    wl = WL.Workload("ffn_hot", 2, 96, 256, 2, 4, WL.X_BF16, ffn_intermediate=256, seed=22)
    inp = WL.make_inputs(wl)
    ids = inp["expert_ids"]
    ids[..., 0] = 0
    ids[..., 1] = np.where(ids[..., 1] == 0, 1 + (np.arange(ids.shape[1]) % 3)[None, :], ids[..., 1])
    check(wl, inp, np.arange(wl.ep_world_size * wl.bs))


def test_ffn_decode_layer_all_tokens():
    """The decode MoE layer (8 ranks x 64 tokens, h 2048, 128 experts, top-8,
    intermediate 512): every one of the 512 tokens against the fp64 oracle,
    and every expert's rows are among those compared (each expert's tiles and
    the cooperative grid's gate/up -> down hand-off are all checked)."""
    wl = WL.WORKLOADS["w8_bs64_h2048_k8_e128_bf16_ffn"]
    inp = WL.make_inputs(wl)
    ids = inp["expert_ids"].reshape(-1)
    assert np.array_equal(np.unique(ids[ids < wl.moe_expert_num]), np.arange(wl.moe_expert_num))
    check(wl, inp, np.arange(wl.ep_world_size * wl.bs))


def test_ffn_many_tokens_per_scatter_cta():
    """More tokens than the dispatch scatter's resident CTAs hold in their
    rings, so most tokens are handed out by the workspace ticket counter."""
    wl = WL.Workload("ffn_many", 8, 1024, 256, 2, 16, WL.X_BF16, ffn_intermediate=128, seed=24)
    inp = WL.make_inputs(wl)
    check(wl, inp, np.arange(wl.ep_world_size * wl.bs))


def test_ffn_deterministic():
    wl = WL.Workload("ffn_det", 4, 32, 512, 4, 16, WL.X_BF16, ffn_intermediate=256, seed=23)
    inp = WL.make_inputs(wl)
    a, ws = run_ffn(wl, inp)
    b, _ = run_ffn(wl, inp, ws=ws)
    assert np.array_equal(a, b)


def test_ffn_unsupported_shapes():
    wl = WL.Workload("ffn_bad", 2, 4, 256, 2, 4, WL.X_FP16, ffn_intermediate=128)
    cfg = H.make_cfg(wl, ffn_intermediate=128)
    t = torch.zeros(64, dtype=torch.float16, device="cuda")
    with pytest.raises(M.MoeError) as ei:
        M.dispatch_ffn_combine(cfg, t, t, None, t, t, t, t, t, ws=torch.zeros(1 << 20, dtype=torch.uint8,
                                                                               device="cuda"))
    assert ei.value.name in ("UNSUPPORTED", "WORKSPACE")
    cfg = H.make_cfg(wl.with_(x_dtype=WL.X_BF16), ffn_intermediate=96)  # not a multiple of 128
    with pytest.raises(M.MoeError) as ei:
        M.dispatch_ffn_combine(cfg, t, t, None, t, t, t, t, t, ws=torch.zeros(1 << 20, dtype=torch.uint8,
                                                                               device="cuda"))
    assert ei.value.name == "UNSUPPORTED"


def test_ffn_call_replays_from_a_cuda_graph():
    """The fused call (cooperative FFN kernel chained by programmatic
    dependent launch) captures into a CUDA graph; replays give the eager
    call's bytes."""
    wl = WL.Workload("ffn_graph", 4, 32, 512, 4, 16, WL.X_BF16, ffn_intermediate=256, seed=25)
    inp = WL.make_inputs(wl)
    eager, _ = run_ffn(wl, inp)
    dev = H.device_inputs(wl, inp)
    w = {k: H.to_dev(inp[k], WL.X_BF16) for k in ("w_gate", "w_up", "w_down")}
    cfg = H.make_cfg(wl, ffn_intermediate=wl.ffn_intermediate)
    ws = M.alloc_workspace(cfg)
    x_out = torch.empty_like(dev["x"])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=torch.cuda.Stream()):
        M.dispatch_ffn_combine(cfg, dev["x"], dev["expert_ids"], dev["active_mask"], dev["expert_scales"],
                               w["w_gate"], w["w_up"], w["w_down"], x_out, ws)
    for _ in range(2):
        x_out.view(torch.uint8).fill_(0x7F)
        graph.replay()
        torch.cuda.synchronize()
        assert M.get_device_status(ws) == 0
        got = WL.bf16_bits_to_fp32(H.to_host(x_out)).astype(np.float64).reshape(-1, wl.h)
        assert np.array_equal(got, eager)
