"""Dispatch with quantMode 1 (static int8), 2 with per-expert smoothing, 3
(per-group FP8) and 4 (MX FP8 / FP4) on the GPU against the oracle: expand_x
codes, dynamic scales (fp32 bits / E8M0 bytes), assist_info and the receive
counts are compared byte for byte (both sides round the same fp32 values to
nearest even, so every code is unique)."""
import numpy as np
import pytest
import torch

import workloads as WL
from oracle import oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gpu_harness as H
    from combine_route_scan_gb300 import build as B
    from combine_route_scan_gb300 import moe as M
    B.build()

# (quant_mode, expand type, scales kind)
MODES = [(1, "", 1), (1, "", 2), (1, "", 3), (2, "", 3), (3, "fp8_e4m3", 0), (3, "fp8_e5m2", 0),
         (3, "fp8_e4m3", 3), (4, "fp8_e4m3", 0), (4, "fp8_e5m2", 0), (4, "fp4_e2m1", 0)]
# the modes with per-expert smoothing and a data-dependent scale (the expert-major kernel)
PE_MODES = [(2, "", 3), (3, "fp8_e4m3", 3), (3, "fp8_e5m2", 3)]


def mode_id(m):
    return f"q{m[0]}_{m[1] or 'int8'}_s{m[2]}"


def run(wl, plane_policy=M.PLANE_RULE if torch.cuda.is_available() else 0, bulk_min_bytes=None):
    inp = WL.make_inputs(wl)
    ref = O.dispatch(wl, inp)
    dev = H.device_inputs(wl, inp)
    kw = {} if bulk_min_bytes is None else {"bulk_min_bytes": bulk_min_bytes}
    got, ws, _ = H.gpu_dispatch(wl, dev, plane_policy=plane_policy, **kw)
    H.compare_dispatch(wl, got, ref)
    return got, ref


@pytest.mark.parametrize("mode", MODES, ids=mode_id)
@pytest.mark.parametrize("dt", [WL.X_BF16, WL.X_FP16])
def test_quant_small_tma_rows(mode, dt):
    """h = 256: TMA rows, several tokens per CTA, masks and special experts."""
    q, y, k = mode
    wl = WL.Workload("qs", 4, 16, 256, 4, 16, dt, zero_expert_num=1, copy_expert_num=1, mask_kind=2,
                     special_p=0.1, mask_false_p=0.1, quant_mode=q, y_dtype=y, scales_kind=k, seed=31)
    run(wl)


@pytest.mark.parametrize("mode", MODES, ids=mode_id)
def test_quant_bulk_plane(mode):
    """Every remote segment on the TMA bulk plane (rows leave from the shared
    quantised-row buffers by bulk copies)."""
    q, y, k = mode
    wl = WL.Workload("qb", 4, 32, 512, 4, 8, WL.X_BF16, ids="zipf", quant_mode=q, y_dtype=y, scales_kind=k, seed=32)
    run(wl, plane_policy=M.PLANE_BULK_ALL)


@pytest.mark.parametrize("mode", MODES, ids=mode_id)
def test_quant_ragged_rows(mode):
    """h = 200 (partial last group / block; rows that are not 16-byte
    multiples go by plain stores) and h = 12 fp16."""
    q, y, k = mode
    for h, dt in ((200, WL.X_BF16), (12, WL.X_FP16)):
        wl = WL.Workload("qr", 4, 9, h, 3, 8, dt, mask_kind=1, quant_mode=q, y_dtype=y, scales_kind=k, seed=33)
        run(wl)


@pytest.mark.parametrize("mode", [(2, "", 3), (3, "fp8_e4m3", 0), (3, "fp8_e5m2", 3), (4, "fp4_e2m1", 0),
                                  (4, "fp8_e4m3", 0), (1, "", 3)], ids=mode_id)
def test_quant_decode_shape(mode):
    """The perf shape of the combine README (W8 bs32 h7168 K8, 8 experts per
    rank), every row compared."""
    q, y, k = mode
    wl = WL.WORKLOADS["w8_bs32_h7168_k8_e64_f16"].with_(quant_mode=q, y_dtype=y, scales_kind=k)
    run(wl)


@pytest.mark.parametrize("mode", [(2, "", 0), (3, "fp8_e4m3", 0), (3, "fp8_e5m2", 0), (4, "fp8_e4m3", 0),
                                  (4, "fp8_e5m2", 0), (4, "fp4_e2m1", 0)], ids=mode_id)
@pytest.mark.parametrize("h", [32, 48, 96, 1000, 2080])
def test_quant_direct_store_shapes(mode, h):
    """Every pick on the store plane, so every token's codes leave straight
    from registers: whole MX blocks a thread (FP4) or half blocks on lane pairs
    (FP8) when h is a multiple of 32, two vectors a thread for per-token int8
    and per-group FP8 when h / 8 is even (partial groups below 128 and at the
    row's end), the vector-a-thread forms or the shared buffer otherwise; 2080
    needs a second, partial pass over the CTA's threads."""
    q, y, k = mode
    wl = WL.Workload("qd", 4, 12, h, 4, 16, WL.X_FP16 if h == 1000 else WL.X_BF16, zero_expert_num=1,
                     mask_kind=2, special_p=0.1, mask_false_p=0.1, quant_mode=q, y_dtype=y, scales_kind=k,
                     seed=38)
    run(wl, plane_policy=M.PLANE_STORES_ONLY)


def test_quant_values_cover_the_ranges():
    """Scale the inputs so that FP8 E4M3 / MX blocks see saturation, subnormal
    codes and zero groups, then compare bytes."""
    wl = WL.Workload("qv", 2, 8, 384, 2, 4, WL.X_BF16, quant_mode=3, y_dtype="fp8_e4m3", seed=34)
    inp = WL.make_inputs(wl)
    x = WL.bf16_bits_to_fp32(inp["x"])
    x[0, 0, :128] = 0.0                       # a zero group
    x[0, 1, :] *= np.float32(1e-30)           # tiny values
    x[1, 2, 5] = np.float32(3e4)              # one huge outlier per group
    inp["x"] = WL.fp32_to_bf16_bits(x)
    for q, y in ((3, "fp8_e4m3"), (3, "fp8_e5m2"), (4, "fp8_e4m3"), (4, "fp4_e2m1"), (4, "fp8_e5m2")):
        w = wl.with_(quant_mode=q, y_dtype=y)
        ref = O.dispatch(w, inp)
        dev = H.device_inputs(w, inp)
        got, _, _ = H.gpu_dispatch(w, dev)
        H.compare_dispatch(w, got, ref)


def _to_input_type(x: np.ndarray, dt: str) -> np.ndarray:
    x = x.astype(np.float32)
    return x.astype(np.float16) if dt == WL.X_FP16 else WL.fp32_to_bf16_bits(x)


def _from_input_type(x: np.ndarray, dt: str) -> np.ndarray:
    return x.astype(np.float32) if dt == WL.X_FP16 else WL.bf16_bits_to_fp32(x)


@pytest.mark.parametrize("dt", [WL.X_BF16, WL.X_FP16])
@pytest.mark.parametrize("k", [0, 3])
def test_token_int8_ties_and_near_half_quotients(dt, k):
    """Per-token int8 where x / scale lands on or next to half-integers, the
    cases where rounding the quotient is most fragile. Even tokens: the row
    maximum is 127 * 2^j, so the scale is 2^j exactly, and every other element
    is (n + 1/2) * 2^j: exact ties, which round to even. Odd tokens: a random
    maximum, and elements the input type's nearest value to (n + 1/2) * scale
    for small n, so many quotients fall within 2^-14 of a half-integer
    without being one. With smoothing each expert's scales row is one power of
    two, which keeps the products on the same points. Bytes against the oracle."""
    W, bs, h, E = 2, 16, 512, 8
    wl = WL.Workload("qt", W, bs, h, 4, E, dt, quant_mode=2, scales_kind=k, seed=36)
    inp = WL.make_inputs(wl)
    rng = np.random.Generator(np.random.PCG64(360))
    x = np.zeros((W, bs, h), np.float32)
    for s in range(W):
        for t in range(bs):
            if t % 2 == 0:
                j = float(rng.integers(-4, 5))
                row = (rng.integers(-127, 127, size=h) + 0.5) * 2.0 ** j
                row[0] = 127.0 * 2.0 ** j
            else:
                amax = _from_input_type(_to_input_type(np.array([rng.uniform(1.0, 100.0)]), dt), dt)[0]
                scale = np.float32(amax) / np.float32(127.0)
                row = (rng.integers(-4, 4, size=h) + 0.5) * np.float64(scale)
                row[0] = amax
            x[s, t] = row
    inp["x"] = _to_input_type(x, dt)
    if k == 3:
        inp["quant_scales"] = np.repeat(2.0 ** rng.integers(-2, 3, size=(E, 1)), h, axis=1).astype(np.float32)

    # the case mix really is there: quotients within 2^-14 of a half-integer
    xf = _from_input_type(inp["x"], dt)
    amax = np.abs(xf).max(axis=2, keepdims=True)
    q = xf / (amax / np.float32(127.0))
    near = np.abs(np.abs(q - np.floor(q)) - np.float32(0.5)) <= np.float32(2.0 ** -14)
    assert near[:, 0::2].mean() > 0.9 and near[:, 1::2].sum() > 100

    ref = O.dispatch(wl, inp)
    dev = H.device_inputs(wl, inp)
    got, _, _ = H.gpu_dispatch(wl, dev)
    H.compare_dispatch(wl, got, ref)


@pytest.mark.parametrize("dt", [WL.X_BF16, WL.X_FP16])
@pytest.mark.parametrize("k", [0, 3])
@pytest.mark.parametrize("y", ["fp8_e4m3", "fp8_e5m2"])
def test_group_fp8_ties_and_near_midpoint_quotients(y, k, dt):
    """Per-group FP8 where x / scale lands on or next to a midpoint of two
    neighbouring FP8 values, the cases where rounding the quotient is most
    fragile. Each 128-element group's maximum is fmax * 2^j (scale 2^j
    exactly) and its other elements are (m + 1/2) * 2^(e - mbits) * 2^j, the
    format's midpoints: exact ties. With smoothing each expert's scales row is
    one value 1 + r * 2^-10, so the rounded products and the rounded scale
    move every quotient a few fp32 ulps off the midpoint. Bytes against the
    oracle."""
    W, bs, h, E = 2, 16, 512, 8
    fmax, mbits, e_top = (448.0, 3, 8) if y == "fp8_e4m3" else (57344.0, 2, 15)
    wl = WL.Workload("qg", W, bs, h, 4, E, dt, quant_mode=3, y_dtype=y, scales_kind=k, seed=37)
    inp = WL.make_inputs(wl)
    rng = np.random.Generator(np.random.PCG64(370))
    n_groups = h // 128
    x = np.zeros((W, bs, h), np.float64)
    for s in range(W):
        for t in range(bs):
            for g in range(n_groups):
                j = float(rng.integers(-3, 1))
                e = rng.integers(e_top - 6, e_top + 1, size=128)
                m = rng.integers(2 ** mbits, 2 ** (mbits + 1), size=128)
                mid = np.minimum((m + 0.5) * 2.0 ** (e - mbits), fmax) * rng.choice([-1.0, 1.0], size=128)
                mid[0] = fmax
                x[s, t, g * 128:(g + 1) * 128] = mid * 2.0 ** j
    inp["x"] = _to_input_type(x, dt)
    assert np.array_equal(_from_input_type(inp["x"], dt).astype(np.float64), x)  # exactly representable
    if k == 3:
        r = 1.0 + rng.integers(1, 1024, size=(E, 1)) * 2.0 ** -10
        inp["quant_scales"] = np.repeat(r, h, axis=1).astype(np.float32)

    ref = O.dispatch(wl, inp)
    dev = H.device_inputs(wl, inp)
    got, _, _ = H.gpu_dispatch(wl, dev)
    H.compare_dispatch(wl, got, ref)


def _fragile_rows(wl, inp, rng):
    """Every other token a row whose quotients sit on or next to rounding
    boundaries of the quantisation (exact half-integers for per-token int8 with
    power-of-two smoothing rows; FP8 midpoints moved a few fp32 ulps by
    smoothing rows 1 + r * 2^-10 for per-group FP8); the other tokens keep
    their random values."""
    W, bs, h, E, dt = wl.ep_world_size, wl.bs, wl.h, wl.moe_expert_num, wl.x_dtype
    x = _from_input_type(inp["x"], dt).astype(np.float64).reshape(W, bs, h)
    for s in range(W):
        for t in range(0, bs, 2):
            if wl.quant_mode == 2:
                j = float(rng.integers(-4, 5))
                row = (rng.integers(-127, 127, size=h) + 0.5) * 2.0 ** j
                row[0] = 127.0 * 2.0 ** j
            else:
                fmax, mbits, e_top = (448.0, 3, 8) if wl.y_dtype == "fp8_e4m3" else (57344.0, 2, 15)
                row = np.empty(h)
                for g0 in range(0, h, 128):
                    n = min(128, h - g0)
                    e = rng.integers(e_top - 6, e_top + 1, size=n)
                    m = rng.integers(2 ** mbits, 2 ** (mbits + 1), size=n)
                    mid = np.minimum((m + 0.5) * 2.0 ** (e - mbits), fmax) * rng.choice([-1.0, 1.0], size=n)
                    mid[0] = fmax
                    row[g0:g0 + n] = mid * 2.0 ** float(rng.integers(-3, 1))
            x[s, t] = row
    inp["x"] = _to_input_type(x, dt)
    if wl.quant_mode == 2:
        inp["quant_scales"] = np.repeat(2.0 ** rng.integers(-2, 3, size=(E, 1)), h, axis=1).astype(np.float32)
    else:
        r = 1.0 + rng.integers(1, 1024, size=(E, 1)) * 2.0 ** -10
        inp["quant_scales"] = np.repeat(r, h, axis=1).astype(np.float32)


@pytest.mark.parametrize("mode", PE_MODES, ids=mode_id)
@pytest.mark.parametrize("policy", ["rule", "bulk"])
def test_quant_per_expert_deferred_exact_codes(mode, policy):
    """The expert-major kernel's exact path: rows whose quotients sit on
    rounding boundaries make most of their threads queue for the IEEE
    division after the CTA's last row, enough to overflow the queue (every
    row from there recomputed whole), mixed with random rows; store and bulk
    planes, ready flags and per-rank times on. Bytes against the oracle, every
    segment's flag set, status OK."""
    q, y, k = mode
    wl = WL.Workload("qdx", 4, 256, 2048, 4, 32, WL.X_BF16, mask_kind=2, mask_false_p=0.1, ids="zipf",
                     quant_mode=q, y_dtype=y, scales_kind=k, seed=88)
    inp = WL.make_inputs(wl)
    _fragile_rows(wl, inp, np.random.Generator(np.random.PCG64(880)))
    ref = O.dispatch(wl, inp)
    dev = H.device_inputs(wl, inp)
    L = wl.moe_expert_num // wl.ep_world_size
    cfg = H.make_cfg(wl, plane_policy=M.PLANE_RULE if policy == "rule" else M.PLANE_BULK_ALL,
                     bulk_min_bytes=0 if policy == "rule" else M.BULK_MIN_BYTES)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_dispatch_outputs(cfg, H.TORCH_DT[wl.x_dtype])
    flags = torch.zeros((wl.ep_world_size, L * wl.ep_world_size), dtype=torch.int32, device="cuda")
    perf = torch.zeros(wl.ep_world_size, dtype=torch.int64, device="cuda")
    c = M.with_performance_info(M.with_seg_ready(cfg, flags, 9), perf)
    M.dispatch(c, dev["x"], dev["expert_ids"], dev["active_mask"], dev["expert_scales"], out["expand_x"],
               out["dynamic_scales"], out["assist_info"], out["ep_recv_count"], out["expand_scales"], None, ws,
               scales=dev["quant_scales"])
    assert M.get_device_status(ws) == 0
    assert bool((flags == 9).all())
    assert bool((perf >= 0).all())
    H.compare_dispatch(wl, out, ref)


def test_quant_ready_flags_and_performance_info():
    """The quantising scatter publishes ready flags and per-rank times too."""
    wl = WL.Workload("qf", 4, 24, 512, 4, 16, WL.X_BF16, quant_mode=3, y_dtype="fp8_e4m3", scales_kind=3, seed=35)
    inp = WL.make_inputs(wl)
    ref = O.dispatch(wl, inp)
    dev = H.device_inputs(wl, inp)
    L = wl.moe_expert_num // wl.ep_world_size
    for policy in (M.PLANE_RULE, M.PLANE_BULK_ALL):
        cfg = H.make_cfg(wl, plane_policy=policy)
        ws = M.alloc_workspace(cfg)
        out = M.alloc_dispatch_outputs(cfg, H.TORCH_DT[wl.x_dtype])
        flags = torch.zeros((wl.ep_world_size, L * wl.ep_world_size), dtype=torch.int32, device="cuda")
        perf = torch.zeros(wl.ep_world_size, dtype=torch.int64, device="cuda")
        c = M.with_performance_info(M.with_seg_ready(cfg, flags, 5), perf)
        M.dispatch(c, dev["x"], dev["expert_ids"], dev["active_mask"], dev["expert_scales"], out["expand_x"],
                   out["dynamic_scales"], out["assist_info"], out["ep_recv_count"], out["expand_scales"], None, ws,
                   scales=dev["quant_scales"])
        assert M.get_device_status(ws) == 0
        assert bool((flags == 5).all())
        assert bool((perf >= 0).all())
        H.compare_dispatch(wl, out, ref)


def test_quant_argument_errors():
    wl = WL.Workload("qe", 2, 4, 64, 2, 4, WL.X_BF16, quant_mode=1, scales_kind=2, seed=36)
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    cfg = H.make_cfg(wl)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_dispatch_outputs(cfg, torch.bfloat16)
    args = (dev["x"], dev["expert_ids"], None, dev["expert_scales"], out["expand_x"], None, out["assist_info"],
            out["ep_recv_count"], None, None, ws)
    with pytest.raises(M.MoeError) as ei:  # scales declared but not passed
        M.dispatch(cfg, *args)
    assert ei.value.name == "INVALID_ARG"
    buf = torch.zeros(80, dtype=torch.float32, device="cuda")
    with pytest.raises(M.MoeError) as ei:  # scales not 16-byte aligned
        M.dispatch(cfg, *args, scales=buf[1:65])
    assert ei.value.name == "INVALID_ARG"
    M.dispatch(cfg, *args, scales=buf[4:68])
    assert M.get_device_status(ws) == 0


@pytest.mark.parametrize("seed", range(24))
def test_quant_random_shapes(seed):
    """Random shapes (ragged and TMA rows, 1D / 2D masks, zero / copy experts),
    a random quantised mode, element type and scales input, a random plane
    policy: every routed row's codes and dynamic scales byte for byte."""
    rng = np.random.default_rng(7000 + seed)
    q, y, k = MODES[int(rng.integers(0, len(MODES)))]
    W = int(rng.integers(2, 7))
    L = int(rng.integers(1, 5))
    K = int(rng.integers(1, min(W * L, 8) + 1))
    h = int(rng.choice([16, 32, 48, 96, 130, 256, 384, 1000, 2048]))
    if y == "fp4_e2m1" and h % 2:
        h += 1
    wl = WL.Workload(f"qrand{seed}", W, int(rng.integers(1, 24)), h, K, W * L,
                     WL.X_BF16 if rng.random() < 0.5 else WL.X_FP16,
                     zero_expert_num=int(rng.integers(0, 3)), copy_expert_num=int(rng.integers(0, 3)),
                     mask_kind=int(rng.integers(0, 3)), special_p=0.2, mask_false_p=0.2,
                     ids="zipf" if rng.random() < 0.5 else "uniform",
                     quant_mode=q, y_dtype=y, scales_kind=k, seed=int(rng.integers(0, 2**31)))
    policy = [M.PLANE_RULE, M.PLANE_STORES_ONLY, M.PLANE_BULK_ALL][int(rng.integers(0, 3))]
    run(wl, plane_policy=policy, bulk_min_bytes=0 if policy == M.PLANE_RULE else None)


@pytest.mark.parametrize("mode", [(2, "", 3), (3, "fp8_e5m2", 3), (4, "fp4_e2m1", 0), (1, "", 2)], ids=mode_id)
def test_quant_top32(mode):
    """The largest top-k: 32 picks per token, a variant per pick with
    per-expert scales, every plane policy."""
    q, y, k = mode
    wl = WL.Workload("qk32", 4, 12, 512, 32, 64, WL.X_BF16, mask_kind=2, mask_false_p=0.1, quant_mode=q,
                     y_dtype=y, scales_kind=k, seed=51)
    for policy in (M.PLANE_RULE, M.PLANE_BULK_ALL):
        run(wl, plane_policy=policy, bulk_min_bytes=0)


# Every quantising-scatter instantiation the tests and the bench run, plus the
# per-token int8 form without scales.
ALL_MODES = MODES + [(2, "", 0)]


def _resident_limit():
    """An upper bound on the quantising scatter's resident grid: 8 CTAs of 256
    threads per SM (2048 threads, the SM's limit)."""
    return torch.cuda.get_device_properties(0).multi_processor_count * 8


def _many_tokens_workload(mode, dt, seed):
    q, y, k = mode
    return WL.Workload("qmany", 8, 1024, 256, 4, 32, dt, zero_expert_num=2, copy_expert_num=2, mask_kind=2,
                       special_p=0.1, mask_false_p=0.1, ids="zipf", quant_mode=q, y_dtype=y, scales_kind=k,
                       seed=seed)


@pytest.mark.parametrize("mode", ALL_MODES, ids=mode_id)
@pytest.mark.parametrize("policy", ["rule", "bulk"])
def test_quant_many_tokens_per_cta(mode, policy):
    """8192 tokens against at most 8 CTAs per SM: every CTA of the quantising
    scatter takes several tokens in turn, so the source-row ring reuses its
    slots with the barrier parity flipped, warp 0 loads destination lists one
    and two tokens ahead, the rows of token i-1 are counted while token i is
    quantised, and the two shared quantised-row buffers alternate. Zipf
    routing with masks and zero / copy experts; the page's rule with a zero
    size threshold (every above-mean remote segment by bulk copies) or every
    remote segment by bulk copies. Codes, dynamic scales, assist_info,
    expand_scales and counts byte for byte."""
    dt = WL.X_BF16 if policy == "rule" else WL.X_FP16
    wl = _many_tokens_workload(mode, dt, 41 + ALL_MODES.index(mode))
    assert wl.ep_world_size * wl.bs >= 4 * _resident_limit()
    if policy == "rule":
        run(wl, plane_policy=M.PLANE_RULE, bulk_min_bytes=0)
    else:
        run(wl, plane_policy=M.PLANE_BULK_ALL)


@pytest.mark.parametrize("mode", [(2, "", 0), (4, "fp4_e2m1", 0), (3, "fp8_e4m3", 3)], ids=mode_id)
def test_quant_many_tokens_ready_flags_and_performance_info(mode):
    """The multi-token path with ready flags and performance info on: every
    segment flagged with the call's ticket, per-rank times positive, outputs
    still byte-exact."""
    wl = _many_tokens_workload(mode, WL.X_BF16, 60)
    inp = WL.make_inputs(wl)
    ref = O.dispatch(wl, inp)
    dev = H.device_inputs(wl, inp)
    L = wl.moe_expert_num // wl.ep_world_size
    cfg = H.make_cfg(wl, plane_policy=M.PLANE_RULE, bulk_min_bytes=0)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_dispatch_outputs(cfg, H.TORCH_DT[wl.x_dtype])
    for t in out.values():
        if t is not None:
            t.view(torch.uint8).fill_(0xA5)
    flags = torch.zeros((wl.ep_world_size, L * wl.ep_world_size), dtype=torch.int32, device="cuda")
    perf = torch.zeros(wl.ep_world_size, dtype=torch.int64, device="cuda")
    c = M.with_performance_info(M.with_seg_ready(cfg, flags, 11), perf)
    M.dispatch(c, dev["x"], dev["expert_ids"], dev["active_mask"], dev["expert_scales"], out["expand_x"],
               out["dynamic_scales"], out["assist_info"], out["ep_recv_count"], out["expand_scales"], None, ws,
               scales=dev["quant_scales"])
    assert M.get_device_status(ws) == 0
    assert bool((flags == 11).all()), int((flags != 11).sum())
    assert bool((perf > 0).all()), perf
    H.compare_dispatch(wl, out, ref)


@pytest.mark.parametrize("mode", [(2, "", 0), (3, "fp8_e4m3", 0), (2, "", 3), (3, "fp8_e4m3", 3), (4, "fp4_e2m1", 0)],
                         ids=mode_id)
def test_quant_full_size_bench_workload(mode):
    """The bench workload (16 ranks, 256 tokens each, h 7168, top-8 of 256
    Zipf-routed experts, 2D mask, zero and copy experts): 4096 tokens, about
    5 per resident CTA, every routed row's codes and dynamic scales byte for
    byte against the oracle, and the planes the page's rule gives to the
    quantised row sizes (int8 and FP8 rows of 7168 bytes, packed FP4 of 3584:
    no segment reaches 2 MiB) are the oracle's."""
    q, y, k = mode
    wl = WL.WORKLOADS["w16_bs256_h7168_k8_e256_bf16_zipf"].with_(quant_mode=q, y_dtype=y, scales_kind=k)
    got, ref = run(wl)
    assert np.array_equal(H.to_host(got["seg_plane"]), O.dispatch_plane(wl, ref["ep_recv_count"]))


@pytest.mark.parametrize("mode", PE_MODES, ids=mode_id)
@pytest.mark.parametrize("policy", ["rule", "bulk"])
def test_quant_per_expert_wide_rows(mode, policy):
    """Per-token int8 and per-group FP8 with per-expert smoothing on rows wider
    than the expert-major kernel holds (h 16640 > 15360 elements): the
    token-major kernel quantises them, a warp a pick; more tokens than
    resident CTAs."""
    q, y, k = mode
    wl = WL.Workload("qwide", 4, 256, 16640, 4, 16, WL.X_BF16, zero_expert_num=1, copy_expert_num=1, mask_kind=2,
                     special_p=0.05, mask_false_p=0.1, ids="zipf", quant_mode=q, y_dtype=y, scales_kind=k, seed=81)
    if policy == "rule":
        run(wl, plane_policy=M.PLANE_RULE, bulk_min_bytes=0)
    else:
        run(wl, plane_policy=M.PLANE_BULK_ALL)


@pytest.mark.parametrize("mode", PE_MODES, ids=mode_id)
@pytest.mark.parametrize("dt", [WL.X_FP16, WL.X_BF16])
def test_quant_per_expert_expert_major_shapes(mode, dt):
    """The expert-major kernel (per-token int8 and per-group FP8 with
    per-expert smoothing) at shapes that exercise its row list and CTA
    sizing: h 15360 (the widest row it takes: 15 warps and the producer, 512
    threads), h 9216 (9 warps, 4 vectors a thread), h 8192 (8 warps), h 1008
    (one warp, a partial last group, vectors past the row's end), a run of
    receive rows longer than one 256-entry list chunk per CTA (16 ranks x 2048
    tokens), fp16 and bf16 input; bulk plane for every remote segment above
    zero bytes."""
    q, y, k = mode
    for h, W, bs in ((15360, 2, 64), (9216, 4, 64), (8192, 4, 64), (1008, 4, 96), (256, 16, 2048)):
        wl = WL.Workload(f"qpe_h{h}", W, bs, h, 4, 32, dt, mask_kind=2, mask_false_p=0.1, ids="zipf",
                         quant_mode=q, y_dtype=y, scales_kind=k, seed=82 + h)
        run(wl, plane_policy=M.PLANE_RULE, bulk_min_bytes=0)
