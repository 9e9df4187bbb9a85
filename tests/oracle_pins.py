"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function raises AssertionError (or OracleError) when the oracle
disagrees with:
  * hand-worked fixtures under tests/golden/ (each cites the page it follows);
  * a sort-based brute force of the dispatch layout, written independently of
    the oracle's counting sort;
  * closed forms (identity expert: x_out = x * sum of contributing weights);
  * invariants (counts, bijection of assist_info onto the routed picks);
  * exact rational arithmetic with IEEE round-to-nearest-even (quantisers of
    every quantMode), with FP8 / FP4 codes found by brute force over each
    format's table decoded from its definition;
  * library routines (numpy float16 and torch bfloat16 / float8 conversions,
    torch fp64 matmul and silu for the SwiGLU expert).
They are plain functions so that tests/test_oracle_mutants.py can rerun them
against deliberately broken builds of the oracle.
"""
from __future__ import annotations

import json
import math
import os
import struct
from fractions import Fraction

import numpy as np

import workloads as WL
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


# ------------------------------------------------------------------ helpers

def brute_force_layout(wl: WL.Workload, inp: dict):
    """Dispatch layout by sorting: every routed pick becomes the key
    (rank d, local expert le, source s, token t, topk k); sorted keys give the
    rows of each rank, and counting keys per (le, s) gives the segment sizes."""
    W, bs, K, E = wl.ep_world_size, wl.bs, wl.topk, wl.moe_expert_num
    L = E // W
    ids = inp["expert_ids"]
    mask = inp.get("active_mask")
    keys = []
    for s in range(W):
        for t in range(bs):
            for k in range(K):
                if mask is not None:
                    act = mask[s, t] if mask.ndim == 2 else mask[s, t, k]
                    if not act:
                        continue
                e = int(ids[s, t, k])
                if 0 <= e < E:
                    keys.append((e // L, e % L, s, t, k))
    keys.sort()
    rows = [[] for _ in range(W)]
    seg = np.zeros((W, L * W), dtype=np.int64)
    for d, le, s, t, k in keys:
        rows[d].append((s, t, k))
        seg[d, le * W + s] += 1
    return rows, seg


def contributing_weight_sum(wl: WL.Workload, inp: dict) -> np.ndarray:
    """Sum over picks that are active and routed or copy (int64 / float64)."""
    ids = inp["expert_ids"].astype(np.int64)
    E, Z, C = wl.moe_expert_num, wl.zero_expert_num, wl.copy_expert_num
    contrib = (ids >= 0) & (ids < E)
    contrib |= (ids >= E + Z) & (ids < E + Z + C)
    mask = inp.get("active_mask")
    if mask is not None:
        m = mask.astype(bool)
        contrib &= m[..., None] if m.ndim == 2 else m
    w = inp["expert_scales"]
    if w.dtype == np.int32:
        return (w.astype(np.int64) * contrib).sum(-1)
    return (w.astype(np.float64) * contrib).sum(-1)


def rn_f32(q: Fraction) -> Fraction:
    """Round a rational to the nearest fp32 value, ties to even (normal range)."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    assert e >= -126, "subnormal results are outside this helper"
    ulp = Fraction(2) ** (e - 23)
    n = a / ulp
    fl = n.numerator // n.denominator
    r = n - fl
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def round_half_even(q: Fraction) -> int:
    fl = math.floor(q)
    r = q - fl
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return int(fl)


def f32_bits(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0]


def quantize_exact(values) -> tuple:
    """quantMode 2 by exact rational arithmetic: returns (q list, scale)."""
    xs = [Fraction(float(v)) for v in values]
    amax = max(abs(v) for v in xs)
    if amax == 0:
        return [0] * len(xs), Fraction(0)
    scale = rn_f32(amax / 127)
    q = []
    for v in xs:
        r = round_half_even(rn_f32(v / scale)) if v != 0 else 0
        q.append(max(-127, min(127, r)))
    return q, scale


# small float formats, decoded from their definitions (sign, biased
# exponent, mantissa with an implicit leading one; exponent field 0 is
# subnormal). E4M3 reserves S.1111.111 for NaN and has no infinity; E5M2
# reserves exponent 31 for inf / NaN; E2M1 has neither.
MINIFLOAT = {
    "fp8_e4m3": dict(eb=4, mb=3, bias=7, emax=8, nonfinite=lambda E, M: E == 15 and M == 7),
    "fp8_e5m2": dict(eb=5, mb=2, bias=15, emax=15, nonfinite=lambda E, M: E == 31),
    "fp4_e2m1": dict(eb=2, mb=1, bias=1, emax=2, nonfinite=lambda E, M: False),
}


def minifloat_table(fmt: str):
    """Sorted [(value, code)] of the non-negative finite values of a format."""
    f = MINIFLOAT[fmt]
    out = []
    for code in range(1 << (f["eb"] + f["mb"])):
        E, M = code >> f["mb"], code & ((1 << f["mb"]) - 1)
        if f["nonfinite"](E, M):
            continue
        if E == 0:
            v = Fraction(M, 1 << f["mb"]) * Fraction(2) ** (1 - f["bias"])
        else:
            v = (1 + Fraction(M, 1 << f["mb"])) * Fraction(2) ** (E - f["bias"])
        out.append((v, code))
    return sorted(out)


def nearest_code(v, fmt: str, negative: bool = None) -> int:
    """Brute force: the code of the representable value nearest to v (an exact
    Fraction or a float), ties to the even code, saturating at the largest
    finite value; the sign bit follows v's sign (negative=True for -0.0)."""
    f = MINIFLOAT[fmt]
    table = minifloat_table(fmt)
    a = abs(Fraction(v))
    if negative is None:
        negative = Fraction(v) < 0
    best = None
    for val, code in table:
        dist = abs(val - a)
        if best is None or dist < best[0] or (dist == best[0] and code % 2 == 0):
            best = (dist, code)
    code = table[-1][1] if a >= table[-1][0] else best[1]
    return code | ((1 << (f["eb"] + f["mb"])) if negative else 0)


def fmax_of(fmt: str) -> Fraction:
    return minifloat_table(fmt)[-1][0]


def row_values(row: np.ndarray, dt: str) -> list:
    return [float(v) for v in (row.astype(np.float64) if dt == "float16"
                               else WL.bf16_bits_to_fp32(row).astype(np.float64))]


def is_neg(v: float) -> bool:
    return math.copysign(1.0, v) < 0


def group_quant_exact(xs: list, fmt: str):
    """quantMode 3 on one row of fp32 values (already smoothed), exact
    arithmetic with IEEE rounding: (codes, scales)."""
    fm = fmax_of(fmt)
    codes, scales = [], []
    for g0 in range(0, len(xs), 128):
        grp = xs[g0:g0 + 128]
        amax = max(abs(Fraction(v)) for v in grp)
        if amax == 0:
            codes += [0] * len(grp)
            scales.append(Fraction(0))
            continue
        scale = rn_f32(amax / fm)
        scales.append(scale)
        for v in grp:
            if v == 0:
                codes.append(nearest_code(0, fmt, is_neg(v)))
            else:
                codes.append(nearest_code(rn_f32(Fraction(v) / scale), fmt, v < 0))
    return codes, scales


def mx_quant_exact(xs: list, fmt: str):
    """quantMode 4 (OCP MX) on one row: (codes, E8M0 bytes)."""
    emax = MINIFLOAT[fmt]["emax"]
    codes, scale_bytes = [], []
    for b0 in range(0, len(xs), 32):
        blk = xs[b0:b0 + 32]
        amax = max(abs(v) for v in blk)
        se = -127
        if amax > 0:
            se = max(-127, min(127, math.frexp(amax)[1] - 1 - emax))
        scale_bytes.append(se + 127)
        X = Fraction(2) ** se
        for v in blk:
            codes.append(nearest_code(Fraction(v) / X, fmt, is_neg(v)))
    return codes, scale_bytes


def unpack_fp4(q: np.ndarray) -> list:
    out = []
    for b in q.tolist():
        out += [b & 0xF, b >> 4]
    return out


# -------------------------------------------------------------------- pins

def pin_dispatch_combine_hand():
    g = golden("dispatch_hand.json")
    for case in g["cases"]:
        wl = WL.Workload(case["name"], case["W"], case["bs"], case["h"], case["K"], case["E"],
                         WL.X_INT32, zero_expert_num=case["Z"], copy_expert_num=case["C"],
                         mask_kind=case["mask_kind"])
        inp = {
            "x": np.array(case["x"], dtype=np.int32),
            "expert_ids": np.array(case["expert_ids"], dtype=np.int32),
            "expert_scales": np.array(case["expert_scales"], dtype=np.int32),
            "active_mask": (None if case["active_mask"] is None
                            else np.array(case["active_mask"], dtype=np.uint8)),
        }
        assert O.capacity(wl) == case["capacity"], case["name"]
        d = O.dispatch(wl, inp)
        assert d["ep_recv_count"].tolist() == case["ep_recv_count"], case["name"]
        for r in range(wl.ep_world_size):
            n = len(case["assist_info"][r])
            assert d["assist_info"][r, :n].tolist() == case["assist_info"][r], (case["name"], r)
            assert d["expand_x"][r, :n].tolist() == case["expand_x"][r], (case["name"], r)
        x_out = O.combine(wl, d["expand_x"], d["assist_info"], d["ep_recv_count"], inp)
        assert x_out.tolist() == case["x_out"], case["name"]
    for cc in g["capacity_cases"]:
        wl = WL.Workload("cap", cc["W"], cc["bs"], 16, cc["K"], cc["E"], WL.X_INT32)
        assert O.capacity(wl) == cc["A"], cc


def pin_layout_bruteforce(wl: WL.Workload, inp: dict):
    d = O.dispatch(wl, inp)
    rows, seg = brute_force_layout(wl, inp)
    assert np.array_equal(d["ep_recv_count"], np.cumsum(seg, axis=1)), "ep_recv_count"
    for r in range(wl.ep_world_size):
        n = len(rows[r])
        got = [tuple(v) for v in d["assist_info"][r, :n].tolist()]
        assert got == rows[r], f"assist_info of rank {r}"
    return d


def pin_invariants(wl: WL.Workload, inp: dict, d: dict):
    W, bs, K = wl.ep_world_size, wl.bs, wl.topk
    L = wl.moe_expert_num // W
    ep = d["ep_recv_count"].astype(np.int64)
    assert (np.diff(ep, axis=1) >= 0).all() and (ep[:, 0] >= 0).all(), "running counts"
    ids = inp["expert_ids"]
    mask = inp.get("active_mask")
    active = np.ones((W, bs, K), dtype=bool)
    if mask is not None:
        active = np.broadcast_to(mask.astype(bool)[..., None], active.shape) if mask.ndim == 2 \
            else mask.astype(bool)
    routed = active & (ids >= 0) & (ids < wl.moe_expert_num)
    assert int(ep[:, -1].sum()) == int(routed.sum()), "sum of counts = routed picks"
    seen = np.zeros((W, bs, K), dtype=np.int64)
    for r in range(W):
        n = int(ep[r, -1])
        assert n <= O.capacity(wl)
        for row in range(n):
            s, t, k = d["assist_info"][r, row]
            seen[s, t, k] += 1
            e = int(ids[s, t, k])
            assert e // L == r, "row lands on the rank that owns its expert"
            j = int(np.searchsorted(ep[r], row, side="right"))
            assert j == (e % L) * W + s, "row lies in segment (local expert, source)"
            if wl.quant_mode == 0:
                assert np.array_equal(d["expand_x"][r, row], inp["x"][s, t]), "payload row"
            if d.get("expand_scales") is not None:
                assert d["expand_scales"][r, row] == inp["expert_scales"][s, t, k]
    assert np.array_equal(seen, routed.astype(np.int64)), "assist_info is a bijection onto routed picks"


def pin_combine_closed_form_int(wl: WL.Workload, inp: dict, d: dict):
    """Identity expert: x_out = x * (sum of contributing weights), exactly."""
    assert wl.x_dtype == WL.X_INT32
    x_out = O.combine(wl, d["expand_x"], d["assist_info"], d["ep_recv_count"], inp)
    want = inp["x"].astype(np.int64) * contributing_weight_sum(wl, inp)[..., None]
    assert np.array_equal(x_out.astype(np.int64), want), "closed form x * sum(w)"


def pin_combine_gather(wl: WL.Workload, inp: dict, d: dict, seed: int = 7):
    """Non-identity expert: give every expert-output row its own random values;
    x_out must be the weighted sum of the rows the brute-force layout assigns."""
    assert wl.x_dtype == WL.X_INT32
    rng = np.random.default_rng(seed)
    y = rng.integers(-50, 51, size=d["expand_x"].shape, dtype=np.int32)
    rows, _ = brute_force_layout(wl, inp)
    x_out = O.combine(wl, y, d["assist_info"], d["ep_recv_count"], inp)
    W, bs, K, h = wl.ep_world_size, wl.bs, wl.topk, wl.h
    E, Z, C = wl.moe_expert_num, wl.zero_expert_num, wl.copy_expert_num
    want = np.zeros((W, bs, h), dtype=np.int64)
    where = {}
    for r in range(W):
        for row, key in enumerate(rows[r]):
            where[key] = (r, row)
    mask = inp.get("active_mask")
    for s in range(W):
        for t in range(bs):
            for k in range(K):
                if mask is not None and not (mask[s, t] if mask.ndim == 2 else mask[s, t, k]):
                    continue
                e = int(inp["expert_ids"][s, t, k])
                w = int(inp["expert_scales"][s, t, k])
                if e < E:
                    r, row = where[(s, t, k)]
                    want[s, t] += w * y[r, row].astype(np.int64)
                elif E + Z <= e < E + Z + C:
                    want[s, t] += w * inp["x"][s, t].astype(np.int64)
    assert np.array_equal(x_out.astype(np.int64), want), "gather by assist_info"


def pin_combine_closed_form_float(wl: WL.Workload, inp: dict, d: dict):
    """Identity expert, float data: x_out = round(x * sum(w)) up to fp32
    accumulation error (a few fp32 ulps before the final rounding)."""
    x_out = O.combine(wl, d["expand_x"], d["assist_info"], d["ep_recv_count"], inp)
    if wl.x_dtype == WL.X_FP16:
        xf = inp["x"].astype(np.float64)
        got = x_out.astype(np.float64)
        ulp_rel = 2.0 ** -10
    else:
        xf = WL.bf16_bits_to_fp32(inp["x"]).astype(np.float64)
        got = WL.bf16_bits_to_fp32(x_out).astype(np.float64)
        ulp_rel = 2.0 ** -7
    want = xf * contributing_weight_sum(wl, inp)[..., None]
    err = np.abs(got - want)
    bound = np.abs(want) * ulp_rel + 1e-6 * np.abs(xf) * wl.topk + 2.0 ** -24
    assert (err <= bound).all(), f"max err {err.max()}"


def pin_combine_order_hand():
    g = golden("combine_order_hand.json")
    wl = WL.Workload("order", g["W"], g["bs"], g["h"], g["K"], g["E"], WL.X_FP16,
                     copy_expert_num=g["C"])
    inp = {
        "x": np.array(g["x_fp16_bits"], dtype=np.uint16).view(np.float16),
        "expert_ids": np.array(g["expert_ids"], dtype=np.int32),
        "expert_scales": np.array([[[int(b, 16) for b in tk] for tk in r] for r in g["expert_scales_f32_bits"]],
                                  dtype=np.uint32).view(np.float32),
        "active_mask": None,
    }
    d = O.dispatch(wl, inp)
    x_out = O.combine(wl, d["expand_x"], d["assist_info"], d["ep_recv_count"], inp)
    assert x_out.view(np.uint16).tolist() == g["x_out_fp16_bits"], x_out.view(np.uint16).tolist()


def pin_quant_hand():
    g = golden("quant_hand.json")
    for case in g["cases"]:
        for dt in ("float16", "bfloat16"):
            x = np.array(case["x"], dtype=np.float32)
            row = x.astype(np.float16) if dt == "float16" else WL.fp32_to_bf16_bits(x)
            q, scale = O.quantize_row(row, dt)
            assert q.tolist() == case["q"], (case["name"], dt, q.tolist())
            assert f32_bits(scale) == int(case["scale_bits"], 16), (case["name"], dt, hex(f32_bits(scale)))


def pin_quant_exact(n_rows: int = 40, h: int = 48, seed: int = 11):
    """Random fp16 / bf16 rows (including exact .5 ties at scale 1) against
    exact rational arithmetic with IEEE rounding."""
    rng = np.random.default_rng(seed)
    for i in range(n_rows):
        dt = "float16" if i % 2 == 0 else "bfloat16"
        kind = i % 4
        if kind < 2:
            x = (rng.standard_normal(h) * (10.0 ** rng.integers(-3, 3))).astype(np.float32)
        else:
            # amax 127 makes the scale exactly 1: half-integers are exact ties
            x = (rng.integers(-254, 255, size=h) / 2.0).astype(np.float32)
            x[0] = 127.0
        row = x.astype(np.float16) if dt == "float16" else WL.fp32_to_bf16_bits(x)
        vals = row.astype(np.float64) if dt == "float16" else WL.bf16_bits_to_fp32(row).astype(np.float64)
        q, scale = O.quantize_row(row, dt)
        want_q, want_scale = quantize_exact(vals)
        assert q.tolist() == want_q, (i, dt)
        assert Fraction(scale) == want_scale, (i, dt)


def pin_quant_dispatch(wl: WL.Workload, inp: dict):
    """quantMode 2 through dispatch: each routed row holds its token's int8 row
    and scale, and |x - q*scale| <= scale/2 (plus the scale's own rounding)."""
    d = O.dispatch(wl, inp)
    ep = d["ep_recv_count"]
    xf = (inp["x"].astype(np.float64) if wl.x_dtype == WL.X_FP16
          else WL.bf16_bits_to_fp32(inp["x"]).astype(np.float64))
    for r in range(wl.ep_world_size):
        for row in range(int(ep[r, -1])):
            s, t, k = d["assist_info"][r, row]
            q = d["expand_x"][r, row].astype(np.int64)
            sc = float(d["dynamic_scales"][r, row])
            assert np.abs(q).max() <= 127
            amax = np.abs(xf[s, t]).max()
            if amax == 0:
                assert sc == 0 and not q.any()
                continue
            assert abs(q[np.argmax(np.abs(xf[s, t]))]) == 127
            assert np.all(np.abs(xf[s, t] - q * sc) <= sc * 0.5 * (1 + 1e-5) + amax * 2e-7)
    return d


def pin_plane_hand():
    g = golden("plane_hand.json")
    for sc in g["scenarios"]:
        wl = WL.Workload("plane", sc["W"], 1, sc["h"], 1, sc["E"], sc["x_dtype"])
        ep = np.array(sc["ep_recv_count"], dtype=np.int32)
        # the fixture's segment sizes and running counts agree
        seg = np.array(sc["segment_rows"], dtype=np.int64).reshape(sc["W"], -1)
        assert np.array_equal(np.cumsum(seg, axis=1), ep), sc["name"]
        got_c = O.combine_plane(wl, ep, sc["bulk_min_bytes"])
        assert got_c.tolist() == sc["combine_plane"], (sc["name"], got_c.tolist())
        got_d = O.dispatch_plane(wl, ep, sc["bulk_min_bytes"])
        assert got_d.tolist() == sc["dispatch_plane"], (sc["name"], got_d.tolist())


def pin_conversions(n: int = 20000, seed: int = 3):
    """fp32 -> fp16 / bf16 round-to-nearest-even against numpy and torch."""
    import torch
    rng = np.random.default_rng(seed)
    vals = np.concatenate([
        rng.standard_normal(n).astype(np.float32) * np.float32(10.0) ** rng.integers(-8, 5, n).astype(np.float32),
        # exact ties between bf16 neighbours and between fp16 neighbours
        (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.float32(1.0) + np.float32(2.0 ** -11) * np.arange(1, 64, 2, dtype=np.float32),
        np.array([0.0, -0.0, 65504.0, 65520.0, 6e-8, 3e-8, 1e-40], dtype=np.float32),
    ]).astype(np.float32)
    L = O.lib()
    want_h = vals.astype(np.float16).view(np.uint16)
    want_b = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got_h = np.array([L.orc_f32_to_fp16(float(v)) for v in vals], dtype=np.uint16)
    got_b = np.array([L.orc_f32_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got_h, want_h), "fp16 rounding"
    assert np.array_equal(got_b, want_b), "bf16 rounding"
    back_h = np.array([L.orc_fp16_to_f32(int(b)) for b in want_h[:2000]], dtype=np.float32)
    assert np.array_equal(back_h, want_h[:2000].view(np.float16).astype(np.float32))
    back_b = np.array([L.orc_bf16_to_f32(int(b)) for b in want_b[:2000]], dtype=np.float32)
    assert np.array_equal(back_b, WL.bf16_bits_to_fp32(want_b[:2000]))


def pin_swiglu_torch(seed: int = 5):
    """SwiGLU expert rows against torch fp64 linear algebra and silu (library
    routines); weights out-major: w_gate, w_up [E, I, h], w_down [E, h, I]."""
    import torch
    rng = np.random.default_rng(seed)
    E, h, I, n = 3, 16, 8, 7
    wg = WL.fp32_to_bf16_bits(rng.standard_normal((E, I, h)).astype(np.float32) * np.float32(0.3))
    wu = WL.fp32_to_bf16_bits(rng.standard_normal((E, I, h)).astype(np.float32) * np.float32(0.3))
    wd = WL.fp32_to_bf16_bits(rng.standard_normal((E, h, I)).astype(np.float32) * np.float32(0.3))
    x = WL.fp32_to_bf16_bits(rng.standard_normal((n, h)).astype(np.float32))
    ex = rng.integers(0, E, size=n).astype(np.int32)
    y = O.swiglu_rows(x, ex, wg, wu, wd)
    t = lambda a: torch.from_numpy(WL.bf16_bits_to_fp32(a).astype(np.float64))
    X, G, U, D = t(x), t(wg), t(wu), t(wd)
    for i in range(n):
        e = int(ex[i])
        a = torch.nn.functional.linear(X[i], G[e])
        b = torch.nn.functional.linear(X[i], U[e])
        want = torch.nn.functional.linear(torch.nn.functional.silu(a) * b, D[e])
        assert np.allclose(y[i], want.numpy(), rtol=1e-12, atol=1e-12), i


def pin_ffn_tokens_compose(seed: int = 9):
    """The FFN variant for a token = sum_k w_k * expert_{e_k}(x) + copy terms:
    checked by composing swiglu_rows over the token's picks by hand."""
    wl = WL.Workload("ffn_tiny", 2, 3, 16, 2, 4, WL.X_BF16, copy_expert_num=1,
                     zero_expert_num=1, special_p=0.3, ffn_intermediate=8, seed=seed)
    inp = WL.make_inputs(wl)
    # plant special picks so that every kind of term appears: a copy expert
    # (id 5) beside a routed one, a zero expert (id 4), a token of two copies
    ids = inp["expert_ids"].copy()
    ids[0, 0, 1] = 5
    ids[0, 1, 0] = 4
    ids[1, 2, :] = 5
    inp = dict(inp, expert_ids=ids)
    toks = np.arange(wl.ep_world_size * wl.bs)
    got = O.moe_ffn_tokens(wl, inp, toks)
    xs = inp["x"].reshape(-1, wl.h)
    ids = inp["expert_ids"].reshape(-1, wl.topk)
    ws = inp["expert_scales"].reshape(-1, wl.topk).astype(np.float64)
    for i in toks:
        want = np.zeros(wl.h)
        for k in range(wl.topk):
            e = int(ids[i, k])
            if e < wl.moe_expert_num:
                want += ws[i, k] * O.swiglu_rows(xs[i:i + 1], np.array([e]), inp["w_gate"], inp["w_up"],
                                                 inp["w_down"])[0]
            elif e >= wl.moe_expert_num + wl.zero_expert_num:
                want += ws[i, k] * WL.bf16_bits_to_fp32(xs[i]).astype(np.float64)
        assert np.allclose(got[i], want, rtol=1e-12, atol=1e-14), i


def pin_errors():
    """Rejections the pages state: id ranges, the 1D mask order, config ranges."""
    base = WL.Workload("err", 2, 4, 16, 2, 4, WL.X_INT32, zero_expert_num=1, copy_expert_num=1)
    inp = WL.make_inputs(base)

    def status(wl, inp):
        return O.dispatch(wl, inp, raise_on_error=False)["status"]

    assert status(base, inp) == 0
    bad = dict(inp, expert_ids=inp["expert_ids"].copy())
    bad["expert_ids"][1, 2, 1] = 6  # E + Z + C = 6 is out of range
    assert status(base, bad) == 4
    bad["expert_ids"][1, 2, 1] = -1
    assert status(base, bad) == 4
    dup = dict(inp, expert_ids=inp["expert_ids"].copy())
    dup["expert_ids"][0, 0, :] = 3  # the same routed expert twice in one token
    assert status(base, dup) == 4
    dup["expert_ids"][0, 0, :] = 5  # the same copy expert twice is allowed
    assert status(base, dup) == 0
    m1 = base.with_(mask_kind=1)
    good = dict(inp, active_mask=np.array([[1, 1, 0, 0], [1, 1, 1, 1]], dtype=np.uint8))
    assert status(m1, good) == 0
    badm = dict(inp, active_mask=np.array([[1, 0, 1, 0], [1, 1, 1, 1]], dtype=np.uint8))
    assert status(m1, badm) == 5
    # a masked pick's id is not looked at
    masked = dict(good, expert_ids=good["expert_ids"].copy())
    masked["expert_ids"][0, 3, 0] = 99
    assert status(m1, masked) == 0
    assert status(base.with_(ep_world_size=1, moe_expert_num=4), inp) == 1
    assert status(base.with_(moe_expert_num=5), inp) == 1
    # topk in [1, 32]
    k32 = base.with_(topk=32, moe_expert_num=64)
    assert status(k32, WL.make_inputs(k32)) == 0
    k33 = base.with_(topk=33, moe_expert_num=66)
    assert status(k33, WL.make_inputs(k33)) == 1
    assert status(base.with_(quant_mode=2), inp) == 2
    # quantisation rules: modes 1..4 take 16-bit float x; output types and the
    # scales input as the quantMode constraints say
    fb = base.with_(x_dtype=WL.X_BF16)
    finp = WL.make_inputs(fb)
    assert status(fb.with_(quant_mode=5), finp) == 2
    assert status(fb.with_(quant_mode=1), finp) == 1                       # static needs a coefficient
    assert status(fb.with_(quant_mode=1, scales_kind=1), dict(finp, quant_scales=np.ones(1, np.float32))) == 0
    assert status(fb.with_(quant_mode=2, scales_kind=1), dict(finp, quant_scales=np.ones(1, np.float32))) == 1
    assert status(fb.with_(quant_mode=3), finp) == 1                       # per-group needs an fp8 type
    assert status(fb.with_(quant_mode=3, y_dtype="fp4_e2m1"), finp) == 1
    assert status(fb.with_(quant_mode=3, y_dtype="fp8_e5m2"), finp) == 0
    assert status(fb.with_(quant_mode=4, y_dtype="fp4_e2m1"), finp) == 0
    assert status(fb.with_(quant_mode=4, y_dtype="fp4_e2m1", h=15), WL.make_inputs(fb.with_(h=15))) == 1
    assert status(fb.with_(quant_mode=4, y_dtype="fp8_e4m3", scales_kind=3),
                  dict(finp, quant_scales=np.ones((4, 16), np.float32))) == 1  # MX takes no scales
    assert status(fb.with_(quant_mode=2, scales_kind=3), finp) == 1          # scales declared, none given


def pin_minifloat_bruteforce(n: int = 1500, seed: int = 13):
    """fp32 -> FP8 E4M3 / E5M2 / FP4 E2M1 against the brute-force nearest value
    of each format's decoded table (exact midpoints, just-off midpoints,
    subnormals, the saturation edge), and FP8 against torch's conversion on
    values inside the finite range."""
    import torch
    rng = np.random.default_rng(seed)
    for fmt in ("fp8_e4m3", "fp8_e5m2", "fp4_e2m1"):
        table = minifloat_table(fmt)
        vals = [float(v) for v, _ in table]
        mids = [float((a + b) / 2) for (a, _), (b, _) in zip(table, table[1:])]
        near = [float(np.nextafter(np.float32(m), np.float32(np.inf))) for m in mids] + \
               [float(np.nextafter(np.float32(m), np.float32(0))) for m in mids if m > 0]
        top = float(table[-1][0])
        rand = (rng.uniform(-1, 1, n) * 2.0 ** rng.integers(-12, 18, n)).astype(np.float32).tolist()
        xs = np.array(vals + mids + near + rand + [0.0, -0.0, top, top * 1.01, top * 4, -top * 3, 1e-30, -1e-30],
                      dtype=np.float32)
        xs = np.concatenate([xs, -xs])
        got = O.f32_to_minifloat(xs, fmt)
        want = [nearest_code(float(v), fmt, is_neg(float(v))) for v in xs]
        assert got.tolist() == want, fmt
        if fmt.startswith("fp8"):
            tdt = torch.float8_e4m3fn if fmt == "fp8_e4m3" else torch.float8_e5m2
            inside = xs[np.abs(xs) <= top]
            lib = torch.from_numpy(inside.copy()).to(tdt).view(torch.uint8).numpy()
            assert np.array_equal(O.f32_to_minifloat(inside, fmt), lib), fmt


def pin_quant_static_hand():
    g = golden("quant_static_hand.json")
    for case in g["cases"]:
        for dt in ("float16", "bfloat16"):
            x = np.array(case["x"], dtype=np.float32)
            row = x.astype(np.float16) if dt == "float16" else WL.fp32_to_bf16_bits(x)
            q, _ = O.quantize_pick(row, 1, dt, expert=case["expert"], scales_kind=case["scales_kind"],
                                   quant_scales=np.array(case["scales"], dtype=np.float32),
                                   moe_expert_num=case["E"])
            assert q.view(np.int8).tolist() == case["q"], (case["name"], dt, q.view(np.int8).tolist())


def pin_quant_mx_group_hand():
    g = golden("quant_mx_group_hand.json")
    for case in g["cases"]:
        for dt in ("float16", "bfloat16"):
            x = np.zeros(case["h"], dtype=np.float32)
            x[:len(case["x"])] = case["x"]
            row = x.astype(np.float16) if dt == "float16" else WL.fp32_to_bf16_bits(x)
            q, dyn = O.quantize_pick(row, case["mode"], dt, case["y"])
            want = [int(b, 16) for b in case["q_hex"].split()]
            assert q[:len(want)].tolist() == want, (case["name"], dt, q[:len(want)].tolist())
            assert not q[len(want):].any(), (case["name"], dt)
            if "dyn" in case:
                assert dyn.tolist() == case["dyn"], (case["name"], dt)
            else:
                assert [f32_bits(float(v)) for v in dyn] == [int(b, 16) for b in case["dyn_bits"]], (case["name"], dt)


def pin_quant_smooth_reduces(seed: int = 17):
    """Per-expert smoothing weights that are powers of two make x * s exact in
    bf16: quantMode 2 / 3 with smoothing for expert e must equal the plain
    mode on the pre-multiplied row (itself pinned by exact arithmetic)."""
    rng = np.random.default_rng(seed)
    h, E = 260, 4
    x = rng.standard_normal(h).astype(np.float32)
    row = WL.fp32_to_bf16_bits(x)
    xf = WL.bf16_bits_to_fp32(row)
    sm = (2.0 ** rng.integers(-2, 3, size=(E, h))).astype(np.float32)
    for e in range(E):
        pre = WL.fp32_to_bf16_bits(xf * sm[e])
        assert np.array_equal(WL.bf16_bits_to_fp32(pre), xf * sm[e])
        for mode, y in ((2, ""), (3, "fp8_e4m3"), (3, "fp8_e5m2")):
            q1, d1 = O.quantize_pick(row, mode, "bfloat16", y, expert=e, quant_scales=sm, scales_kind=3,
                                     moe_expert_num=E)
            q0, d0 = O.quantize_pick(pre, mode, "bfloat16", y)
            assert np.array_equal(q1, q0) and np.array_equal(d1, d0), (e, mode, y)
    # the smoothing row is the pick's expert's: distinct experts, distinct rows
    qa, _ = O.quantize_pick(row, 2, "bfloat16", expert=0, quant_scales=sm, scales_kind=3, moe_expert_num=E)
    qb, _ = O.quantize_pick(row, 2, "bfloat16", expert=1, quant_scales=sm, scales_kind=3, moe_expert_num=E)
    assert not np.array_equal(qa, qb)


def pin_quant_group_exact(seed: int = 19):
    """quantMode 3 by exact arithmetic: groups of 128 (the last one ragged),
    fp32 scales amax / FMAX, fp8 codes of the IEEE quotient; zero groups and
    signed zeros included."""
    rng = np.random.default_rng(seed)
    for i, (fmt, dt, h) in enumerate([("fp8_e4m3", "bfloat16", 300), ("fp8_e5m2", "float16", 300),
                                      ("fp8_e4m3", "float16", 128), ("fp8_e5m2", "bfloat16", 70)]):
        x = (rng.standard_normal(h) * 10.0 ** rng.integers(-2, 3)).astype(np.float32)
        if h > 256:
            x[128:256] = 0.0
            x[130] = -0.0
        x[3] = -0.0
        row = x.astype(np.float16) if dt == "float16" else WL.fp32_to_bf16_bits(x)
        xs = row_values(row, dt)
        q, dyn = O.quantize_pick(row, 3, dt, fmt)
        codes, scales = group_quant_exact(xs, fmt)
        assert q.tolist() == codes, (i, fmt)
        assert [Fraction(float(v)) for v in dyn] == scales, (i, fmt)


def pin_quant_mx_exact(seed: int = 23):
    """quantMode 4 against the OCP MX conversion worked exactly: E8M0 bytes
    from frexp, element codes by brute force (fp4 unpacked low nibble first);
    zero, power-of-two and ragged blocks included."""
    rng = np.random.default_rng(seed)
    for i, (fmt, dt, h) in enumerate([("fp8_e4m3", "bfloat16", 200), ("fp8_e5m2", "float16", 96),
                                      ("fp4_e2m1", "bfloat16", 200), ("fp4_e2m1", "float16", 64)]):
        x = (rng.standard_normal(h) * 10.0 ** rng.integers(-3, 3)).astype(np.float32)
        x[32:64] = 0.0
        x[40] = -0.0
        if h > 96:
            x[64:96] = rng.integers(-8, 9, 32).astype(np.float32) / 4.0
            x[70] = 2.0      # block amax an exact power of two
        row = x.astype(np.float16) if dt == "float16" else WL.fp32_to_bf16_bits(x)
        xs = row_values(row, dt)
        q, dyn = O.quantize_pick(row, 4, dt, fmt)
        codes, sbytes = mx_quant_exact(xs, fmt)
        got = unpack_fp4(q) if fmt == "fp4_e2m1" else q.tolist()
        assert got == codes, (i, fmt)
        assert dyn.tolist() == sbytes, (i, fmt)


def pin_quant_modes_dispatch(seed: int = 29):
    """Every quantised mode through dispatch: each routed row (found through
    assist_info) holds its token's row quantised for the pick's expert, worked
    out here exactly; the layout equals the unquantised one."""
    cases = [(1, "", 1), (1, "", 2), (1, "", 3), (2, "", 3), (3, "fp8_e4m3", 0), (3, "fp8_e5m2", 3),
             (4, "fp8_e4m3", 0), (4, "fp4_e2m1", 0)]
    for i, (mode, y, sk) in enumerate(cases):
        wl = WL.Workload(f"qd{i}", 2, 3, 160, 2, 4, WL.X_BF16, quant_mode=mode, y_dtype=y, scales_kind=sk,
                         mask_kind=2, mask_false_p=0.2, seed=seed + i)
        inp = WL.make_inputs(wl)
        d = O.dispatch(wl, inp)
        base = O.dispatch(wl.with_(quant_mode=0, y_dtype="", scales_kind=0), inp)
        assert np.array_equal(d["ep_recv_count"], base["ep_recv_count"])
        assert np.array_equal(d["assist_info"], base["assist_info"])
        qs = inp.get("quant_scales")
        for r in range(wl.ep_world_size):
            for row in range(int(d["ep_recv_count"][r, -1])):
                s, t, k = d["assist_info"][r, row]
                e = int(inp["expert_ids"][s, t, k])
                xs = row_values(inp["x"][s, t], WL.X_BF16)
                if sk:
                    sv = {1: lambda j: qs[0], 2: lambda j: qs[j], 3: lambda j: qs[e, j]}[sk]
                    xs = [float(np.float32(v) * np.float32(sv(j))) for j, v in enumerate(xs)]
                got = d["expand_x"][r, row]
                if mode == 1:
                    want = [max(-128, min(127, round_half_even(Fraction(v)))) for v in xs]
                    assert got.tolist() == want, (i, r, row)
                elif mode == 2:
                    want, scale = quantize_exact(xs)
                    assert got.tolist() == want and Fraction(float(d["dynamic_scales"][r, row])) == scale
                elif mode == 3:
                    codes, scales = group_quant_exact(xs, y)
                    assert got.tolist() == codes and [Fraction(float(v)) for v in d["dynamic_scales"][r, row]] == scales
                else:
                    codes, sbytes = mx_quant_exact(xs, y)
                    g = unpack_fp4(got) if y == "fp4_e2m1" else got.tolist()
                    assert g == codes and d["dynamic_scales"][r, row].tolist() == sbytes, (i, r, row)


def pin_combine_rejects_inconsistent_assist(seed: int = 31):
    """Combine takes dispatch's assist_info / ep_recv_count unchanged ([DISP]
    约束说明: dispatch outputs go into combine as they are). Layouts that cannot
    have come from the routing are rejected with BAD_ASSIST (9): a routed pick
    that no row names (the last row cut off by its count), a pick named by two
    rows, a row naming a pick that is not routed (masked, zero or copy), a row
    naming a pick outside the batch, and a count above the capacity A."""
    wl = WL.Workload("assist", 2, 6, 8, 2, 4, WL.X_INT32, zero_expert_num=1, copy_expert_num=1,
                     mask_kind=2, special_p=0.25, mask_false_p=0.2, seed=seed)
    inp = WL.make_inputs(wl)
    d = O.dispatch(wl, inp)
    ex, ai, erc = d["expand_x"], d["assist_info"], d["ep_recv_count"]
    A = ai.shape[1]
    assert O.combine(wl, ex, ai, erc, inp, raise_on_error=False)[1] == 0
    routed = {tuple(ai[r, i].tolist()) for r in range(2) for i in range(erc[r, -1])}
    others = [(s, t, k) for s in range(2) for t in range(wl.bs) for k in range(wl.topk)
              if (s, t, k) not in routed]
    assert others, "the fixture needs a pick that is not routed"
    r = int(np.argmax(erc[:, -1]))          # a rank that holds rows
    n = int(erc[r, -1])
    assert 0 < n < A

    def status(ai2, erc2):
        return O.combine(wl, ex, ai2, erc2, inp, raise_on_error=False)[1]

    cut = erc.copy()
    cut[r, -1] -= 1
    assert status(ai, cut) == 9                      # a routed pick with no row
    grow = erc.copy()
    grow[r, -1] += 1
    dup = ai.copy()
    dup[r, n] = ai[r, 0]
    assert status(dup, grow) == 9                    # one pick, two rows
    extra = ai.copy()
    extra[r, n] = others[0]
    assert status(extra, grow) == 9                  # a row for a pick that is not routed
    outside = ai.copy()
    outside[r, n] = (0, wl.bs, 0)
    assert status(outside, grow) == 9                # a token outside the batch
    over = erc.copy()
    over[0, -1] = A + 1
    assert status(ai, over) == 9                     # more rows than the capacity


def pin_combine_int32_wraps():
    """int32 data: the weighted sum is exact integer arithmetic taken modulo
    2^32 (two's complement), like int32 arithmetic on any machine; nothing
    saturates. Token (0, 0) has weights 1 and 3 on one row each (identity
    expert), so its output is 4 x: 2^30 * 4 = 2^32 -> 0, (2^31 - 1) * 4 =
    2^33 - 4 -> -4, -2^31 * 4 = -2^33 -> 0, 5 * 4 = 20. Token (1, 1) has
    weights 1 and 1: -2^31 * 2 = -2^32 -> 0."""
    wl = WL.Workload("wrap", 2, 2, 4, 2, 4, WL.X_INT32, seed=0)
    ids = np.array([[[0, 2], [1, 3]], [[2, 0], [3, 1]]], dtype=np.int32)
    x = np.zeros((2, 2, 4), dtype=np.int32)
    x[0, 0] = [2 ** 30, 2 ** 31 - 1, -2 ** 31, 5]
    x[0, 1] = [7, -7, 1, 0]
    x[1, 0] = [2 ** 30, 1, -1, 2 ** 31 - 1]
    x[1, 1] = [-2 ** 31, 3, 0, 1]
    w = np.array([[[1, 3], [2, 2]], [[4, 0], [1, 1]]], dtype=np.int32)
    inp = {"x": x, "expert_ids": ids, "expert_scales": w, "active_mask": None}
    d = O.dispatch(wl, inp)
    got = O.combine(wl, O.identity_expert(d), d["assist_info"], d["ep_recv_count"], inp)
    tot = w.astype(object).sum(-1)
    for s in range(2):
        for t in range(2):
            for j in range(4):
                v = int(x[s, t, j]) * int(tot[s, t])
                want = (v + 2 ** 31) % 2 ** 32 - 2 ** 31
                assert int(got[s, t, j]) == want, (s, t, j, int(got[s, t, j]), want)
    assert got[0, 0].tolist() == [0, -4, 0, 20] and int(got[1, 1, 0]) == 0


def pin_mx_scale_floor():
    """OCP MX: the shared scale X = 2^(floor(log2 amax) - emax) is stored as an
    E8M0 byte, whose smallest value is 2^-127 (byte 0). Blocks of tiny bf16
    values whose exponent would fall below that are clamped to 2^-127:
      E4M3 (emax 8):  amax = 2^-120 -> 2^-128 -> clamped 2^-127, byte 0;
                      2^-120 / 2^-127 = 128 = 1.0 * 2^7 -> code (7+7) << 3 = 0x70;
                      1.5 * 2^-121 / 2^-127 = 96 = 1.5 * 2^6 -> (13 << 3) | 4 = 0x6C.
      E5M2 (emax 15): amax = 2^-115 -> 2^-130 -> 2^-127, byte 0;
                      2^-115 / 2^-127 = 4096 = 2^12 -> (12+15) << 2 = 0x6C.
      E2M1 (emax 2):  amax = 2^-120 -> 2^-122, byte 5 (no clamp);
                      2^-120 / 2^-122 = 4 -> code 0b110 = 6."""
    def row(vals):
        x = np.zeros(32, dtype=np.float32)
        x[:len(vals)] = vals
        return WL.fp32_to_bf16_bits(x)

    q, dyn = O.quantize_pick(row([2.0 ** -120, -1.5 * 2.0 ** -121]), 4, "bfloat16", "fp8_e4m3")
    assert dyn.tolist() == [0] and q[:2].tolist() == [0x70, 0x80 | 0x6C] and not q[2:].any()
    q, dyn = O.quantize_pick(row([2.0 ** -115]), 4, "bfloat16", "fp8_e5m2")
    assert dyn.tolist() == [0] and q[0] == 0x6C and not q[1:].any()
    q, dyn = O.quantize_pick(row([2.0 ** -120]), 4, "bfloat16", "fp4_e2m1")
    assert dyn.tolist() == [5] and q[0] == 0x06 and not q[1:].any()
    # the exact rational model agrees on the clamped blocks
    for fmt, v in (("fp8_e4m3", [2.0 ** -120, -1.5 * 2.0 ** -121]), ("fp8_e5m2", [2.0 ** -115])):
        xs = WL.bf16_bits_to_fp32(row(v)).tolist()
        codes, sb = mx_quant_exact(xs, fmt)
        q, dyn = O.quantize_pick(row(v), 4, "bfloat16", fmt)
        assert q.tolist() == codes and dyn.tolist() == sb


def run_all():
    """Every pin, on the fixtures plus small and random workloads."""
    pin_dispatch_combine_hand()
    pin_combine_order_hand()
    pin_quant_hand()
    pin_plane_hand()
    pin_errors()
    for name in ("w2_bs8_h16_k2_e4_i32", "w8_bs8_h16_k2_e64_i32", "w2_bs8_h256_k2_e4_i32"):
        wl = WL.WORKLOADS[name]
        inp = WL.make_inputs(wl)
        d = pin_layout_bruteforce(wl, inp)
        pin_invariants(wl, inp, d)
        pin_combine_closed_form_int(wl, inp, d)
        pin_combine_gather(wl, inp, d)
    rng = np.random.default_rng(2024)
    for _ in range(25):
        wl = WL.small_random_workload(rng)
        inp = WL.make_inputs(wl)
        d = pin_layout_bruteforce(wl, inp)
        pin_invariants(wl, inp, d)
        pin_combine_closed_form_int(wl, inp, d)
        pin_combine_gather(wl, inp, d)
    wl = WL.WORKLOADS["w8_bs8_h16_k2_e64_f16"]
    inp = WL.make_inputs(wl)
    d = pin_layout_bruteforce(wl, inp)
    pin_invariants(wl, inp, d)
    pin_combine_closed_form_float(wl, inp, d)
    wlb = WL.Workload("bf16_small", 4, 6, 32, 3, 8, WL.X_BF16, zero_expert_num=2, copy_expert_num=2,
                      mask_kind=2, special_p=0.2, mask_false_p=0.2, seed=17)
    inp = WL.make_inputs(wlb)
    d = pin_layout_bruteforce(wlb, inp)
    pin_invariants(wlb, inp, d)
    pin_combine_closed_form_float(wlb, inp, d)
    wq = WL.Workload("q2_small", 4, 5, 64, 3, 8, WL.X_FP16, quant_mode=2, mask_kind=1, seed=19)
    inp = WL.make_inputs(wq)
    d = pin_quant_dispatch(wq, inp)
    pin_invariants(wq, inp, d)
    pin_quant_exact()
    pin_minifloat_bruteforce(n=300)
    pin_quant_static_hand()
    pin_quant_mx_group_hand()
    pin_quant_smooth_reduces()
    pin_quant_group_exact()
    pin_quant_mx_exact()
    pin_quant_modes_dispatch()
    pin_conversions(n=4000)
    pin_swiglu_torch()
    pin_ffn_tokens_compose()
    pin_combine_rejects_inconsistent_assist()
    pin_combine_int32_wraps()
    pin_mx_scale_floor()
