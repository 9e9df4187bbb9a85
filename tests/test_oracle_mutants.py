"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
the pins catch every one: a dropped term, a wrong index, a swapped loop, the
wrong rounding, an off-by-one comparison, a missing consistency check.

Two guards have no mutant here because no input can tell them apart: the
dispatch capacity check (with a token's routed ids distinct, a rank receives at
most bs * W * min(L, K) = A rows, so the check never fires) and combine's bound
of a rank's row count by A (without it, a count above A on a rank reads the
next rank's first rows, whose picks the duplicate check then reports with the
same status; on the last rank it would read past the array, which no test
may make it do)."""
import os
import subprocess
import tempfile

import pytest

import oracle_pins as P
from oracle import oracle as O

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "moe_oracle.c")

MUTANTS = {
    "rank_from_modulo": [("int d = e / L;", "int d = e % W;")],
    "exclusive_counts": [("run += cnt[g];\n        ep_recv_count[g] = (int32_t)run;",
                          "ep_recv_count[g] = (int32_t)run;\n        run += cnt[g];")],
    "source_major_segments": [(
        "for (int le = 0; le < L; ++le)\n      for (int s = 0; s < W; ++s) {\n        size_t g = ((size_t)d * L + le) * W + s;\n        next[g] = run;",
        "for (int s = 0; s < W; ++s)\n      for (int le = 0; le < L; ++le) {\n        size_t g = ((size_t)d * L + le) * W + s;\n        next[g] = run;")],
    "tokens_reversed_in_segment": [("for (int t = 0; t < bs; ++t) {\n      size_t src",
                                    "for (int t = bs - 1; t >= 0; --t) {\n      size_t src")],
    "assist_fields_swapped": [("assist[row * 3 + 0] = s;\n        assist[row * 3 + 1] = t;",
                               "assist[row * 3 + 0] = t;\n        assist[row * 3 + 1] = s;")],
    "capacity_uses_k": [("return (int64_t)c->bs * c->W * (L < c->K ? L : c->K);",
                         "return (int64_t)c->bs * c->W * c->K;")],
    "mask_ignored": [("if (c->mask_kind == 0 || mask == NULL) return 1;", "return 1;")],
    "mask_order_unchecked": [("else if (seen_false) return ORC_ERR_MASK_ORDER;", "else if (seen_false) {}")],
    "duplicates_allowed": [("if (classify(c, ids, mask, s, t, k2, &e2) == PICK_ROUTED && e2 == e) {",
                            "if (0) {")],
    "zero_as_copy": [("if ((int64_t)e < (int64_t)c->E + c->Z) return PICK_ZERO;",
                      "if ((int64_t)e < (int64_t)c->E + c->Z) return PICK_COPY;")],
    "copy_weight_dropped_int": [("acc += w * ((const int32_t*)x)[tok * h + j];",
                                 "acc += ((const int32_t*)x)[tok * h + j];")],
    "copy_weight_dropped_float": [("acc = fmaf(w, load_f(c, x, tok * h + j), acc);",
                                   "acc += load_f(c, x, tok * h + j);")],
    "combine_unfused": [("acc = fmaf(w, load_f(c, x, tok * h + j), acc);",
                         "acc = acc + w * load_f(c, x, tok * h + j);")],
    "combine_k_descending": [("for (int k = 0; k < K; ++k) {\n            float w",
                              "for (int k = K - 1; k >= 0; --k) {\n            float w")],
    "combine_routed_weight_dropped": [(
        "acc += w * ((const int32_t*)expert_out)[(size_t)where[tok * K + k] * h + j];",
        "acc += ((const int32_t*)expert_out)[(size_t)where[tok * K + k] * h + j];")],
    "quant_reciprocal": [("float r = amax == 0.0f ? 0.0f : nearbyintf(xs[j] / scale);",
                          "float r = amax == 0.0f ? 0.0f : nearbyintf(xs[j] * (127.0f / amax));")],
    "quant_round_away": [("float r = amax == 0.0f ? 0.0f : nearbyintf(", "float r = amax == 0.0f ? 0.0f : roundf(")],
    "quant_scale_255": [("float scale = amax / 127.0f;", "float scale = amax / 255.0f;")],
    "bf16_truncates": [("u += 0x7FFFu + lsb;", "u += 0u * lsb;")],
    "plane_size_strict": [("bytes >= c->bulk_min_bytes && bytes * den > num);\n      }\n  }\n  return ORC_OK;\n}\n\n/* Dispatch",
                           "bytes > c->bulk_min_bytes && bytes * den > num);\n      }\n  }\n  return ORC_OK;\n}\n\n/* Dispatch")],
    "plane_mean_non_strict": [("bytes >= c->bulk_min_bytes && bytes * den > num);\n      }\n  }\n  return ORC_OK;\n}\n\n/* Dispatch",
                               "bytes >= c->bulk_min_bytes && bytes * den >= num);\n      }\n  }\n  return ORC_OK;\n}\n\n/* Dispatch")],
    "plane_remote_counts_local": [("if (s != d) remote += seg_rows", "remote += seg_rows")],
    "dispatch_plane_wrong_den": [("const int64_t row_bytes = row_out_bytes(c);\n  const int64_t den = (int64_t)(W - 1 > 1 ? W - 1 : 1) * L;",
                                  "const int64_t row_bytes = row_out_bytes(c);\n  const int64_t den = (int64_t)W * L;")],
    "static_clamp_symmetric": [("if (r < -128.0f) r = -128.0f;", "if (r < -127.0f) r = -127.0f;")],
    "smooth_ignored": [("case ORC_SC_EXPERT: return v * quant_scales[(size_t)e * c->h + j];",
                        "case ORC_SC_EXPERT: return v;")],
    "smooth_first_expert_row": [("case ORC_SC_EXPERT: return v * quant_scales[(size_t)e * c->h + j];",
                                 "case ORC_SC_EXPERT: return v * quant_scales[j];")],
    "group_of_64": [("for (int g0 = 0; g0 < h; g0 += 128) {\n      int g1 = g0 + 128 < h ? g0 + 128 : h;",
                     "for (int g0 = 0; g0 < h; g0 += 64) {\n      int g1 = g0 + 64 < h ? g0 + 64 : h;")],
    "e4m3_fmax_240": [("const float fmax = c->y_kind == ORC_Y_FP8_E4M3 ? 448.0f : 57344.0f;",
                       "const float fmax = c->y_kind == ORC_Y_FP8_E4M3 ? 240.0f : 57344.0f;")],
    "mx_emax_off_by_one": [("const int emax = c->y_kind == ORC_Y_FP8_E4M3 ? 8 :",
                            "const int emax = c->y_kind == ORC_Y_FP8_E4M3 ? 7 :")],
    "mx_scale_ceil": [("se = (ex - 1) - emax;", "se = ex - emax;")],
    "minifloat_ties_away": [("double n = nearbyint(a / quantum);", "double n = round(a / quantum);")],
    "minifloat_no_subnormals": [("if (a < ldexp(1.0, emin)) e = emin;", "if (0) e = emin;")],
    "fp4_nibbles_swapped": [("q[j / 2] |= (uint8_t)(code << (4 * (j % 2)));",
                             "q[j / 2] |= (uint8_t)(code << (4 * (1 - j % 2)));")],
    "mask_2d_transposed": [("return mask[((size_t)s * c->bs + t) * c->K + k] != 0;",
                            "return mask[((size_t)s * c->K + k) * c->bs + t] != 0;")],
    "mask_order_across_ranks": [("for (int s = 0; s < c->W; ++s) {\n    int seen_false = 0;",
                                 "int seen_false = 0;\n  for (int s = 0; s < c->W; ++s) {")],
    "copy_range_inclusive": [("if ((int64_t)e < (int64_t)c->E + c->Z + c->C) return PICK_COPY;",
                              "if ((int64_t)e <= (int64_t)c->E + c->Z + c->C) return PICK_COPY;")],
    "topk_33_accepted": [("c->K <= 0 || c->K > 32)", "c->K <= 0 || c->K > 33)")],
    "expand_scales_first_pick": [("(const char*)scales + (src * K + k) * 4, 4);",
                                  "(const char*)scales + (src * K) * 4, 4);")],
    "segment_rows_first_rank_only": [("return (g % LW == 0) ? ep_recv_count[g]", "return (g == 0) ? ep_recv_count[g]")],
    "dispatch_plane_counts_local": [("if (d != s)\n        for (int le = 0; le < L; ++le) remote +=",
                                     "for (int le = 0; le < L; ++le) remote +=")],
    "combine_duplicate_row_accepted": [("if (where[p] >= 0) { st = ORC_ERR_BAD_ASSIST; break; }",
                                        "if (0) { st = ORC_ERR_BAD_ASSIST; break; }")],
    "combine_missing_row_accepted": [(
        "if (cls[k] == PICK_ROUTED && where[tok * K + k] < 0) { st = ORC_ERR_BAD_ASSIST; break; }", "")],
    "combine_unrouted_row_accepted": [(
        "if (cls[k] != PICK_ROUTED && where[tok * K + k] >= 0) { st = ORC_ERR_BAD_ASSIST; break; }", "")],
    "int32_combine_saturates": [(
        "((int32_t*)x_out)[tok * h + j] = (int32_t)(uint32_t)(uint64_t)acc;",
        "((int32_t*)x_out)[tok * h + j] = acc > 2147483647 ? 2147483647 : "
        "(acc < -2147483647 ? -2147483647 : (int32_t)acc);")],
    "group_amax_signed": [("for (int j = g0; j < g1; ++j) if (fabsf(xs[j]) > amax) amax = fabsf(xs[j]);",
                           "for (int j = g0; j < g1; ++j) if (xs[j] > amax) amax = xs[j];")],
    "e4m3_saturates_to_nan": [("f.maxv = 448.0; f.max_code = 0x7E;", "f.maxv = 448.0; f.max_code = 0x7F;")],
    "mx_scale_bias_128": [("((uint8_t*)dyn)[b0 / 32] = (uint8_t)(se + 127);",
                           "((uint8_t*)dyn)[b0 / 32] = (uint8_t)(se + 128);")],
    "mx_scale_floor_126": [("if (se < -127) se = -127;", "if (se < -126) se = -126;")],
    "ffn_copy_weight_dropped": [("for (int j = 0; j < h; ++j) o[j] += w * bf16_to_f32(x[(size_t)tok * h + j]);",
                                 "for (int j = 0; j < h; ++j) o[j] += bf16_to_f32(x[(size_t)tok * h + j]);")],
    "silu_sign": [("a[i] = g / (1.0 + exp(-g)) * u;", "a[i] = g / (1.0 + exp(g)) * u;")],
    "gate_up_swapped": [("g += xv[j] * bf16_to_f32(wg[", "g += xv[j] * bf16_to_f32(wu[")],
    "down_transposed": [("acc += a[i] * bf16_to_f32(wd[(size_t)j * I + i]);",
                         "acc += a[i] * bf16_to_f32(wd[(size_t)i * h + j]);")],
}


def _build_mutant(text: str, workdir: str, name: str) -> str:
    src = os.path.join(workdir, f"{name}.c")
    lib = os.path.join(workdir, f"lib_{name}.so")
    with open(src, "w") as f:
        f.write(text)
    subprocess.run(["gcc", "-O1", "-std=gnu11", "-ffp-contract=off", "-fPIC", "-shared", "-w",
                    "-o", lib, src, "-lm"], check=True)
    return lib


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory(prefix="oracle_mutants_") as d:
        yield d


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, workdir):
    with open(SRC) as f:
        text = f.read()
    for old, new in MUTANTS[name]:
        assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
        text = text.replace(old, new)
    lib = _build_mutant(text, workdir, name)
    O.use_library(lib)
    try:
        with pytest.raises((AssertionError, O.OracleError, KeyError)):
            P.run_all()
    finally:
        O.use_library(None)


def test_unmutated_copy_passes(workdir):
    with open(SRC) as f:
        lib = _build_mutant(f.read(), workdir, "clean")
    O.use_library(lib)
    try:
        P.run_all()
    finally:
        O.use_library(None)
