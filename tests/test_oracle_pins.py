"""The CPU oracle against hand-worked fixtures, brute force, closed forms,
exact arithmetic and library routines (no GPU)."""
import numpy as np
import pytest

import oracle_pins as P
import workloads as WL


def test_dispatch_combine_hand_fixtures():
    P.pin_dispatch_combine_hand()


def test_combine_fma_order_hand_fixture():
    P.pin_combine_order_hand()


def test_quantiser_hand_fixtures():
    P.pin_quant_hand()


def test_quantiser_exact_rational():
    P.pin_quant_exact()


def test_plane_rule_hand_fixture():
    P.pin_plane_hand()


def test_error_rules():
    P.pin_errors()


def test_scalar_conversions_vs_numpy_torch():
    P.pin_conversions()


def test_swiglu_vs_torch_fp64():
    P.pin_swiglu_torch()


def test_ffn_variant_composition():
    P.pin_ffn_tokens_compose()


@pytest.mark.parametrize("name", ["w2_bs8_h16_k2_e4_i32", "w8_bs8_h16_k2_e64_i32", "w2_bs8_h256_k2_e4_i32"])
def test_int32_workloads_layout_and_closed_form(name):
    wl = WL.WORKLOADS[name]
    inp = WL.make_inputs(wl)
    d = P.pin_layout_bruteforce(wl, inp)
    P.pin_invariants(wl, inp, d)
    P.pin_combine_closed_form_int(wl, inp, d)
    P.pin_combine_gather(wl, inp, d)


@pytest.mark.parametrize("seed", range(40))
def test_random_small_layout_and_combine(seed):
    rng = np.random.default_rng(1000 + seed)
    wl = WL.small_random_workload(rng)
    inp = WL.make_inputs(wl)
    d = P.pin_layout_bruteforce(wl, inp)
    P.pin_invariants(wl, inp, d)
    P.pin_combine_closed_form_int(wl, inp, d)
    P.pin_combine_gather(wl, inp, d)


def test_float_closed_forms():
    for wl in (WL.WORKLOADS["w8_bs8_h16_k2_e64_f16"],
               WL.Workload("bf16_small", 4, 6, 32, 3, 8, WL.X_BF16, zero_expert_num=2, copy_expert_num=2,
                           mask_kind=2, special_p=0.2, mask_false_p=0.2, seed=17)):
        inp = WL.make_inputs(wl)
        d = P.pin_layout_bruteforce(wl, inp)
        P.pin_invariants(wl, inp, d)
        P.pin_combine_closed_form_float(wl, inp, d)


def test_quant_dispatch_properties():
    wq = WL.Workload("q2_small", 4, 5, 64, 3, 8, WL.X_FP16, quant_mode=2, mask_kind=1, seed=19)
    inp = WL.make_inputs(wq)
    d = P.pin_quant_dispatch(wq, inp)
    P.pin_invariants(wq, inp, d)


def test_skewed_workload_invariants_and_closed_form():
    """The full-size skewed workload: invariants and the identity-expert closed
    form, checked on the oracle's own output."""
    wl = WL.WORKLOADS["w16_bs256_h7168_k8_e256_bf16_zipf"]
    inp = WL.make_inputs(wl)
    from oracle import oracle as O
    d = O.dispatch(wl, inp)
    ep = d["ep_recv_count"].astype(np.int64)
    routed = inp["active_mask"].astype(bool) & (inp["expert_ids"] < wl.moe_expert_num)
    assert ep[:, -1].sum() == routed.sum()
    # some (expert, source) segments exceed 2 MiB, so the bulk plane is used
    seg = np.diff(np.concatenate([np.zeros((wl.ep_world_size, 1), np.int64), ep], axis=1), axis=1)
    assert (seg * wl.h * wl.es >= 2 * 1024 * 1024).sum() > 0
    assert O.dispatch_plane(wl, d["ep_recv_count"]).sum() > 0
    x_out = O.combine(wl, d["expand_x"], d["assist_info"], d["ep_recv_count"], inp)
    xf = WL.bf16_bits_to_fp32(inp["x"]).astype(np.float64)
    want = xf * P.contributing_weight_sum(wl, inp)[..., None]
    got = WL.bf16_bits_to_fp32(x_out).astype(np.float64)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -7 + 1e-5)


def test_small_float_conversions_bruteforce_and_torch():
    P.pin_minifloat_bruteforce()


def test_static_quant_hand_fixture():
    P.pin_quant_static_hand()


def test_smoothing_reduces_to_plain_modes():
    P.pin_quant_smooth_reduces()


def test_per_group_quant_exact():
    P.pin_quant_group_exact()


def test_mx_quant_exact():
    P.pin_quant_mx_exact()


def test_quant_modes_through_dispatch():
    P.pin_quant_modes_dispatch()


def test_mx_and_group_hand_fixture():
    P.pin_quant_mx_group_hand()


def test_combine_rejects_layouts_dispatch_cannot_make():
    P.pin_combine_rejects_inconsistent_assist()


def test_int32_combine_wraps_modulo_2_32():
    P.pin_combine_int32_wraps()


def test_mx_scale_clamped_at_e8m0_floor():
    P.pin_mx_scale_floor()
