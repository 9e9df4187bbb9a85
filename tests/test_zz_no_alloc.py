"""moe_combine_noalloc: the gather combine for callers that cannot allocate
device memory (a plugin or custom-op host that hands the library only its
input and output buffers, or a serving loop that must not allocate once it
runs). Its pick -> row scratch is one fixed device array inside the library,
shared by every call on a device and left holding the last call's map.

Checked through the C ABI against the CPU oracle's combine (int32 bit-exact;
floats within 1e-3 * max |x_out|, and in fact the same bytes, since both fix
the fp32 multiply-add order). Two different routings alternate call by call,
so each call starts with the other routing's map in the shared scratch: a
map entry the call failed to rewrite would send a pick to the wrong row.

Kept in a file of its own that pytest collects last."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from combine_route_scan_gb300 import build
    build.build()
    from combine_route_scan_gb300 import moe as M
    return M


def _prepared(wl):
    """Inputs on the device, a GPU dispatch of them (its assist_info and
    counts checked against the oracle's), and the oracle's combine of the
    identity expert."""
    import gpu_harness as H
    from oracle import oracle as O
    inp = WL.make_inputs(wl)
    ref = O.dispatch(wl, inp)
    dev = H.device_inputs(wl, inp)
    got, _, _ = H.gpu_dispatch(wl, dev)
    H.compare_dispatch(wl, got, ref)
    x_ref = O.combine(wl, ref["expand_x"], ref["assist_info"], ref["ep_recv_count"], inp)
    return dev, got, x_ref


def _call(moe, wl, dev, got, status):
    import gpu_harness as H
    cfg = H.make_cfg(wl, quant_mode=0)
    x_out = torch.empty_like(dev["x"])
    x_out.view(torch.uint8).fill_(0x33)
    rc = moe.lib().moe_combine_noalloc(
        ctypes.byref(cfg), ctypes.c_void_p(got["expand_x"].data_ptr()),
        ctypes.c_void_p(got["assist_info"].data_ptr()), ctypes.c_void_p(got["ep_recv_count"].data_ptr()),
        ctypes.c_void_p(dev["expert_ids"].data_ptr()), ctypes.c_void_p(dev["expert_scales"].data_ptr()),
        None if dev["active_mask"] is None else ctypes.c_void_p(dev["active_mask"].data_ptr()),
        ctypes.c_void_p(dev["x"].data_ptr()), ctypes.c_void_p(x_out.data_ptr()),
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, moe.status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, moe.status_string(int(status.item()))
    return x_out


# pairs of routings of the same shape (the scratch then holds entries for the
# same picks, pointing to other rows) and of different shapes
PAIRS = [
    ("w16_bs256_h7168_k8_e256_bf16_zipf", "w16_bs256_h7168_k8_e256_bf16_zipf@seed=91"),
    ("w8_bs8_h16_k2_e64_i32", "w8_bs8_h16_k2_e64_i32@seed=92"),
    ("w8_bs8_h16_k2_e64_f16", "w8_bs32_h7168_k8_e64_f16"),
]


def _workload(tag):
    name, _, seed = tag.partition("@seed=")
    wl = WL.WORKLOADS[name]
    return wl.with_(seed=int(seed)) if seed else wl


@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: "+".join(p))
def test_noalloc_combine_matches_the_oracle_across_alternating_routings(moe, pair):
    import gpu_harness as H
    wls = [_workload(t) for t in pair]
    prepared = [_prepared(wl) for wl in wls]
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    # A, B, A, B: every call after the first finds the other routing's map
    for call in range(4):
        i = call % 2
        wl, (dev, got, x_ref) = wls[i], prepared[i]
        x_out = H.to_host(_call(moe, wl, dev, got, status))
        H.compare_combine(wl, x_out, x_ref)
        assert np.array_equal(x_out.view(np.uint8), x_ref.view(np.uint8)), f"call {call} ({wl.name})"


def test_noalloc_rejects_calls_beyond_its_scratch(moe):
    cfg = moe.config(16, 4096, 64, 8, 256, torch.bfloat16)  # 524288 picks > 262144
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.combine_noalloc(cfg, t, t, t, t, t, None, t, t, status)
    assert ei.value.name == "INVALID_ARG"
