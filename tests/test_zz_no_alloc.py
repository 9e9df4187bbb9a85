"""moe_combine_noalloc: the gather combine for callers that cannot allocate
device memory (a host that passes only input and output buffers, or a serving
loop that must not allocate after start-up). Its scratch is a fixed device
array inside the library. Checked through the C ABI against moe_combine on the
same inputs, twice in a row (the shared scratch keeps the previous call's
contents, which must not leak into the next result).

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


@pytest.mark.parametrize("name", ["w16_bs256_h7168_k8_e256_bf16_zipf", "w8_bs8_h16_k2_e64_i32",
                                  "w8_bs8_h16_k2_e64_f16"])
def test_noalloc_combine_matches_moe_combine(moe, name):
    import gpu_harness as H
    wl = WL.WORKLOADS[name]
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    got, _, _ = H.gpu_dispatch(wl, dev)
    ref, st, _ = H.gpu_combine(wl, dev, got["expand_x"], got["assist_info"], got["ep_recv_count"])
    assert st == 0
    cfg = H.make_cfg(wl, quant_mode=0)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    L = moe.lib()
    for call in range(2):
        x_out = torch.empty_like(ref)
        x_out.view(torch.uint8).fill_(0x33 + call)
        rc = L.moe_combine_noalloc(
            ctypes.byref(cfg), ctypes.c_void_p(got["expand_x"].data_ptr()),
            ctypes.c_void_p(got["assist_info"].data_ptr()), ctypes.c_void_p(got["ep_recv_count"].data_ptr()),
            ctypes.c_void_p(dev["expert_ids"].data_ptr()), ctypes.c_void_p(dev["expert_scales"].data_ptr()),
            None if dev["active_mask"] is None else ctypes.c_void_p(dev["active_mask"].data_ptr()),
            ctypes.c_void_p(dev["x"].data_ptr()), ctypes.c_void_p(x_out.data_ptr()),
            ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, moe.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # the tolerance the other combine tests use, and the bytes themselves
        H.compare_combine(wl, H.to_host(x_out), H.to_host(ref))
        assert torch.equal(x_out, ref)


def test_noalloc_rejects_calls_beyond_its_scratch(moe):
    cfg = moe.config(16, 4096, 64, 8, 256, torch.bfloat16)  # 524288 picks > 262144
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.combine_noalloc(cfg, t, t, t, t, t, None, t, t, status)
    assert ei.value.name == "INVALID_ARG"
