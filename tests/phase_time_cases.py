"""Cases for the phase-time test build (run by test_phase_times_gpu.py in a
child process with CRS_MOE_PHASE=1; collected only when named on the command
line).

Every kernel of a call records (%globaltimer) its earliest CTA start, the
earliest and latest passage of its CTAs past the wait for the previous
kernel's results, and its latest CTA end. The small 7168-hidden workload is
timed as the bench times it: a 512 MB write before every step, CUDA events
around dispatch and combine, medians over the steps; each phase is printed in
microseconds from the routing kernel's first CTA start, next to the event
times and the launch floor (events around one kernel touching 16 bytes)."""
import ctypes
import os
import statistics

import numpy as np
import pytest
import torch

import workloads as WL

pytestmark = pytest.mark.gpu

if os.environ.get("CRS_MOE_PHASE") != "1":
    pytest.skip("needs the phase-time build (CRS_MOE_PHASE=1)", allow_module_level=True)

import gpu_harness as H  # noqa: E402
from combine_route_scan_gb300 import moe as M  # noqa: E402

KERNELS = ("routing", "scatter", "inverse map", "reduce")


def phase_table(name, steps=30):
    wl = WL.WORKLOADS[name]
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    cfg = H.make_cfg(wl)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_dispatch_outputs(cfg, H.TORCH_DT[wl.x_dtype])
    x_out = torch.empty_like(dev["x"])
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    tiny = torch.zeros(4, dtype=torch.int32, device="cuda")
    buf = torch.zeros(16, dtype=torch.int64, device="cuda")
    lib = M.lib()
    lib.moe_test_set_phase_buffer.argtypes = [ctypes.c_void_p]
    lib.moe_test_set_phase_buffer.restype = ctypes.c_int32
    assert lib.moe_test_set_phase_buffer(ctypes.c_void_p(buf.data_ptr())) == 0
    st = torch.cuda.current_stream()
    phases, disp, comb, floor = [], [], [], []
    try:
        for i in range(steps + 3):
            flush.fill_(i & 0xFF)
            buf.zero_()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            ev[0].record(st)
            M.dispatch(cfg, dev["x"], dev["expert_ids"], dev["active_mask"], dev["expert_scales"], out["expand_x"],
                       out["dynamic_scales"], out["assist_info"], out["ep_recv_count"], out["expand_scales"], None, ws)
            ev[1].record(st)
            if wl.quant_mode == 0:
                M.combine(cfg, out["expand_x"], out["assist_info"], out["ep_recv_count"], dev["expert_ids"],
                          dev["expert_scales"], dev["active_mask"], dev["x"], x_out, None, ws)
            ev[2].record(st)
            flush.fill_((i + 1) & 0xFF)
            ev[3].record(st)
            tiny.add_(1)
            ev[4].record(st)
            torch.cuda.synchronize()
            if i >= 3:
                phases.append(buf.cpu().numpy().view(np.uint64).copy())
                disp.append(ev[0].elapsed_time(ev[1]) * 1e3)
                comb.append(ev[1].elapsed_time(ev[2]) * 1e3)
                floor.append(ev[3].elapsed_time(ev[4]) * 1e3)
    finally:
        lib.moe_test_set_phase_buffer(None)
    assert M.get_device_status(ws) == 0

    def rel(t, k, j):  # phase j of kernel k in us from the routing start, or None
        v = t[4 * k + j]
        if v == 0:
            return None
        v = ~v if j in (0, 1) else v
        return (int(np.uint64(v)) - int(np.uint64(~t[0]))) / 1e3

    rows = []
    for k, kname in enumerate(KERNELS):
        vals = [[rel(t, k, j) for t in phases] for j in range(4)]
        if vals[0][0] is None:
            continue
        med = [statistics.median(v) for v in vals]
        rows.append((kname, med))
    print(f"\n{name}: median over {len(phases)} steps, us from the routing kernel's first CTA start")
    print("| kernel | first CTA start | first CTA past the wait | last CTA past the wait | last CTA end |")
    print("|---|---|---|---|---|")
    for kname, m in rows:
        print(f"| {kname} | {m[0]:.1f} | {m[1]:.1f} | {m[2]:.1f} | {m[3]:.1f} |")
    print(f"CUDA events: dispatch {statistics.median(disp):.1f} us, combine {statistics.median(comb):.1f} us; "
          f"one kernel touching 16 bytes {statistics.median(floor):.1f} us")
    return dict(rows)


@pytest.mark.parametrize("name", ["w8_bs32_h7168_k8_e64_f16", "w8_bs32_h7168_k8_e64_i32"])
def test_small_workload_phases(name):
    r = phase_table(name)
    route, scatter, reduce = r["routing"], r["scatter"], r["reduce"]
    # each kernel passes its wait only once the previous grid has ended
    assert scatter[1] >= route[3] - 0.05 and reduce[1] >= scatter[3] - 0.05
    for m in (route, scatter, reduce):
        assert m[0] <= m[1] <= m[2] <= m[3] + 0.05
