"""The bounds-checked build (-DMOE_BOUNDS_CHECK: every index a kernel derives
from data is checked against its buffer; a miss records MOE_ERR_OUT_OF_BOUNDS
and skips the access) runs a selection of the parity tests clean: same bytes
as the oracle, status OK. It runs in a child process because the library is
loaded once per process (CRS_MOE_CHECKED=1 picks the checked one)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SELECTION = [
    ("tests/test_parity_gpu.py", "random_small or empty_batch or ready_flags or two_phase_matches or reuses "
                                 "or row_map or performance_info or one_expert or all_masked"),
    ("tests/test_quant_gpu.py", "small_tma_rows or ragged or bulk_plane or random_shapes or expert_major "
                               "or (many_tokens_per_cta and (q2_int8_s3 or q3_fp8_e4m3_s0 or q3_fp8_e4m3_s3 or q4_fp4_e2m1_s0))"),
    ("tests/test_ffn_gpu.py", "small_all_tokens or several_token_passes"),
]


def test_checked_build_runs_the_parity_selection():
    from combine_route_scan_gb300 import build as B
    lib = B.build(checked=True)
    assert os.path.exists(lib)
    # the child loads this build alone, whatever build the parent selected
    env = {k: v for k, v in os.environ.items() if k not in ("CRS_MOE_CHECKED", "CRS_MOE_OBSERVER", "CRS_MOE_PHASE")}
    env["CRS_MOE_CHECKED"] = "1"
    probe = subprocess.run([sys.executable, "-c", "from combine_route_scan_gb300 import moe; print(moe.lib()._name)"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert probe.returncode == 0 and os.path.join("_build", "checked") in probe.stdout, probe.stdout + probe.stderr
    for path, expr in SELECTION:
        r = subprocess.run([sys.executable, "-m", "pytest", path, "-k", expr, "-q", "-x", "-m", "gpu",
                            "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
        assert r.returncode == 0, f"{path}:\n{r.stdout[-3000:]}\n{r.stderr[-2000:]}"
        assert " passed" in r.stdout


def test_two_phase_rejects_counts_beyond_capacity():
    """A receive count above the capacity A is reported (not followed past
    rank d's rows) by the two-phase combine, as by the gather combine."""
    import numpy as np
    import torch
    import workloads as WL
    import gpu_harness as H
    from combine_route_scan_gb300 import moe as M
    from oracle import oracle as O
    wl = WL.WORKLOADS["w8_bs8_h16_k2_e64_f16"]
    inp = WL.make_inputs(wl)
    dev = H.device_inputs(wl, inp)
    got, _, _ = H.gpu_dispatch(wl, dev)
    ep = got["ep_recv_count"].clone()
    ep[-1, -1] = O.capacity(wl) + 5
    for mode in (M.COMBINE_GATHER, M.COMBINE_TWO_PHASE, M.COMBINE_PUT_ONLY):
        _, st, _ = H.gpu_combine(wl, dev, got["expand_x"], got["assist_info"], ep, combine_mode=mode,
                                 check_status=False)
        assert M.STATUS[st] == "BAD_ASSIST", (mode, M.STATUS[st])
