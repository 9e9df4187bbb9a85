"""Where a small call's time goes: runs tests/phase_time_cases.py in a child
process against the phase-time test build (-DMOE_PHASE_TIMES,
CRS_MOE_PHASE=1), which records every kernel's %globaltimer phases, and
prints the table for the small 7168-hidden workload (8 ranks x 32 tokens)
next to the call's CUDA-event times and the launch floor, all timed after a
512 MB write as the bench times the calls."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_small_workload_phase_table():
    from combine_route_scan_gb300 import build as B
    lib = B.build(phase=True)
    assert os.path.exists(lib)
    # the child loads this build alone, whatever build the parent selected
    env = {k: v for k, v in os.environ.items() if k not in ("CRS_MOE_CHECKED", "CRS_MOE_OBSERVER", "CRS_MOE_PHASE")}
    env["CRS_MOE_PHASE"] = "1"
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/phase_time_cases.py", "-q", "-x", "-s", "-m", "gpu",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"{r.stdout[-4000:]}\n{r.stderr[-2000:]}"
    assert " passed" in r.stdout, r.stdout[-2000:]
    print(r.stdout[-3000:])
