"""A ready flag is never visible before its segment's rows (the
combine_doubleplane README, 实现逻辑: status written only after the payload).

Runs tests/flag_observer_cases.py in a child process against the
flag-observer test build (-DMOE_FLAG_OBSERVER, CRS_MOE_OBSERVER=1): the
dispatch payload grid's last CTA, launched cooperatively with the storing
CTAs, acquire-polls every flag with a bounded wait and copies each segment as
soon as its flag shows the call's ticket; the copies are compared with the
final output and the oracle. The observer is part of the same launch, so no
kernel waits on a separately launched one."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_flags_never_precede_their_rows():
    from combine_route_scan_gb300 import build as B
    lib = B.build(observer=True)
    assert os.path.exists(lib)
    # the child loads this build alone, whatever build the parent selected
    env = {k: v for k, v in os.environ.items() if k not in ("CRS_MOE_CHECKED", "CRS_MOE_OBSERVER", "CRS_MOE_PHASE")}
    env["CRS_MOE_OBSERVER"] = "1"
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/flag_observer_cases.py", "-q", "-x", "-s", "-m", "gpu",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"{r.stdout[-4000:]}\n{r.stderr[-2000:]}"
    assert " passed" in r.stdout and "skipped" not in r.stdout.split("\n")[-2], r.stdout[-2000:]
    print(r.stdout[-2000:])
