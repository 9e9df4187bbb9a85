"""The multi-shape sweep tool (combine_route_scan_gb300.sweep): its grid and CSV
writing on the CPU, one small sweep on the GPU."""
import csv
import os

import pytest
import torch

from combine_route_scan_gb300 import sweep as S


def test_grid_follows_the_lists_and_skips_impossible_topk():
    args = S.parse_args(["--pes-list", "2,4", "--bs-list", "8", "--h-list", "64,256", "--topk-list", "2,8",
                         "--expert-per-pe-list", "1,2"])
    got = list(S.shapes(args))
    assert (2, 8, 64, 2, 1) in got and (4, 8, 256, 8, 2) in got
    assert (2, 8, 64, 8, 1) not in got       # 8 picks from 2 experts
    # 16 combinations; K = 8 needs W * L >= 8, which only (W 4, L 2) gives: 6 dropped
    assert len(got) == 10
    assert all(K <= W * L for W, _, _, K, L in got)


def test_csv_writer_formats_floats(tmp_path):
    p = tmp_path / "x.csv"
    S.write_csv(str(p), ["a", "b"], [{"a": 1, "b": 2.345678}])
    rows = list(csv.DictReader(open(p)))
    assert rows == [{"a": "1", "b": "2.346"}]


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["int32", "bf16"])
def test_small_sweep_on_gpu(tmp_path, dtype):
    out = tmp_path / "sweep"
    rc = S.main(["--pes-list", "2,4", "--bs-list", "8", "--h-list", "64,256", "--topk-list", "2",
                 "--expert-per-pe-list", "2", "--type", dtype, "--warmup", "2", "--loops", "5",
                 "--out-dir", str(out)])
    assert rc == 0
    summary = list(csv.DictReader(open(out / "perf_summary.csv")))
    assert len(summary) == 4 and all(r["two_phase_matches_gather"] == "True" for r in summary)
    assert all(float(r["full_op_us"]) > 0 and float(r["comm_only_us"]) > 0 for r in summary)
    for d in range(4):
        rows = list(csv.DictReader(open(out / f"perf_rank{d}.csv")))
        assert len(rows) == (4 if d < 2 else 2)    # ranks 2, 3 exist only in the 4-rank shapes
        assert set(S.RANK_FIELDS) == set(rows[0])
    # the per-rank received rows add up to the routed total: W * bs * K picks
    for s in summary:
        W = int(s["pes"])
        tot = sum(int(r["recv_rows"]) for d in range(W) for r in csv.DictReader(open(out / f"perf_rank{d}.csv"))
                  if r["pes"] == s["pes"] and r["h"] == s["h"])
        assert tot == int(s["routed_rows"]) == W * 8 * 2
