"""The bench's multi-rank host logic on CPU, world size 2 over gloo: per-rank
seeds, max over ranks of the timings, whole-job aggregation, and the
reference arm running on rank 0 only."""
import importlib.util
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    B = _bench()
    wl = B.WL.WORKLOADS["w2_bs8_h16_k2_e4_i32"]
    local_ms = 10.0 + 5.0 * rank
    m = B.max_over_ranks(local_ms, world)
    seed = B.rank_seed(wl, rank)
    dist.barrier()
    q.put((rank, m, seed))
    dist.destroy_process_group()


def test_two_ranks_max_and_seeds():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [15.0, 15.0]  # every rank sees the slowest rank's time
    assert out[0][2] != out[1][2]  # independent batches


def test_whole_job_aggregation():
    B = _bench()
    # two ranks, 100 MB per step each, 10 steps in 1 ms (max over ranks)
    assert B.whole_job_gbps(100_000_000, 10, 1.0, 2) == pytest.approx(2000.0)
    assert B.whole_job_gbps(100_000_000, 10, 1.0, 1) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    B = _bench()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        workload = "w2_bs8_h16_k2_e4_i32"
        steps = 1
        warmup = 0
        gpus = 2
    assert B.run_reference(A()) == 0
    assert capsys.readouterr().out == ""


def test_rotation_sets_keep_steps_out_of_l2():
    """Timed regions rotate over enough buffer sets that a set's data has left
    the L2 before it is used again; a step larger than four L2s needs one."""
    B = _bench()
    assert B.rotation_sets(4 * B.L2_BYTES) == 1
    assert B.rotation_sets(931_000_000) == 1
    n = B.rotation_sets(66_000_000)
    assert n >= 2 and n * 66_000_000 >= 4 * B.L2_BYTES and (n - 1) * 66_000_000 < 4 * B.L2_BYTES
    cfg = B.bench_config(B.WL.WORKLOADS["w8_bs32_h7168_k8_e64_f16"], None, 66_000_000)
    assert f"{n} buffer sets" in cfg["l2"]


@pytest.mark.parametrize("bs,n", [(256, 16), (256, 7), (8, 16), (1, 4), (10, 3)])
def test_token_slices_cover_the_batch_once(bs, n):
    B = _bench()
    parts = B.token_slices(bs, n)
    assert len(parts) == min(n, bs)
    assert parts[0][0] == 0 and parts[-1][1] == bs
    assert all(a < b for a, b in parts)
    assert all(parts[i][1] == parts[i + 1][0] for i in range(len(parts) - 1))


def test_oracle_threads_give_the_serial_results():
    """The all-cores CPU baseline runs the oracle on several threads at once;
    the C oracle must then give every slice the bytes it gives it alone."""
    import threading

    import numpy as np
    from oracle import oracle as O
    B = _bench()
    wl = B.WL.WORKLOADS["w8_bs8_h16_k2_e64_f16"]
    inp = B.WL.make_inputs(wl)
    parts = [B.subsample(wl, inp, b - a, start=a) for a, b in B.token_slices(wl.bs, 4)]

    def run(swl, sinp):
        d = O.dispatch(swl, sinp)
        y = O.combine(swl, d["expand_x"], d["assist_info"], d["ep_recv_count"], sinp)
        return d, y

    serial = [run(*p) for p in parts]
    got = [None] * len(parts)

    def worker(i):
        for _ in range(20):
            got[i] = run(*parts[i])

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(len(parts))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    for (d0, y0), (d1, y1) in zip(serial, got):
        for k in ("expand_x", "assist_info", "ep_recv_count", "expand_scales"):
            np.testing.assert_array_equal(d0[k], d1[k])
        np.testing.assert_array_equal(np.asarray(y0), np.asarray(y1))
    # the slices are the batch's tokens, in order
    np.testing.assert_array_equal(np.concatenate([p[1]["x"] for p in parts], axis=1), inp["x"])


def test_all_cores_baseline_counts_whole_slices():
    B = _bench()
    wl = B.WL.WORKLOADS["w2_bs8_h16_k2_e4_i32"]
    inp = B.WL.make_inputs(wl)
    r = B.time_oracle_all_cores(wl, inp, target_s=0.2, threads=3)
    assert r["threads"] == 3 and r["tokens_per_slice"] == (2, 3)
    per = [sum(v for k, v in B.algorithmic_bytes(*B.subsample(wl, inp, b - a, start=a)).items()
               if k in ("dispatch", "combine")) for a, b in B.token_slices(wl.bs, 3)]
    assert r["slices_done"] >= 3 and r["seconds"] >= 0.2
    assert min(per) * r["slices_done"] <= r["bytes"] <= max(per) * r["slices_done"]


def test_reference_arm_line_on_rank_zero(monkeypatch, capsys):
    import json
    B = _bench()
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")

    class A:
        workload = "w8_bs8_h16_k2_e64_f16"
        steps = 2
        warmup = 1
        gpus = 1
        plane_policy = 0
    assert B.run_reference(A()) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert 1 <= line["cpu_baseline"]["cores"] <= min(B.host_cores(), 8)
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "w8_bs8_h16_k2_e64_f16"
