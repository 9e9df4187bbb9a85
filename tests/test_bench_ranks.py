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
