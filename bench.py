#!/usr/bin/env python
"""Dispatch + combine throughput of the GB300 MoE library.

One step = one pass of the whole hot path over one batch: moe_dispatch (route +
scatter, with expand_scales) then moe_combine (inverse map + gather reduce)
with the identity expert (the expert output is expand_x), as in the
combine_doubleplane example. Default workload: skewed (Zipf) routing, W=16
emulated EP ranks, bs=256 tokens per rank, h=7168, topk 8, 256 experts plus 4
zero and 4 copy experts, 2D active mask, bf16 data.

Prints one JSON line. ``value`` is the algorithmic bytes of dispatch + combine
moved per second (GB/s, whole job over all ranks); ``tokens_per_s`` and the
fraction of the 8 TB/s HBM roofline ride along. ``--impl reference`` times the
CPU oracle on the same workload instead, on all host cores (the reference arm).

Multi-GPU (torchrun): every rank runs its own independent batch (the W
emulated ranks live inside each GPU), no collective on the data path; weak
scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402

METRIC = "dispatch+combine GB/s and tokens/s on 1 GB300; fraction of 8 TB/s HBM roofline"
DEFAULT_WORKLOAD = "w16_bs256_h7168_k8_e256_bf16_zipf"
FFN_WORKLOAD = "w8_bs64_h2048_k8_e128_bf16_ffn"
SMALL_WORKLOADS = ("w8_bs32_h7168_k8_e64_f16", "w8_bs32_h7168_k8_e64_f16_q2", "w8_bs32_h7168_k8_e64_i32")
# quantised dispatch variants: quantMode, expanded element type, scales input kind
QUANT_MODES = ("q2_int8_s0", "q1_int8_s1", "q2_int8_s3", "q3_fp8_e4m3_s0", "q3_fp8_e4m3_s3", "q4_fp8_e4m3_s0",
               "q4_fp4_e2m1_s0")
HBM_NOMINAL_GBPS = 8000.0
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBPS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WL.WORKLOADS))
    ap.add_argument("--plane-policy", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--ffn-workload", default=FFN_WORKLOAD, choices=sorted(WL.WORKLOADS))
    ap.add_argument("--no-ffn", action="store_true")
    ap.add_argument("--ffn-steps", type=int, default=100)
    ap.add_argument("--small-workloads", default=",".join(SMALL_WORKLOADS),
                    help="workloads that fit in L2, timed per call with an L2 flush before each step")
    ap.add_argument("--small-steps", type=int, default=50)
    ap.add_argument("--quant-modes", default=",".join(QUANT_MODES),
                    help="quantised dispatch variants timed on the main workload (mode/type/scales)")
    ap.add_argument("--quant-steps", type=int, default=50)
    ap.add_argument("--only-quant", action="store_true",
                    help="time only the quantised dispatch variants (for profiling); prints their JSON")
    ap.add_argument("--only-small", action="store_true",
                    help="time only the small (L2-sized) workloads and their floors; prints their JSON")
    return ap.parse_args()


# ------------------------------------------------------------ accounting

def pick_counts(wl: WL.Workload, inp: dict) -> dict:
    """Routed picks P, copy picks, tokens with at least one routed pick."""
    ids = inp["expert_ids"].astype(np.int64)
    E, Z, C = wl.moe_expert_num, wl.zero_expert_num, wl.copy_expert_num
    act = np.ones(ids.shape, dtype=bool)
    m = inp.get("active_mask")
    if m is not None:
        act = np.broadcast_to(m.astype(bool)[..., None], ids.shape) if m.ndim == 2 else m.astype(bool)
    routed = act & (ids >= 0) & (ids < E)
    copy = act & (ids >= E + Z) & (ids < E + Z + C)
    return {"P": int(routed.sum()), "copy": int(copy.sum()), "tok_routed": int(routed.any(-1).sum())}


def row_out_bytes(wl: WL.Workload) -> int:
    """Bytes of one expand_x row: x's row unquantised, h for int8 / fp8, h / 2
    for packed fp4."""
    if wl.quant_mode == 0:
        return wl.h * wl.es
    return wl.h // 2 if wl.y_dtype == "fp4_e2m1" else wl.h


def algorithmic_bytes(wl: WL.Workload, inp: dict) -> dict:
    """Bytes the method must move (inputs read once, outputs written once)."""
    c = pick_counts(wl, inp)
    W, bs, K, h = wl.ep_world_size, wl.bs, wl.topk, wl.h
    L = wl.moe_expert_num // W
    r_in = h * wl.es
    r_out = row_out_bytes(wl)
    picks = W * bs * K
    mask = 0 if inp.get("active_mask") is None else inp["active_mask"].size
    ep = W * L * W * 4
    P, Cp, Nt = c["P"], c["copy"], c["tok_routed"]
    meta = P * (4 + 12 + 4)  # weights read; assist, expand_scales written
    # dynamic scales written: one fp32 per row (mode 2), per 128-group (3), one byte per 32-block (4)
    dyn = {2: 4, 3: 4 * ((h + 127) // 128), 4: (h + 31) // 32}.get(wl.quant_mode, 0)
    # the scales input, read once: (1,), (h,) or (E, h) fp32
    qs = {1: 4, 2: h * 4, 3: wl.moe_expert_num * h * 4}.get(wl.scales_kind, 0) if wl.quant_mode else 0
    scatter = Nt * r_in + P * r_out + meta + P * dyn + qs
    dispatch = scatter + picks * 4 + mask + ep
    reduce_ = P * r_in + Cp * r_in + picks * 8 + mask + W * bs * r_in
    combine = reduce_ + P * 12 + ep
    return {"dispatch": dispatch, "combine": combine, "scatter": scatter, "reduce": reduce_, **c}


# ------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples with host timestamps."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                self.samples.append((time.time(), float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i, v in enumerate(s[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside)}


def gpu_id_for_smi(local_rank: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[local_rank] if vis else str(local_rank)


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBPS, "source": "fallback"}


# the source files each profiled kernel is built from
KERNEL_SOURCES = {
    "scatter": ("scatter.cu", "scatter_common.cuh", "common.cuh", "internal.h"),
    "scatter_quant": ("scatter_quant.cu", "scatter_common.cuh", "common.cuh", "internal.h"),
    "combine_reduce": ("combine.cu", "common.cuh", "internal.h"),
}


def source_hash(kernel: str) -> str:
    """First 16 hex digits of the sha256 over the kernel's source files."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "combine_route_scan_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (their hash is recorded beside the figure)."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(p):
        return None
    h = source_hash(kernel)
    vals = {}
    with open(p) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256_16") != h or "dram_bytes_per_launch_full_size" not in vals:
        return None
    return float(vals["dram_bytes_per_launch_full_size"])


# ------------------------------------------------------------ oracle timing

def time_oracle(wl: WL.Workload, inp: dict, target_s: float, max_steps: int = 20):
    from oracle import oracle as O
    t = []
    while True:
        t0 = time.perf_counter()
        d = O.dispatch(wl, inp)
        O.combine(wl, d["expand_x"], d["assist_info"], d["ep_recv_count"], inp)
        t.append(time.perf_counter() - t0)
        if sum(t) >= target_s or len(t) >= max_steps:
            return t


def subsample(wl: WL.Workload, inp: dict, bs: int, start: int = 0):
    """Tokens [start, start + bs) of every rank (same routing law, smaller batch)."""
    sub = wl.with_(bs=bs, name=wl.name + (f"_first{bs}" if start == 0 else f"_tokens{start}_{start + bs}"))
    out = {k: (None if v is None else np.ascontiguousarray(v[:, start:start + bs])) for k, v in inp.items()
           if k in ("x", "expert_ids", "active_mask", "expert_scales")}
    return sub, out


def host_cores() -> int:
    """Cores this process may run on."""
    if hasattr(os, "sched_getaffinity"):
        return len(os.sched_getaffinity(0))
    return os.cpu_count() or 1


def token_slices(bs: int, n: int):
    """`n` contiguous token ranges (at most `bs` of them) that cover [0, bs) once."""
    n = max(1, min(n, bs))
    return [(i * bs // n, (i + 1) * bs // n) for i in range(n)]


def time_oracle_all_cores(wl: WL.Workload, inp: dict, target_s: float, threads: int = 0) -> dict:
    """The unchanged oracle on every host core at once. The batch's tokens are
    split into one contiguous slice per thread (every rank's tokens [a, b)); each
    slice is a smaller problem of the same routing law, and each thread runs
    dispatch + combine on its own slice over and over until `target_s` has
    passed. ctypes lets go of the GIL inside the C calls, so the threads run in
    parallel. Throughput = algorithmic bytes of every completed slice / the
    time until the last thread finished its last slice."""
    from oracle import oracle as O
    n = threads or host_cores()
    parts = [subsample(wl, inp, b - a, start=a) for a, b in token_slices(wl.bs, n)]
    part_bytes = [sum(v for k, v in algorithmic_bytes(swl, sinp).items() if k in ("dispatch", "combine"))
                  for swl, sinp in parts]
    done = [0] * len(parts)
    ends = [0.0] * len(parts)
    errors = []
    go = threading.Barrier(len(parts) + 1)
    t0 = [0.0]

    def run(i):
        swl, sinp = parts[i]
        try:
            go.wait()
            while True:
                d = O.dispatch(swl, sinp)
                O.combine(swl, d["expand_x"], d["assist_info"], d["ep_recv_count"], sinp)
                done[i] += 1
                ends[i] = time.perf_counter()
                if ends[i] - t0[0] >= target_s:
                    return
        except Exception as e:  # reported by the caller
            errors.append(e)

    workers = [threading.Thread(target=run, args=(i,), daemon=True) for i in range(len(parts))]
    for w in workers:
        w.start()
    t0[0] = time.perf_counter()
    go.wait()
    for w in workers:
        w.join()
    if errors:
        raise errors[0]
    elapsed = max(ends) - t0[0]
    moved = sum(c * b for c, b in zip(done, part_bytes))
    return {"bytes": moved, "seconds": elapsed, "threads": len(parts), "slices_done": sum(done),
            "tokens_per_slice": (min(b - a for a, b in token_slices(wl.bs, n)),
                                 max(b - a for a, b in token_slices(wl.bs, n)))}


# ------------------------------------------------------------ distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(wl: WL.Workload, rank: int) -> int:
    """Every rank draws its own independent batch."""
    return wl.seed + rank


def max_over_ranks(v: float, world: int) -> float:
    """The slowest rank's value (barrier-bracketed timings are maxed)."""
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(step_bytes: int, steps: int, max_ms: float, world: int) -> float:
    """Bytes every rank moved over all timed steps, divided by the slowest
    rank's time (weak scaling: each rank has its own batch)."""
    return world * step_bytes * steps / (max_ms * 1e-3) / 1e9


def rotation_sets(step_bytes: int) -> int:
    """Buffer sets the timed regions rotate over: one when a step moves more
    than four times the L2, else enough that a set's data has left the L2
    before it is used again."""
    return 1 if step_bytes >= 4 * L2_BYTES else int(np.ceil(4 * L2_BYTES / step_bytes))


def bench_config(wl: WL.Workload, args, step_bytes: int) -> dict:
    """The `config` object of the JSON line, the same for both arms."""
    n_sets = rotation_sets(step_bytes)
    l2 = (f"no flush: one step moves {step_bytes / 1e6:.0f} MB (> 4x the {L2_BYTES >> 20} MiB L2)" if n_sets == 1 else
          f"no flush: steps rotate over {n_sets} buffer sets of {step_bytes / 1e6:.0f} MB each "
          f"(> 4x the {L2_BYTES >> 20} MiB L2 together)")
    return {"workload": wl.name, "ep_world_size": wl.ep_world_size, "bs": wl.bs, "h": wl.h,
            "topk": wl.topk, "moe_expert_num": wl.moe_expert_num, "zero_experts": wl.zero_expert_num,
            "copy_experts": wl.copy_expert_num, "mask": wl.mask_kind, "quant_mode": wl.quant_mode,
            "plane_policy": getattr(args, "plane_policy", 0), "combine": "gather",
            "l2": l2,
            "accumulate": "fp32"}


def oracle_step_all_cores(pool, parts) -> float:
    """One step of the unchanged oracle on the host's cores: every token slice
    (see time_oracle_all_cores) goes through dispatch + combine once, one slice
    a thread; returns the wall time until the last slice is done."""
    from oracle import oracle as O

    def run(p):
        swl, sinp = p
        d = O.dispatch(swl, sinp)
        O.combine(swl, d["expand_x"], d["assist_info"], d["ep_recv_count"], sinp)

    t0 = time.perf_counter()
    for f in [pool.submit(run, p) for p in parts]:
        f.result()
    return time.perf_counter() - t0


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from concurrent.futures import ThreadPoolExecutor
    wl = WL.WORKLOADS[args.workload]
    inp = WL.make_inputs(wl)
    from oracle import build as OB
    OB.build()
    n = host_cores()
    # size each step so that warmup + steps end within about three minutes
    budget = 180.0
    steps = max(1, args.steps + args.warmup)
    bs = wl.bs
    with ThreadPoolExecutor(max_workers=n) as pool:
        def parts_of(b):
            swl, sinp = (wl, inp) if b == wl.bs else subsample(wl, inp, b)
            return swl, sinp, [subsample(swl, sinp, e - a, start=a) for a, e in token_slices(b, n)]
        swl, sinp, parts = parts_of(bs)
        one = oracle_step_all_cores(pool, parts)
        while bs > 1 and one * (bs / wl.bs) * steps > budget:
            bs //= 2
        if bs != wl.bs:
            swl, sinp, parts = parts_of(bs)
        times = []
        for i in range(args.warmup + args.steps):
            dt = oracle_step_all_cores(pool, parts)
            if i >= args.warmup:
                times.append(dt)
    b = sum(v for p in parts for k, v in algorithmic_bytes(*p).items() if k in ("dispatch", "combine"))
    total = sum(times)
    gbps = b * len(times) / total / 1e9
    lo = min(e - a for a, e in token_slices(bs, n))
    hi = max(e - a for a, e in token_slices(bs, n))
    sample = (f"{len(times)} timed oracle steps of dispatch+combine over "
              + ("the full batch" if bs == wl.bs else f"the first {bs} of {wl.bs} tokens of every rank")
              + f", unchanged single-threaded C on {len(parts)} threads at once, each on its own slice of "
              + f"{lo}" + (f"-{hi}" if hi != lo else "") + " tokens of every rank")
    full = algorithmic_bytes(wl, inp)
    line = {
        "impl": "reference", "metric": METRIC, "value": gbps, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / len(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(wl, args, full["dispatch"] + full["combine"]),
        "tokens_per_s": swl.ep_world_size * swl.bs * len(times) / total,
        "cpu_baseline": {"value": gbps, "unit": "GB/s", "cores": len(parts), "kind": "oracle", "sample": sample},
        "e2e": {"value": gbps, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def measure_ffn(args, M, torch, stream):
    """moe_dispatch_ffn_combine on the decode-layer workload: whole call, and
    the gate/up GEMM alone (CUDA events the library records around it)."""
    wl = WL.WORKLOADS[args.ffn_workload]
    inp = WL.make_inputs(wl)
    I, E, h = wl.ffn_intermediate, wl.moe_expert_num, wl.h

    def dev(a, bf):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf else np.ascontiguousarray(a))
        return (t.view(torch.bfloat16) if bf else t).cuda()

    x, ids = dev(inp["x"], True), dev(inp["expert_ids"], False)
    scales = dev(inp["expert_scales"], False)
    mask = None if inp.get("active_mask") is None else dev(inp["active_mask"], False)
    wg, wu, wd = (dev(inp[k], True) for k in ("w_gate", "w_up", "w_down"))
    cfg = M.config(wl.ep_world_size, wl.bs, h, wl.topk, E, torch.bfloat16, zero_expert_num=wl.zero_expert_num,
                   copy_expert_num=wl.copy_expert_num, mask_kind=wl.mask_kind, ffn_intermediate=I)
    ws = M.alloc_workspace(cfg)
    x_out = torch.empty_like(x)
    for _ in range(3):
        M.dispatch_ffn_combine(cfg, x, ids, mask, scales, wg, wu, wd, x_out, ws)
    torch.cuda.synchronize()
    Kf = max(1, args.ffn_steps)
    evs = [M.ProfEvents() for _ in range(Kf)]
    cfgs = [e.attach(cfg) for e in evs]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for c in cfgs:
        M.dispatch_ffn_combine(c, x, ids, mask, scales, wg, wu, wd, x_out, ws)
    b.record(stream)
    torch.cuda.synchronize()
    st = M.get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {M.STATUS.get(st, st)} in the FFN variant")
    call_ms = a.elapsed_time(b) / Kf
    ffn_ms = statistics.mean(e.elapsed_ms() for e in evs)  # the FFN kernel (both GEMMs, one launch)
    acct = algorithmic_bytes(wl, inp)
    P = acct["P"]
    w_bytes = 3 * E * I * h * 2
    # weights + token rows in + h1 out and back in + y out
    ffn_bytes = w_bytes + P * h * 2 + 2 * P * I * 2 + P * h * 2
    flops = 2 * P * (3 * I * h)
    peaks = measured_peaks()
    return {"workload": wl.name, "ms_per_call": call_ms, "tokens_per_s": wl.ep_world_size * wl.bs / (call_ms * 1e-3),
            "weight_bytes": w_bytes, "routed_picks": P,
            "call_GBps": (w_bytes + acct["dispatch"] + acct["combine"]) / (call_ms * 1e-3) / 1e9,
            "call_TFLOPs": flops / (call_ms * 1e-3) / 1e12,
            "ffn_gemm_ms": ffn_ms, "ffn_gemm_GBps": ffn_bytes / (ffn_ms * 1e-3) / 1e9,
            "ffn_gemm_frac_of_hbm": ffn_bytes / (ffn_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "ffn_gemm_TFLOPs": flops / (ffn_ms * 1e-3) / 1e12,
            "steps": Kf}


def measure_floor(torch, stream, flush, n, ops: dict) -> dict:
    """What one GPU gives a call of this size at all, timed exactly as the
    calls are (512 MB written before every step, CUDA events around the call):
    the launch floor (events around one kernel that touches 16 bytes) and, per
    operation, a plain device-to-device copy moving the operation's
    algorithmic bytes (half read, half written)."""
    tiny = torch.zeros(4, dtype=torch.int32, device="cuda")
    big = max(ops.values())
    src = torch.empty(big // 2 + 16, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)

    def timed(fn):
        ts = []
        for i in range(n + 3):
            flush.fill_((i + 7) & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            if i >= 3:
                ts.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ts)

    res = {"launch_ms": timed(lambda: tiny.add_(1)),
           "how": "median over steps of CUDA-event times after a 512 MB write, as for the calls; the copy is "
                  "torch's device-to-device copy_ of half the operation's algorithmic bytes"}
    for op, nbytes in ops.items():
        half = nbytes // 2
        ms = timed(lambda: dst[:half].copy_(src[:half]))
        res[f"{op}_copy_ms"] = ms
        res[f"{op}_copy_GBps"] = 2 * half / (ms * 1e-3) / 1e9
        res[f"{op}_copy_frac_of_8TBps"] = 2 * half / (ms * 1e-3) / 1e9 / HBM_NOMINAL_GBPS
    del src, dst, tiny
    return res


def measure_small(args, M, torch, stream):
    """Workloads whose working set fits in L2: each step first writes a 512 MB
    buffer (untimed) so dispatch and combine read and write HBM, then times
    moe_dispatch and moe_combine separately with CUDA events."""
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    res = {}
    for name in [w for w in args.small_workloads.split(",") if w]:
        wl = WL.WORKLOADS[name]
        inp = WL.make_inputs(wl)
        bf = wl.x_dtype == WL.X_BF16
        tdt = {WL.X_INT32: torch.int32, WL.X_FP16: torch.float16, WL.X_BF16: torch.bfloat16}[wl.x_dtype]

        def dev(a, as_bf=False):
            if a is None:
                return None
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if as_bf else np.ascontiguousarray(a))
            return (t.view(torch.bfloat16) if as_bf else t).cuda()

        x, ids, scales, mask = dev(inp["x"], bf), dev(inp["expert_ids"]), dev(inp["expert_scales"]), \
            dev(inp.get("active_mask"))
        cfg = M.config(wl.ep_world_size, wl.bs, wl.h, wl.topk, wl.moe_expert_num, tdt,
                       zero_expert_num=wl.zero_expert_num, copy_expert_num=wl.copy_expert_num,
                       quant_mode=wl.quant_mode, mask_kind=wl.mask_kind)
        ws = M.alloc_workspace(cfg)
        out = M.alloc_dispatch_outputs(cfg, tdt)
        x_out = torch.empty_like(x)
        n = max(3, args.small_steps)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        for i in range(n + 3):
            flush.fill_(i & 0xFF)
            e = ev[i - 3] if i >= 3 else None
            if e:
                e[0].record(stream)
            M.dispatch(cfg, x, ids, mask, scales, out["expand_x"], out["dynamic_scales"], out["assist_info"],
                       out["ep_recv_count"], out["expand_scales"], None, ws)
            if e:
                e[1].record(stream)
            if wl.quant_mode == 0:
                M.combine(cfg, out["expand_x"], out["assist_info"], out["ep_recv_count"], ids, scales, mask, x,
                          x_out, None, ws)
            if e:
                e[2].record(stream)
        torch.cuda.synchronize()
        st = M.get_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {M.STATUS.get(st, st)} in {name}")
        acct = algorithmic_bytes(wl, inp)
        d_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
        r = {"dispatch_ms": d_ms, "dispatch_GBps": acct["dispatch"] / (d_ms * 1e-3) / 1e9,
             "dispatch_frac_of_8TBps": acct["dispatch"] / (d_ms * 1e-3) / 1e9 / HBM_NOMINAL_GBPS,
             "dispatch_bytes": acct["dispatch"]}
        if wl.quant_mode == 0:
            c_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
            r.update({"combine_ms": c_ms, "combine_GBps": acct["combine"] / (c_ms * 1e-3) / 1e9,
                      "combine_frac_of_8TBps": acct["combine"] / (c_ms * 1e-3) / 1e9 / HBM_NOMINAL_GBPS,
                      "combine_bytes": acct["combine"]})
        r["steps"] = n
        r["l2"] = "512 MB written before every step (untimed); median of per-call CUDA-event times"
        r["floor"] = measure_floor(torch, stream, flush, n, {"dispatch": acct["dispatch"]} if wl.quant_mode else
                                   {"dispatch": acct["dispatch"], "combine": acct["combine"]})
        del ws, out
        # sustained: back-to-back steps rotating over independent buffer sets,
        # enough of them that a set's data has left the L2 before it is reused
        step_bytes = acct["dispatch"] + (acct["combine"] if wl.quant_mode == 0 else 0)
        n_sets = max(2, int(np.ceil(4 * L2_BYTES / step_bytes)))
        sets = []
        for _ in range(n_sets):
            st_ = {"x": x.clone(), "ids": ids.clone(), "scales": scales.clone(),
                   "mask": None if mask is None else mask.clone(), "x_out": torch.empty_like(x),
                   "ws": M.alloc_workspace(cfg), "out": M.alloc_dispatch_outputs(cfg, tdt)}
            sets.append(st_)

        def run_set(b):
            o = b["out"]
            M.dispatch(cfg, b["x"], b["ids"], b["mask"], b["scales"], o["expand_x"], o["dynamic_scales"],
                       o["assist_info"], o["ep_recv_count"], o["expand_scales"], None, b["ws"])
            if wl.quant_mode == 0:
                M.combine(cfg, o["expand_x"], o["assist_info"], o["ep_recv_count"], b["ids"], b["scales"], b["mask"],
                          b["x"], b["x_out"], None, b["ws"])

        for i in range(2 * n_sets):
            run_set(sets[i % n_sets])
        torch.cuda.synchronize()
        ks = max(n_sets, args.small_steps * 4)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(ks):
            run_set(sets[i % n_sets])
        b.record(stream)
        torch.cuda.synchronize()
        for b_ in sets:
            st = M.get_device_status(b_["ws"])
            if st != 0:
                raise RuntimeError(f"device status {M.STATUS.get(st, st)} in {name}")
        sus_ms = a.elapsed_time(b) / ks
        r["sustained"] = {"ms_per_step": sus_ms, "GBps": step_bytes / (sus_ms * 1e-3) / 1e9,
                          "frac_of_8TBps": step_bytes / (sus_ms * 1e-3) / 1e9 / HBM_NOMINAL_GBPS,
                          "steps": ks, "buffer_sets": n_sets,
                          "what": "dispatch" + (" + combine" if wl.quant_mode == 0 else "")}
        # the same rotation captured once in a CUDA graph and replayed: no
        # host launch cost per step
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(n_sets):
                run_set(sets[i])
        graph.replay()
        torch.cuda.synchronize()
        reps = max(1, ks // n_sets)
        a.record(stream)
        for _ in range(reps):
            graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        for b_ in sets:
            st = M.get_device_status(b_["ws"])
            if st != 0:
                raise RuntimeError(f"device status {M.STATUS.get(st, st)} in {name} (graph)")
        g_ms = a.elapsed_time(b) / (reps * n_sets)
        r["sustained_graph"] = {"ms_per_step": g_ms, "GBps": step_bytes / (g_ms * 1e-3) / 1e9,
                                "frac_of_8TBps": step_bytes / (g_ms * 1e-3) / 1e9 / HBM_NOMINAL_GBPS,
                                "steps": reps * n_sets}
        del graph, sets
        res[name] = r
    del flush
    return res


def parse_quant_mode(tag: str):
    """'q3_fp8_e4m3_s0' -> (3, 'fp8_e4m3', 0); 'q1_int8_s1' -> (1, '', 1)."""
    q, rest = tag.split("_", 1)
    y, k = rest.rsplit("_s", 1)
    return int(q[1:]), "" if y == "int8" else y, int(k)


def measure_quant(args, M, torch, stream, base: WL.Workload):
    """moe_dispatch of the main workload with every quantised variant: the
    payload kernel alone (CUDA events the library records around it) and the
    whole call. Two output sets alternate, so consecutive steps do not share
    their written bytes in L2."""
    res = {}
    peaks = measured_peaks()
    for tag in [t for t in args.quant_modes.split(",") if t]:
        q, y, k = parse_quant_mode(tag)
        wl = base.with_(quant_mode=q, y_dtype=y, scales_kind=k)
        inp = WL.make_inputs(wl)
        bf = wl.x_dtype == WL.X_BF16
        tdt = torch.bfloat16 if bf else torch.float16

        def dev(a, as_bf=False):
            if a is None:
                return None
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if as_bf else np.ascontiguousarray(a))
            return (t.view(torch.bfloat16) if as_bf else t).cuda()

        x, ids, esc, mask = dev(inp["x"], bf), dev(inp["expert_ids"]), dev(inp["expert_scales"]), \
            dev(inp.get("active_mask"))
        qs = dev(inp.get("quant_scales"))
        cfg = M.config(wl.ep_world_size, wl.bs, wl.h, wl.topk, wl.moe_expert_num, tdt,
                       zero_expert_num=wl.zero_expert_num, copy_expert_num=wl.copy_expert_num, quant_mode=q,
                       mask_kind=wl.mask_kind, expand_dtype=y, scales_kind=k)
        ws = M.alloc_workspace(cfg)
        outs = [M.alloc_dispatch_outputs(cfg, tdt) for _ in range(2)]

        def call(c, i):
            o = outs[i & 1]
            M.dispatch(c, x, ids, mask, esc, o["expand_x"], o["dynamic_scales"], o["assist_info"],
                       o["ep_recv_count"], o["expand_scales"], None, ws, scales=qs)

        for i in range(3):
            call(cfg, i)
        torch.cuda.synchronize()
        n = max(3, args.quant_steps)
        evs = [M.ProfEvents() for _ in range(n)]
        cfgs = [e.attach(cfg) for e in evs]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(n):
            call(cfg, i)
        b.record(stream)
        for i, c in enumerate(cfgs):
            call(c, i)
        torch.cuda.synchronize()
        st = M.get_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {M.STATUS.get(st, st)} in quant variant {tag}")
        acct = algorithmic_bytes(wl, inp)
        call_ms = a.elapsed_time(b) / n
        sc_ms = statistics.mean(e.elapsed_ms() for e in evs)
        res[tag] = {"dispatch_ms": call_ms, "dispatch_GBps": acct["dispatch"] / (call_ms * 1e-3) / 1e9,
                    "scatter_ms": sc_ms, "scatter_GBps": acct["scatter"] / (sc_ms * 1e-3) / 1e9,
                    "scatter_frac_of_measured_hbm": acct["scatter"] / (sc_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                    "scatter_bytes": acct["scatter"], "row_out_bytes": row_out_bytes(wl), "steps": n}
        del ws, outs
    return {"workload": base.name, "variants": res,
            "note": "q2_int8_s0 is the per-token int8 kernel of the plain dispatch; the others run the quantising "
                    "scatter (a variant per pick when s3 = per-expert scales)"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from combine_route_scan_gb300 import build as B
    if rank == 0:
        B.build()
    if world > 1:
        dist.barrier()
    from combine_route_scan_gb300 import moe as M

    wl = WL.WORKLOADS[args.workload]
    if args.only_quant:
        print(json.dumps(measure_quant(args, M, torch, torch.cuda.current_stream(), wl)))
        return 0
    if args.only_small:
        print(json.dumps(measure_small(args, M, torch, torch.cuda.current_stream())))
        return 0
    inp = WL.make_inputs(wl, seed=rank_seed(wl, rank))
    acct = algorithmic_bytes(wl, inp)
    step_bytes = acct["dispatch"] + acct["combine"]
    tdt = {WL.X_INT32: torch.int32, WL.X_FP16: torch.float16, WL.X_BF16: torch.bfloat16}[wl.x_dtype]

    def dev(a, bf=False):
        if a is None:
            return None
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf else np.ascontiguousarray(a))
        return (t.view(torch.bfloat16) if bf else t).cuda()

    bf = wl.x_dtype == WL.X_BF16
    x, ids = dev(inp["x"], bf), dev(inp["expert_ids"])
    mask, scales = dev(inp.get("active_mask")), dev(inp["expert_scales"])
    cfg = M.config(wl.ep_world_size, wl.bs, wl.h, wl.topk, wl.moe_expert_num, tdt,
                   zero_expert_num=wl.zero_expert_num, copy_expert_num=wl.copy_expert_num,
                   quant_mode=wl.quant_mode, mask_kind=wl.mask_kind, plane_policy=args.plane_policy)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_dispatch_outputs(cfg, tdt)
    x_out = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    # timed regions A and B rotate over independent buffer sets when one step
    # would stay in L2 (set 0 is the one the other sections use)
    n_sets = rotation_sets(step_bytes)
    sets = [{"x": x, "ids": ids, "mask": mask, "scales": scales, "ws": ws, "out": out, "x_out": x_out}]
    for _ in range(n_sets - 1):
        sets.append({"x": x.clone(), "ids": ids.clone(), "mask": None if mask is None else mask.clone(),
                     "scales": scales.clone(), "ws": M.alloc_workspace(cfg), "out": M.alloc_dispatch_outputs(cfg, tdt),
                     "x_out": torch.empty_like(x)})

    def step(cfg_d, cfg_c, b=None):
        b = sets[0] if b is None else b
        o = b["out"]
        M.dispatch(cfg_d, b["x"], b["ids"], b["mask"], b["scales"], o["expand_x"], o["dynamic_scales"],
                   o["assist_info"], o["ep_recv_count"], o["expand_scales"], None, b["ws"])
        if wl.quant_mode == 0:
            M.combine(cfg_c, o["expand_x"], o["assist_info"], o["ep_recv_count"], b["ids"], b["scales"], b["mask"],
                      b["x"], b["x_out"], None, b["ws"])

    for i in range(max(3, args.warmup, 2 * n_sets)):
        step(cfg, cfg, sets[i % n_sets])
    torch.cuda.synchronize()
    st = M.get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {M.STATUS.get(st, st)} during warmup")

    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    # Timed region A (the headline): K steps exactly as a user runs them, the
    # kernels chained by programmatic dependent launch.
    sampler = ClockSampler(gpu_id_for_smi(local)) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    h0 = time.time()
    n_launch0 = M.launch_count()
    t_start.record(stream)
    for k in range(K):
        step(cfg, cfg, sets[k % n_sets])
    t_end.record(stream)
    n_launches = M.launch_count() - n_launch0
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    h1 = time.time()
    total_ms = t_start.elapsed_time(t_end)
    # keep the same load going until the clock record covers at least 1.5 s
    h_ext = h1
    if sampler and h1 - h0 < 1.5:
        while time.time() - h0 < 1.5:
            for i in range(50):
                step(cfg, cfg, sets[i % n_sets])
            torch.cuda.synchronize()
        h_ext = time.time()
    total_ms = max_over_ranks(total_ms, world)

    # The same steps replayed from a CUDA graph of one step per buffer set (no
    # host launch cost per step); reported beside region A.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for b in sets:
            step(cfg, cfg, b)
    graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, K // n_sets)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    g0.record(stream)
    for k in range(reps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(g0.elapsed_time(g1), world) / (reps * n_sets)
    del graph

    # Timed region B (kernel attribution): the same K steps with CUDA events the
    # library records on the launching stream around the scatter and the
    # combine reduce, and around each call. An event between two kernels stops
    # the next one from starting early, so region B's step is a little slower.
    ev_scatter = [M.ProfEvents() for _ in range(K)]
    ev_reduce = [M.ProfEvents() for _ in range(K)]
    cfg_s = [e.attach(cfg) for e in ev_scatter]
    cfg_r = [e.attach(cfg) for e in ev_reduce]
    b_start, b_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    b_start.record(stream)
    for k in range(K):
        step(cfg_s[k], cfg_r[k], sets[k % n_sets])
    b_end.record(stream)
    torch.cuda.synchronize()
    instrumented_ms = max_over_ranks(b_start.elapsed_time(b_end), world) / K
    for b in sets:
        st = M.get_device_status(b["ws"])
        if st != 0:
            raise RuntimeError(f"device status {M.STATUS.get(st, st)} in the timed region")

    scatter_ms = statistics.mean(e.elapsed_ms() for e in ev_scatter)
    reduce_ms = statistics.mean(e.elapsed_ms() for e in ev_reduce) if wl.quant_mode == 0 else 0.0
    step_ms = total_ms / K
    kernels = {"scatter": (scatter_ms, acct["scatter"]), "combine_reduce": (reduce_ms, acct["reduce"])}
    dom = max(kernels, key=lambda k: kernels[k][0])
    dom_ms, dom_bytes = kernels[dom]
    peaks = measured_peaks()
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = committed_traffic(dom, wl.name)

    # the page's split of the two-phase combine: full_op (put + flags + wait +
    # reduce) and comm_only (put + flags), timed on their own workspace
    two_phase = None
    if wl.quant_mode == 0 and wl.h * wl.es % 16 == 0:
        cfg_tp = M.MoeConfig.from_buffer_copy(cfg)
        cfg_tp.combine_mode = M.COMBINE_TWO_PHASE
        cfg_put = M.MoeConfig.from_buffer_copy(cfg)
        cfg_put.combine_mode = M.COMBINE_PUT_ONLY
        ws_tp = M.alloc_workspace(cfg_tp)
        x_tp = torch.empty_like(x)

        def tp_call(c):
            M.combine(c, out["expand_x"], out["assist_info"], out["ep_recv_count"], ids, scales, mask, x, x_tp,
                      None, ws_tp)

        Kt = max(1, min(K, 200))
        res = {}
        # the README's comparison: the classic single plane (every segment by
        # SM stores) against the two planes
        cfg_tp_c = M.MoeConfig.from_buffer_copy(cfg_tp)
        cfg_tp_c.plane_policy = M.PLANE_STORES_ONLY
        cfg_put_c = M.MoeConfig.from_buffer_copy(cfg_put)
        cfg_put_c.plane_policy = M.PLANE_STORES_ONLY
        for name, c in (("full_op", cfg_tp), ("comm_only", cfg_put), ("classic_full_op", cfg_tp_c),
                        ("classic_comm_only", cfg_put_c)):
            for _ in range(3):
                tp_call(c)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(Kt):
                tp_call(c)
            b.record(stream)
            torch.cuda.synchronize()
            res[name] = a.elapsed_time(b) / Kt
        st = M.get_device_status(ws_tp)
        if st != 0:
            raise RuntimeError(f"device status {M.STATUS.get(st, st)} in the two-phase combine")
        put_bytes = 2 * acct["P"] * wl.h * wl.es
        two_phase = {"full_op_ms": res["full_op"], "comm_only_ms": res["comm_only"],
                     "full_op_GBps": acct["combine"] / (res["full_op"] * 1e-3) / 1e9,
                     "comm_only_GBps": put_bytes / (res["comm_only"] * 1e-3) / 1e9,
                     "classic_full_op_ms": res["classic_full_op"], "classic_comm_only_ms": res["classic_comm_only"],
                     "steps": Kt}
        del ws_tp

    # the optional dispatch outputs: per-segment ready flags and per-rank
    # communication time, each timed on its own against the plain call
    options = None
    if world == 1:
        L_ = wl.moe_expert_num // wl.ep_world_size
        flags = torch.zeros((wl.ep_world_size, L_ * wl.ep_world_size), dtype=torch.int32, device="cuda")
        perf = torch.zeros(wl.ep_world_size, dtype=torch.int64, device="cuda")
        variants = {"plain": lambda i: cfg,
                    "seg_ready": lambda i: M.with_seg_ready(cfg, flags, 1000 + i),
                    "performance_info": lambda i: M.with_performance_info(cfg, perf)}
        Ko = max(1, min(K, 200))
        options = {}
        for name, mk in variants.items():
            cfgs = [mk(i) for i in range(Ko + 3)]
            for i in range(3):
                M.dispatch(cfgs[i], x, ids, mask, scales, out["expand_x"], out["dynamic_scales"], out["assist_info"],
                           out["ep_recv_count"], out["expand_scales"], None, ws)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(Ko):
                M.dispatch(cfgs[3 + i], x, ids, mask, scales, out["expand_x"], out["dynamic_scales"],
                           out["assist_info"], out["ep_recv_count"], out["expand_scales"], None, ws)
            b.record(stream)
            torch.cuda.synchronize()
            options[name + "_dispatch_ms"] = a.elapsed_time(b) / Ko
        st = M.get_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {M.STATUS.get(st, st)} with the dispatch options")
        options["per_rank_comm_us_mean"] = float(perf.double().mean().item()) / (Ko + 3) / 1e3
        options["steps"] = Ko
        # the page's split for dispatch: full_op = the whole call (routing +
        # payload), comm_only = the payload kernel (puts and, when on, flags)
        options["full_op_ms"] = options["plain_dispatch_ms"]
        options["comm_only_ms"] = scatter_ms

    ffn = None if args.no_ffn or world > 1 else measure_ffn(args, M, torch, stream)
    small = None if world > 1 or not args.small_workloads else measure_small(args, M, torch, stream)
    quant = None if world > 1 or not args.quant_modes else measure_quant(args, M, torch, stream, wl)

    # End to end through the C ABI with host buffers: every step copies its
    # inputs from pinned host memory (H2D stream), runs dispatch + combine
    # (compute stream) and reads x_out back into pinned host memory (D2H
    # stream). Device inputs and outputs are double-buffered and events order
    # the three streams, so step i's compute overlaps step i+1's upload and
    # step i-1's download, as a serving loop would run it.
    host = {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v)).pin_memory())
            for k, v in (("x", inp["x"].view(np.int16) if bf else inp["x"]), ("ids", inp["expert_ids"]),
                         ("mask", inp.get("active_mask")), ("scales", inp["expert_scales"]))}
    host_out = [torch.empty(x_out.shape, dtype=x_out.dtype, pin_memory=True) for _ in range(2)]
    bufs = [{"x": torch.empty_like(x), "ids": torch.empty_like(ids), "scales": torch.empty_like(scales),
             "mask": None if mask is None else torch.empty_like(mask), "out": torch.empty_like(x_out)}
            for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = host_out[0].numel() * host_out[0].element_size()
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_h2d = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        for i in range(n):
            b = bufs[i & 1]
            with torch.cuda.stream(s_h2d):
                if i >= 2:
                    s_h2d.wait_event(ev_comp[i & 1])  # step i-2 is done reading these inputs
                b["x"].view(torch.int16 if bf else b["x"].dtype).copy_(host["x"], non_blocking=True)
                b["ids"].copy_(host["ids"], non_blocking=True)
                if mask is not None:
                    b["mask"].copy_(host["mask"], non_blocking=True)
                b["scales"].copy_(host["scales"], non_blocking=True)
                ev_h2d[i & 1].record(s_h2d)
            stream.wait_event(ev_h2d[i & 1])
            if i >= 2:
                stream.wait_event(ev_d2h[i & 1])  # step i-2's x_out has been read back
            step(cfg, cfg, {"x": b["x"], "ids": b["ids"], "mask": b["mask"], "scales": b["scales"], "ws": ws,
                            "out": out, "x_out": b["out"]})
            ev_comp[i & 1].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_comp[i & 1])
                host_out[i & 1].copy_(b["out"], non_blocking=True)
                ev_d2h[i & 1].record(s_d2h)
        stream.wait_event(ev_d2h[(n - 1) & 1])

    e2e_run(4)
    torch.cuda.synchronize()
    Ke = max(2, min(args.e2e_steps, K))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    e2e_run(Ke)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / Ke
    e2e_ms = max_over_ranks(e2e_ms, world)
    # the last step's result really came back
    if wl.quant_mode == 0 and not torch.equal(host_out[(Ke - 1) & 1].cuda(), x_out):
        raise RuntimeError("end-to-end result differs from the device-resident run")
    st = M.get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {M.STATUS.get(st, st)} in the e2e region")

    clocks = None
    if sampler:
        sampler.stop()
        clocks = sampler.summary(h0, h_ext)
        clocks["window_s"] = round(h_ext - h0, 3)
        clocks["timed_region_s"] = round(h1 - h0, 3)

    cpu = None
    par = None
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import build as OB
        OB.build()
        times = time_oracle(wl, inp, target_s=10.0, max_steps=10)
        cpu = {"value": step_bytes / statistics.mean(times) / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{len(times)} full steps (dispatch+combine over all {wl.ep_world_size * wl.bs} tokens), "
                         f"single-threaded C, mean {statistics.mean(times) * 1e3:.0f} ms/step"}
        try:
            par = time_oracle_all_cores(wl, inp, target_s=5.0)
        except Exception as e:  # the GPU figures above stand without it
            cpu["all_cores"] = {"error": f"{type(e).__name__}: {e}"}
    if par is not None:
        lo, hi = par["tokens_per_slice"]
        cpu["all_cores"] = {
            "value": par["bytes"] / par["seconds"] / 1e9, "unit": "GB/s", "cores": par["threads"],
            "kind": "oracle",
            "sample": f"{par['slices_done']} dispatch+combine calls of the unchanged single-threaded C oracle "
                      f"on {par['threads']} threads at once, each on its own slice of {lo}"
                      + (f"-{hi}" if hi != lo else "") + f" of every rank's {wl.bs} tokens, "
                      f"{par['seconds']:.1f} s"}

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0
    ws_bytes = inp["x"].nbytes * 2 + acct["P"] * wl.h * wl.es * 2
    value = whole_job_gbps(step_bytes, K, total_ms, world)
    tokens = world * wl.ep_world_size * wl.bs
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.x_dtype == WL.X_BF16 else ("fp16" if wl.x_dtype == WL.X_FP16 else "int32"),
        "data": "synthetic",
        "config": bench_config(wl, args, step_bytes),
        "tokens_per_s": tokens * K / (total_ms * 1e-3),
        "frac_of_8TBps": value / world / HBM_NOMINAL_GBPS,
        "dispatch_bytes": acct["dispatch"], "combine_bytes": acct["combine"], "routed_picks": acct["P"],
        "scatter_ms": scatter_ms, "combine_reduce_ms": reduce_ms,
        "instrumented_ms_per_step": instrumented_ms,
        "graph_ms_per_step": graph_ms,
        "scatter_GBps": acct["scatter"] / (scatter_ms * 1e-3) / 1e9,
        "combine_reduce_GBps": acct["reduce"] / (reduce_ms * 1e-3) / 1e9 if reduce_ms else None,
        "scatter_frac_of_measured_hbm": acct["scatter"] / (scatter_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "combine_reduce_frac_of_measured_hbm": (acct["reduce"] / (reduce_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]
                                                if reduce_ms else None),
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "algorithmic_bytes": dom_bytes, "peak_source": peaks["source"] + " copy bandwidth"},
        "cpu_baseline": cpu,
        "e2e": {"value": step_bytes / (e2e_ms * 1e-3) / 1e9 * world, "unit": "GB/s", "ms_per_step": e2e_ms,
                "streams": "H2D, compute and D2H on three streams, double-buffered",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "two_phase_combine": two_phase,
        "dispatch_options": options,
        "ffn_variant": ffn,
        "small_workloads": small,
        "quant_dispatch": quant,
        "gpu_launches": n_launches,
        "clocks": clocks,
    }
    print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
