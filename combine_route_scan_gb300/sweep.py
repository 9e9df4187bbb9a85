"""Multi-shape performance sweep of combine and dispatch.

Follows the sweep of the combine_doubleplane README (section 性能测试): a grid
of rank counts, batch sizes, hidden sizes, top-k values and experts per rank,
with per-rank CSV files and a summary CSV. For every shape it times, as the
mean of ``--loops`` calls after ``--warmup`` untimed ones (CUDA events on the
launching stream, no L2 flush, as in the README's loop):

  full_op    the two-phase combine: put every expert row into its source's
             window (bulk or store plane by the page's rule), the per-pick
             status protocol, the weighted reduction;
  comm_only  the put phase with its completion / status protocol alone;
  gather     the one-pass gather combine (this library's default);
  dispatch   moe_dispatch, plus each rank's communication time from the
             performance-info output.

The expert is the identity (its outputs are the dispatched rows), as in the
README's check. Each shape also checks that the two-phase combine and the
gather combine give the same bytes.

Files written to ``--out-dir``:
  perf_rank<r>.csv   one row per shape for rank r: rows it received, the rows
                     and bytes it put on the bulk plane in the two-phase
                     combine, the shape's timings and rank r's dispatch time;
  perf_summary.csv   one row per shape: timings, moved bytes, GB/s, and the
                     min / mean / max of the per-rank dispatch times.
``--prof-pe all`` writes every rank's file, ``--prof-pe r`` only rank r's.

Inputs are seeded and synthetic: x uniform in [-1000, 1000] (int32) or N(0, 1)
(fp16 / bf16); K distinct expert ids per token, uniform; weights uniform in
[1, 4] (int32) or a softmax over K of N(0, 1) logits (fp32).

    python -m combine_route_scan_gb300.sweep --pes-list 2,4,8 --bs-list 8,16,32 \\
        --h-list 64,256,1024 --topk-list 2 --expert-per-pe-list 2,8 --type int32 \\
        --prof-pe all --warmup 5 --loops 50 --out-dir sweep_out

``--plane-policy stores`` runs the classic single plane (every segment by SM
stores), the README's comparison point for the two planes.
"""
from __future__ import annotations

import argparse
import csv
import itertools
import os
import statistics
from typing import Dict, List

import torch

from . import build as _build
from . import moe as M

TYPES = {"int32": torch.int32, "int32_t": torch.int32, "fp16": torch.float16, "float16_t": torch.float16,
         "bf16": torch.bfloat16, "bfloat16_t": torch.bfloat16}

PLANES = {"rule": M.PLANE_RULE, "stores": M.PLANE_STORES_ONLY, "bulk": M.PLANE_BULK_ALL}

RANK_FIELDS = ["pes", "bs", "h", "topk", "expert_per_pe", "type", "planes", "rank", "recv_rows", "bulk_put_rows",
               "bulk_put_bytes", "full_op_us", "comm_only_us", "gather_us", "dispatch_us", "dispatch_comm_us"]
SUMMARY_FIELDS = ["pes", "bs", "h", "topk", "expert_per_pe", "type", "planes", "routed_rows", "full_op_us", "comm_only_us",
                  "gather_us", "dispatch_us", "combine_bytes", "gather_GBps", "full_op_GBps", "comm_only_GBps",
                  "dispatch_comm_us_min", "dispatch_comm_us_mean", "dispatch_comm_us_max",
                  "two_phase_matches_gather"]


def int_list(s: str) -> List[int]:
    return [int(v) for v in s.split(",") if v.strip()]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--pes-list", type=int_list, default=[2, 4, 8])
    ap.add_argument("--bs-list", type=int_list, default=[8, 16, 32])
    ap.add_argument("--h-list", type=int_list, default=[64, 256, 1024])
    ap.add_argument("--topk-list", type=int_list, default=[2])
    ap.add_argument("--expert-per-pe-list", type=int_list, default=[2, 8])
    ap.add_argument("--type", default="int32", choices=sorted(TYPES))
    ap.add_argument("--prof-pe", default="all", help="'all' or one rank id")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--loops", type=int, default=50)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--plane-policy", default="rule", choices=sorted(PLANES),
                    help="rule: the README's two planes; stores: the classic single plane; bulk: every remote "
                         "segment by bulk copies")
    ap.add_argument("--out-dir", default="sweep_out")
    return ap.parse_args(argv)


def shapes(args):
    """The grid, skipping shapes the library rejects (top-k above the expert count)."""
    for W, bs, h, K, L in itertools.product(args.pes_list, args.bs_list, args.h_list, args.topk_list,
                                            args.expert_per_pe_list):
        if K <= W * L:
            yield W, bs, h, K, L


def make_inputs(W: int, bs: int, h: int, K: int, E: int, dtype: torch.dtype, seed: int) -> Dict[str, torch.Tensor]:
    g = torch.Generator().manual_seed(seed)
    n = W * bs
    ids = torch.rand(n, E, generator=g).argsort(dim=1)[:, :K].to(torch.int32).reshape(W, bs, K)
    if dtype == torch.int32:
        x = torch.randint(-1000, 1001, (W, bs, h), generator=g, dtype=torch.int32)
        w = torch.randint(1, 5, (W, bs, K), generator=g, dtype=torch.int32)
    else:
        x = torch.randn(W, bs, h, generator=g).to(dtype)
        w = torch.softmax(torch.randn(W, bs, K, generator=g), dim=-1).to(torch.float32)
    return {"x": x.cuda(), "ids": ids.cuda(), "w": w.cuda()}


def mean_event_ms(fn, warmup: int, loops: int) -> float:
    for _ in range(warmup):
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(loops)]
    stream = torch.cuda.current_stream()
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def run_shape(W: int, bs: int, h: int, K: int, L: int, dtype: torch.dtype, args) -> Dict:
    E = W * L
    inp = make_inputs(W, bs, h, K, E, dtype, args.seed + 7919 * W + 131 * bs + h + 17 * K + L)
    cfg_d = M.config(W, bs, h, K, E, dtype, plane_policy=PLANES[args.plane_policy])
    ws = M.alloc_workspace(M.config(W, bs, h, K, E, dtype, combine_mode=M.COMBINE_TWO_PHASE))
    out = M.alloc_dispatch_outputs(cfg_d, dtype)
    perf = torch.zeros(W, dtype=torch.int64, device="cuda")
    cfg_p = M.with_performance_info(cfg_d, perf)

    def dispatch(c=cfg_d):
        M.dispatch(c, inp["x"], inp["ids"], None, inp["w"], out["expand_x"], out["dynamic_scales"],
                   out["assist_info"], out["ep_recv_count"], out["expand_scales"], None, ws)

    dispatch_ms = mean_event_ms(dispatch, args.warmup, args.loops)
    perf.zero_()
    for _ in range(args.loops):
        dispatch(cfg_p)
    torch.cuda.synchronize()
    comm_us = (perf.double() / args.loops / 1e3).cpu().tolist()

    x_gather = torch.empty_like(inp["x"])
    x_tp = torch.empty_like(inp["x"])
    seg_plane = torch.zeros((W, L * W), dtype=torch.uint8, device="cuda")

    def combine(mode, x_out, sp=None):
        c = M.config(W, bs, h, K, E, dtype, combine_mode=mode, plane_policy=PLANES[args.plane_policy])
        return lambda: M.combine(c, out["expand_x"], out["assist_info"], out["ep_recv_count"], inp["ids"],
                                 inp["w"], None, inp["x"], x_out, sp, ws)

    gather_ms = mean_event_ms(combine(M.COMBINE_GATHER, x_gather), args.warmup, args.loops)
    full_ms = mean_event_ms(combine(M.COMBINE_TWO_PHASE, x_tp, seg_plane), args.warmup, args.loops)
    comm_ms = mean_event_ms(combine(M.COMBINE_PUT_ONLY, x_tp), args.warmup, args.loops)
    x_tp2 = torch.empty_like(inp["x"])
    combine(M.COMBINE_TWO_PHASE, x_tp2)()
    st = M.get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {M.STATUS.get(st, st)} at W={W} bs={bs} h={h} K={K} L={L}")

    ep = out["ep_recv_count"].cpu()
    rows = torch.diff(ep, dim=1, prepend=torch.zeros(W, 1, dtype=ep.dtype))  # rows per (le, s) segment
    bulk_rows = (rows * seg_plane.cpu().to(rows.dtype)).sum(dim=1)
    row_bytes = h * torch.tensor([], dtype=dtype).element_size()
    routed = int(ep[:, -1].sum())
    # identity-expert combine: every routed row read once, weights / ids read,
    # tokens written once
    combine_bytes = routed * row_bytes + W * bs * K * 8 + W * bs * row_bytes
    return {
        "routed_rows": routed, "recv_rows": ep[:, -1].tolist(), "bulk_rows": bulk_rows.tolist(),
        "row_bytes": row_bytes, "dispatch_us": dispatch_ms * 1e3, "gather_us": gather_ms * 1e3,
        "full_op_us": full_ms * 1e3, "comm_only_us": comm_ms * 1e3, "dispatch_comm_us": comm_us,
        "combine_bytes": combine_bytes, "two_phase_matches_gather": bool(torch.equal(x_tp2, x_gather)),
    }


def main(argv=None) -> int:
    args = parse_args(argv)
    _build.build()
    dtype = TYPES[args.type]
    os.makedirs(args.out_dir, exist_ok=True)
    ranks_wanted = None if args.prof_pe == "all" else {int(args.prof_pe)}
    rank_rows: Dict[int, List[Dict]] = {}
    summary: List[Dict] = []
    for W, bs, h, K, L in shapes(args):
        r = run_shape(W, bs, h, K, L, dtype, args)
        key = {"pes": W, "bs": bs, "h": h, "topk": K, "expert_per_pe": L, "type": args.type,
               "planes": args.plane_policy}
        for d in range(W):
            if ranks_wanted is not None and d not in ranks_wanted:
                continue
            rank_rows.setdefault(d, []).append({
                **key, "rank": d, "recv_rows": r["recv_rows"][d], "bulk_put_rows": r["bulk_rows"][d],
                "bulk_put_bytes": r["bulk_rows"][d] * r["row_bytes"], "full_op_us": r["full_op_us"],
                "comm_only_us": r["comm_only_us"], "gather_us": r["gather_us"], "dispatch_us": r["dispatch_us"],
                "dispatch_comm_us": r["dispatch_comm_us"][d]})
        cb = r["combine_bytes"]
        summary.append({
            **key, "routed_rows": r["routed_rows"], "full_op_us": r["full_op_us"], "comm_only_us": r["comm_only_us"],
            "gather_us": r["gather_us"], "dispatch_us": r["dispatch_us"], "combine_bytes": cb,
            "gather_GBps": cb / (r["gather_us"] * 1e3), "full_op_GBps": cb / (r["full_op_us"] * 1e3),
            "comm_only_GBps": 2 * r["routed_rows"] * r["row_bytes"] / (r["comm_only_us"] * 1e3),
            "dispatch_comm_us_min": min(r["dispatch_comm_us"]),
            "dispatch_comm_us_mean": statistics.mean(r["dispatch_comm_us"]),
            "dispatch_comm_us_max": max(r["dispatch_comm_us"]),
            "two_phase_matches_gather": r["two_phase_matches_gather"]})
        print(f"pes={W} bs={bs} h={h} topk={K} L={L}: full_op {r['full_op_us']:.1f} us, comm_only "
              f"{r['comm_only_us']:.1f} us, gather {r['gather_us']:.1f} us, dispatch {r['dispatch_us']:.1f} us",
              flush=True)
    for d, rows in sorted(rank_rows.items()):
        write_csv(os.path.join(args.out_dir, f"perf_rank{d}.csv"), RANK_FIELDS, rows)
    write_csv(os.path.join(args.out_dir, "perf_summary.csv"), SUMMARY_FIELDS, summary)
    bad = [s for s in summary if not s["two_phase_matches_gather"]]
    if bad:
        print(f"{len(bad)} shape(s) where the two-phase combine differs from the gather combine")
        return 1
    return 0


def write_csv(path: str, fields: List[str], rows: List[Dict]) -> None:
    with open(path, "w", newline="") as f:
        w = csv.DictWriter(f, fieldnames=fields)
        w.writeheader()
        for r in rows:
            w.writerow({k: (f"{v:.3f}" if isinstance(v, float) else v) for k, v in r.items()})


if __name__ == "__main__":
    raise SystemExit(main())
