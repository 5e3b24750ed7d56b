"""Per-CTA timeline of the single-CTA tensor-core kernel (gemm_trace_set).

    python -m dense_tiled_gemm_02_gb300.timeline --workload skinny8192x128x4096_bf16 \
        [--plan "bn=128,splits=2"] [--calls 20]

Runs the workload's call `--calls` times back to back on rotating input sets
(as the benchmark does), with the timeline hook on, and prints for the last
call the spread over CTAs of each event's global-timer stamp, relative to
the earliest kernel entry, and of the intervals between events:
load latency (2 -> 3), streaming of the K loop (3 -> 4), hand-over to the
epilogue (4 -> 5), epilogue (5 -> 6) and the whole CTA (0 -> 7; 7 is stamped by the first epilogue thread, 0 by thread 0).
"""
from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EVENTS = ("entry", "past_pdl_wait", "first_loads", "first_stage_landed", "last_acc_committed",
          "last_acc_seen", "last_tile_stored", "past_final_barrier", "splits_landed",
          "split_sent", "epilogue_all_in", "epilogue_pos0", "epilogue_pos1", "epilogue_pos2",
          "epilogue_pos3")
INTERVALS = (("load_latency", 2, 3), ("k_loop", 3, 4), ("handover", 4, 5), ("epilogue", 5, 6),
             ("cta", 0, 7))


def stats(v):
    v = sorted(v)
    n = len(v)
    return {"min": round(v[0], 3), "median": round(v[n // 2], 3), "max": round(v[-1], 3)}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", required=True)
    ap.add_argument("--plan", default="")
    ap.add_argument("--calls", type=int, default=20)
    ap.add_argument("--raw", action="store_true", help="also print every CTA's stamps")
    a = ap.parse_args(argv)
    if a.plan:
        os.environ["GEMM_FORCE_PLAN"] = a.plan
    sys.path.insert(0, ROOT)
    import re

    import torch

    import dense_tiled_gemm_02_gb300 as pkg
    from workloads import TORCH_DTYPE, WORKLOADS, make_inputs, storage_shape

    def logical(t, layout):
        return t if layout == 0 else t.t()

    w = WORKLOADS[a.workload]
    dev = torch.device("cuda")
    inp = make_inputs(w)
    sets = []
    for _ in range(4):
        A = logical(inp["A"].to(dev), w.layout_a)
        B = logical(inp["B"].to(dev), w.layout_b)
        C = None if inp["C"] is None else logical(inp["C"].to(dev), w.layout_c)
        D = logical(torch.empty(storage_shape(w.M, w.N, w.layout_d), dtype=TORCH_DTYPE[w.d_type],
                                device=dev), w.layout_d)
        sets.append((A, B, C, D))
    g = pkg.Gemm.like(*sets[0])
    plan = g.plan()
    grid = int(re.search(r"grid=(\d+)", plan).group(1))
    buf = torch.zeros(grid * pkg.GEMM_TRACE_EVENTS, dtype=torch.int64, device=dev)
    for i in range(a.calls):
        g.run(*sets[i % 4])
    torch.cuda.synchronize()
    rc = pkg.gemm_trace_set(g.handle, buf.data_ptr())
    assert rc == pkg.GEMM_OK, rc
    for i in range(a.calls):
        g.run(*sets[i % 4])
    torch.cuda.synchronize()
    pkg.gemm_trace_set(g.handle, None)
    assert g.status() == pkg.GEMM_OK
    t = buf.view(grid, pkg.GEMM_TRACE_EVENTS).cpu().double()
    t0 = t[:, 0].min()
    rel = ((t - t0) / 1e3).tolist()  # us
    units = []  # pair kernel: MMA busy spans per unit of each cluster (even CTAs)
    if "pair=1" in plan:
        for c in range(0, grid, 2):
            row = rel[c]
            spans = [(row[10 + 2 * i], row[11 + 2 * i]) for i in range(11)
                     if t[c, 10 + 2 * i] > 0 and t[c, 11 + 2 * i] > 0]
            units.append(spans)
    out = {"workload": w.name, "plan": plan, "ctas": grid,
           "span_us": round((t[:, 7].max() - t0).item() / 1e3, 3),
           "events_us": {name: stats([r[e] for c, r in enumerate(rel) if t[c, e] > 0])
                         for e, name in enumerate(EVENTS[:10] if "pair=1" in plan else EVENTS)
                         if (t[:, e] > 0).any()},
           "intervals_us": {name: stats([r[j] - r[i] for r in rel])
                            for name, i, j in INTERVALS}}
    if units:
        first = [u[0][0] for u in units if u]
        last = [u[-1][1] for u in units if u]
        gaps = [u[i + 1][0] - u[i][1] for u in units for i in range(len(u) - 1)]
        busy = [sum(b - a for a, b in u) for u in units if u]
        out["mma_units"] = {"per_cluster": stats([len(u) for u in units]),
                            "first_start": stats(first), "last_commit": stats(last),
                            "gap_between_units": stats(gaps) if gaps else None,
                            "issue_span": stats([b - a for a, b in zip(first, last)]),
                            "unit_time": stats([b - a for u in units for a, b in u])}
    if a.raw:
        out["ctas_us"] = [[round(x, 3) for x in r] for r in rel]
    g.close()
    print(json.dumps(out))
    return 0


if __name__ == "__main__":
    sys.exit(main())
