"""Measured plan sweep for the selection table (csrc/plan_table.h).

    python -m dense_tiled_gemm_02_gb300.tune --workload sq4096_bf16 \
        --candidates "default;bn=256;bn=128;bn=256,group=4;cublas" [--repeats 7] [--iters 20]

Every candidate plan (a GEMM_FORCE_PLAN string; "default" for the plan the
library picks, "cublas" for PyTorch's GEMM as context) gets its own handle; the
candidates are timed interleaved, repeat after repeat, so that clock and
power drift hit them alike, and each result is the median over repeats with
its spread (max - min) / median.  A difference smaller than the spreads is
not a result (the "Tuning Triton" skill page, section 2: compare a win to
the noise floor).  Each workload runs in a child process, so a candidate
that fails cannot take the sweep down with it (same page: probe abort-prone
configurations in subprocesses and rate them by exit code).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
L2_BYTES = 129 * 10 ** 6


class LibraryReference:
    """The candidate "cublas": PyTorch's own GEMM on the same operands, timed
    beside the plans as context (torch.addmm / torch.mm for 16-bit types,
    torch._int_mm plus C for int8, torch._scaled_mm with unit scales plus C
    for 8-bit floats).  Not part of the library."""

    def __init__(self, w):
        self.w = w

    def run(self, A, B, C, D):
        import torch
        if A.dtype == torch.int8:
            r = torch._int_mm(A, B)
            torch.add(r, C, out=D) if C is not None else D.copy_(r)
        elif A.element_size() == 1:
            one = getattr(self, "_one", None)
            if one is None:
                one = self._one = torch.ones((), dtype=torch.float32, device=A.device)
            r = torch._scaled_mm(A, B, scale_a=one, scale_b=one, out_dtype=D.dtype)
            torch.add(r, C, out=D) if C is not None else D.copy_(r)
        elif D.dtype == A.dtype:
            if C is not None and C.dtype == D.dtype:
                torch.addmm(C, A, B, out=D)
            else:
                torch.mm(A, B, out=D)
        else:
            D.copy_(torch.mm(A, B))
            if C is not None:
                D.add_(C)

    def plan(self) -> str:
        return "torch (cuBLAS) reference"

    def close(self) -> None:
        pass


def child(args) -> int:
    sys.path.insert(0, ROOT)
    import torch

    import dense_tiled_gemm_02_gb300 as pkg
    from workloads import TORCH_DTYPE, WORKLOADS, make_inputs, storage_shape
    w = WORKLOADS[args.workload]
    dev = torch.device("cuda")
    inp = make_inputs(w)
    lg = lambda t, l: t if l == 0 else t.t()
    set_bytes = sum(t.numel() * t.element_size() for t in inp.values() if t is not None)
    set_bytes += w.M * w.N * TORCH_DTYPE[w.d_type].itemsize
    nsets = max(2, -(-2 * L2_BYTES // set_bytes))
    sets = []
    for _ in range(nsets):
        A = lg(inp["A"].to(dev), w.layout_a)
        B = lg(inp["B"].to(dev), w.layout_b)
        C = None if inp["C"] is None else lg(inp["C"].to(dev), w.layout_c)
        D = lg(torch.empty(storage_shape(w.M, w.N, w.layout_d), dtype=TORCH_DTYPE[w.d_type],
                           device=dev), w.layout_d)
        sets.append((A, B, C, D))
    cands = [c for c in args.candidates.split(";") if c.strip()]
    handles = []
    for c in cands:
        if c == "cublas":
            handles.append(LibraryReference(w))
            continue
        if c == "default":  # the plan the library picks by itself
            os.environ.pop("GEMM_FORCE_PLAN", None)
        else:
            os.environ["GEMM_FORCE_PLAN"] = c
        handles.append(pkg.Gemm.like(*sets[0]))
    os.environ.pop("GEMM_FORCE_PLAN", None)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    def run(g, n, base=0):
        for i in range(n):
            A, B, C, D = sets[(base + i) % nsets]
            if isinstance(g, LibraryReference):
                g.run(A, B, C, D)
                continue
            g.run_ptrs(A.data_ptr(), B.data_ptr(), None if C is None else C.data_ptr(),
                       D.data_ptr(), sp)

    for g in handles:
        run(g, 3)
        if isinstance(g, LibraryReference):
            torch.cuda.synchronize()
            continue
        st = g.status(stream)
        if st != pkg.GEMM_OK:
            raise RuntimeError(f"candidate {g.plan()} failed: {pkg.gemm_strerror(st)}")
    times = [[] for _ in handles]
    for r in range(args.repeats):
        for ci, g in enumerate(handles):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            s.record(stream)
            run(g, args.iters, r)
            e.record(stream)
            torch.cuda.synchronize()
            times[ci].append(s.elapsed_time(e) / args.iters)
    for ci, g in enumerate(handles):
        if not isinstance(g, LibraryReference) and g.status(stream) != pkg.GEMM_OK:
            raise RuntimeError(f"candidate {g.plan()} timed out")
        med = statistics.median(times[ci])
        spread = (max(times[ci]) - min(times[ci])) / med
        print(json.dumps({"workload": w.name, "candidate": cands[ci], "plan": g.plan(),
                          "median_ms": round(med, 5), "spread": round(spread, 4),
                          "tflops": round(w.flops / (med * 1e-3) / 1e12, 1)}), flush=True)
        g.close()
    return 0


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", action="append", required=True)
    ap.add_argument("--candidates", required=True, help="';'-separated GEMM_FORCE_PLAN strings")
    ap.add_argument("--repeats", type=int, default=7)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--child", action="store_true")
    args = ap.parse_args()
    if args.child:
        args.workload = args.workload[0]
        return child(args)
    rc = 0
    for wl in args.workload:
        cmd = [sys.executable, "-m", "dense_tiled_gemm_02_gb300.tune", "--child", "--workload", wl,
               "--candidates", args.candidates, "--repeats", str(args.repeats),
               "--iters", str(args.iters)]
        r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
        sys.stdout.write(r.stdout)
        if r.returncode != 0:
            print(json.dumps({"workload": wl, "error": r.stderr.strip().splitlines()[-1:]}))
            rc = 1
    return rc


if __name__ == "__main__":
    sys.exit(main())
