"""Benchmark: D = A*B + C through the C ABI on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--also NAMES|none]

One step is one D = A*B + C of the workload (default: 4096^3 bf16, A
row-major, B column-major, C and D bf16, the configuration the headline
metric is quoted on).  Inputs are seeded synthetic data, resident in HBM
before the timed region; the step rotates over enough input sets that the
working set of consecutive steps exceeds L2.  Timing: W untimed warm-up
steps, then K steps bracketed by a barrier and a device synchronisation,
CUDA events on the launching stream; the line reports the maximum over
ranks.  The GEMM is not sharded: N > 1 runs N independent replicas (one per
GPU) and `value` sums their throughput ("weak" scaling).

After that region, `repeats` times the same step in R further regions of at
least --repeat-ms each and reports their median and spread (the noise
protocol of the "Tuning Triton" page, section 2); the clock samples cover
all of them.

The default run also measures the rest of the metric with the same protocol
and prints it in the same line under `also`: 8192^3 bf16 (the size the
target names beside 4096^3) and 8192^3 int8 -> int32 (the metric's TOPS).

`e2e` is the same metric measured through the library's host-buffer entry
point (gemm_run_host_batch) with the operands in pinned host memory: every
step copies A, B, C host->device, runs the GEMM and copies D back, all
inside the timed region; the library overlaps one step's input copies with
the previous step's GEMM and output copy.

`--impl reference` times the CPU oracle (test infrastructure, fp64 triple
loop) on the host cores, on a bounded sample of rows of the same workload,
and reports the same metric.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 10 ** 6
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
HEADLINE = "sq4096_bf16"
ALSO_DEFAULT = ("sq8192_bf16", "sq8192_i8")
# Dense tensor-core rate of one SM: 8192 bf16 FLOP per clock (a 128 x 256 x 16
# MMA, 1 M FLOP, every 128 clocks); 8-bit floats twice that.
DENSE_FLOP_PER_CLK_SM = 8192
HBM_NOMINAL_GBS = 7900.0
# Workloads of the CPU-baseline matrix (single core and all cores), and the
# 8192^3 workloads whose sampled check is timed and extrapolated.
CPU_MATRIX = ("sq256_f16_f32", "sq1024_f16", "sq4096_bf16", "rag1000_bf16",
              "rag4095x4097x4099_bf16")
CPU_SAMPLED = ("sq8192_bf16", "sq8192_i8")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--also", default="auto",
                    help="comma-separated extra workloads timed the same way, 'none', or "
                         "'auto' (8192^3 bf16 and int8 with the headline workload)")
    ap.add_argument("--repeats", type=int, default=7)
    ap.add_argument("--repeat-ms", type=float, default=100.0,
                    help="minimum length of each repeat region")
    ap.add_argument("--nsets", type=int, default=0,
                    help="input sets rotated over (0: enough for > 2x L2)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cpu-matrix", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="target CPU time of the whole reference-arm run (the oracle)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    return ap.parse_args()


def job_step_ms(total_ms: float, steps: int, world: int) -> float:
    """Per-step time of the whole job: the slowest rank's timed region (every
    rank holds one replica, so the job ends with the last of them)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_ms], dtype=torch.float64,
                         device="cuda" if dist.get_backend() == "nccl" else "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms / steps


def job_value(flops_per_step: float, step_ms: float, world: int) -> float:
    """Aggregate throughput (TFLOP/s or TOPS) of `world` replicas."""
    return flops_per_step / (step_ms * 1e-3) / 1e12 * world


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


def also_list(args) -> list[str]:
    if args.also == "none":
        return []
    if args.also == "auto":
        return list(ALSO_DEFAULT) if args.workload == HEADLINE else []
    return [a for a in args.also.split(",") if a]


class ClockSampler:
    """nvidia-smi samples during the timed regions."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            try:
                pw.append(float(parts[3]))
            except ValueError:
                pass
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        # "under load": samples while the board draws well above idle power
        load = [s for s, p in zip(sm, pw) if p > 0.5 * max(pw)] if pw else sm
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(load),
                "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------- the CPU oracle
def oracle_rows_runner(w, inp):
    import oracle
    from workloads import I8, bits_of, bits_u16
    orc = oracle.get()
    if w.ab_type == I8:
        A, B = inp["A"].numpy(), inp["B"].numpy()
        C = None if inp["C"] is None else inp["C"].numpy()
        run = lambda rows: orc.gemm_i64_rows(w.M, w.N, w.K, A, B, C, a_col=w.layout_a,
                                             b_col=w.layout_b, c_col=w.layout_c, rows=rows)
    else:
        A, B = bits_of(inp["A"]), bits_of(inp["B"])
        C = None if inp["C"] is None else (inp["C"].numpy() if w.c_type == 3 else
                                           bits_u16(inp["C"]))
        run = lambda rows: orc.gemm_f64_rows(w.M, w.N, w.K, A, B, C, ab_type=w.ab_type,
                                             c_type=w.c_type or 0, a_col=w.layout_a,
                                             b_col=w.layout_b, c_col=w.layout_c, rows=rows,
                                             want_s=False)
    return run, orc.threads()


def oracle_points_runner(w, inp):
    """The oracle's sampled check at full size: 65,536 seeded points plus 64
    full rows (the sampling rule of the parity tests)."""
    import numpy as np

    import oracle
    from workloads import I8, bits_of, bits_u16, sample_points, sample_rows
    orc = oracle.get()
    pi, pj = sample_points(w.M, w.N)
    pi, pj = pi.numpy(), pj.numpy()
    rows = sample_rows(w.M).numpy()
    if w.ab_type == I8:
        A, B = inp["A"].numpy(), inp["B"].numpy()
        C = None if inp["C"] is None else inp["C"].numpy()
        kw = dict(a_col=w.layout_a, b_col=w.layout_b, c_col=w.layout_c)

        def run():
            orc.gemm_i64_points(w.M, w.N, w.K, A, B, C, pi, pj, **kw)
            orc.gemm_i64_rows(w.M, w.N, w.K, A, B, C, rows=rows, **kw)
    else:
        A, B = bits_of(inp["A"]), bits_of(inp["B"])
        C = None if inp["C"] is None else bits_u16(inp["C"])
        kw = dict(ab_type=w.ab_type, c_type=w.c_type or 0, a_col=w.layout_a,
                  b_col=w.layout_b, c_col=w.layout_c)

        def run():
            orc.gemm_f64_points(w.M, w.N, w.K, A, B, C, pi, pj, **kw)
            orc.gemm_f64_rows(w.M, w.N, w.K, A, B, C, rows=rows, want_s=False, **kw)
    return run, int(pi.size + rows.size * w.N)


def calibrate_rows(run, M: int, target_s: float) -> int:
    """Rows per oracle call so that one call takes about target_s seconds.

    A call has a fixed cost (widening B) and a per-row cost; two timed calls
    separate them."""
    import numpy as np
    n1, n2 = min(M, 2), min(M, 10)
    t0 = time.perf_counter()
    run(np.arange(n1))
    t1 = time.perf_counter()
    run(np.arange(n2))
    t2 = time.perf_counter()
    if n2 == n1:
        return n1
    per_row = max((t2 - t1) - (t1 - t0), 1e-9) / (n2 - n1)
    fixed = max((t1 - t0) - n1 * per_row, 0.0)
    return int(max(1, min(M, (target_s - fixed) / per_row)))


def cpu_baseline(w, inp, target_s: float) -> dict:
    """The oracle as it stands, timed on a bounded sample of whole rows."""
    import numpy as np
    from workloads import I8
    run, threads = oracle_rows_runner(w, inp)
    n2 = calibrate_rows(run, w.M, target_s)
    t0 = time.perf_counter()
    run(np.arange(n2))
    dt = time.perf_counter() - t0
    flops = 2.0 * n2 * w.N * w.K
    return {"value": flops / dt / 1e12, "unit": "TOPS" if w.ab_type == I8 else "TFLOPS",
            "cores": threads, "kind": "oracle",
            "sample": f"{n2} of {w.M} output rows ({n2 * w.N} elements), fp64/int64 triple "
                      f"loop, {dt:.1f} s"}


def cpu_matrix(inputs: dict, budget_s: float = 1.5) -> list[dict]:
    """The oracle on one core and on all cores, per workload: the whole GEMM
    when it fits the budget, else a sample of rows with the full time
    extrapolated from it (labelled).  At 8192^3, the sampled parity check
    (65,536 points and 64 rows) is timed and the per-element rate
    extrapolated to all M x N elements (labelled)."""
    import numpy as np

    import oracle
    from workloads import I8, WORKLOADS, make_inputs
    orc = oracle.get()
    all_threads = orc.threads()
    out = []
    try:
        for name in CPU_MATRIX:
            w = WORKLOADS[name]
            inp = inputs.get(name) or make_inputs(w)
            for threads in (1, all_threads):
                orc.set_threads(threads)
                run, _ = oracle_rows_runner(w, inp)
                rows = calibrate_rows(run, w.M, budget_s)
                t0 = time.perf_counter()
                run(np.arange(rows))
                dt = time.perf_counter() - t0
                full = dt * w.M / rows
                out.append({"workload": name, "threads": threads, "rows": rows, "of_rows": w.M,
                            "seconds": round(dt, 4), "full_gemm_seconds": round(full, 4),
                            "extrapolated": rows < w.M,
                            "value": round(w.flops / full / 1e12, 6),
                            "unit": "TOPS" if w.ab_type == I8 else "TFLOPS"})
        orc.set_threads(all_threads)
        for name in CPU_SAMPLED:
            w = WORKLOADS[name]
            inp = inputs.get(name) or make_inputs(w)
            run, elems = oracle_points_runner(w, inp)
            t0 = time.perf_counter()
            run()
            dt = time.perf_counter() - t0
            full = dt * (w.M * w.N) / elems
            out.append({"workload": name, "threads": all_threads,
                        "sample": "65536 points + 64 rows", "elements": elems,
                        "seconds": round(dt, 4), "full_gemm_seconds": round(full, 2),
                        "extrapolated": True,
                        "value": round(w.flops / full / 1e12, 6),
                        "unit": "TOPS" if w.ab_type == I8 else "TFLOPS"})
    finally:
        orc.set_threads(all_threads)
    return out


def run_reference(args, w):
    """The oracle as the reference arm: each step is a bounded sample of rows."""
    import numpy as np
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from workloads import I8, make_inputs
    inp = make_inputs(w)
    total_steps = max(1, args.steps + args.warmup)
    per_step_s = min(10.0, max(0.02, args.ref_seconds / total_steps))
    run, threads = oracle_rows_runner(w, inp)
    rows_per_step = calibrate_rows(run, w.M, per_step_s)
    for i in range(args.warmup):
        run((np.arange(rows_per_step) + i * rows_per_step) % w.M)
    t0 = time.perf_counter()
    for i in range(args.steps):
        run((np.arange(rows_per_step) + i * rows_per_step) % w.M)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows_per_step * w.N * w.K * args.steps
    value = flops / dt / 1e12
    unit = "TOPS" if w.ab_type == I8 else "TFLOPS"
    sample = (f"{rows_per_step} of {w.M} output rows per step ({rows_per_step * w.N} elements), "
              f"fp64/int64 triple loop, {args.steps} timed steps in {dt:.1f} s")
    line = {"impl": "reference", "metric": metric_name(w), "value": value, "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64" if w.ab_type != I8 else "int64",
            "data": "synthetic (seeded)", "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def logical(storage, layout):
    return storage if layout == 0 else storage.t()


def metric_name(w) -> str:
    from workloads import F8, I8
    if w.ab_type in F8:
        return "GEMM TFLOPS (fp8, block-scaled)" if w.mx else "GEMM TFLOPS (fp8)"
    return "GEMM TOPS (int8)" if w.ab_type == I8 else "GEMM TFLOPS (bf16/fp16)"


def config_of(w) -> dict:
    from workloads import TYPE_NAME
    lay = lambda l: "row" if l == 0 else "col"
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
            "types": f"{TYPE_NAME[w.ab_type]}x{TYPE_NAME[w.ab_type]}+"
                     f"{TYPE_NAME[w.c_type] if w.c_type else 'none'}->{TYPE_NAME[w.d_type]}",
            "layouts": f"A {lay(w.layout_a)}, B {lay(w.layout_b)}, C {lay(w.layout_c)}, "
                       f"D {lay(w.layout_d)}",
            "parallelism": "replicas"}


# ---------------------------------------------------------------- one workload on the GPU
def roofline_of(w, plan: str, avg_kernel_ms: float, events_ms: float, single: bool,
                sms: int, sm_max_mhz: float) -> dict:
    """The GEMM kernel's roofline: tensor-bound when its arithmetic intensity
    over the compulsory bytes (A, B, C and D once) is above the ridge of the
    two measured peaks, HBM-bound below it.  `frac` is against the measured
    peak (cuBLAS bf16 burst, or the copy bandwidth); `frac_of_dense_peak`
    against the clock-derived dense tensor peak (SMs x 8192 FLOP/clk x the
    maximum SM clock) or the nominal HBM3e bandwidth."""
    from dense_tiled_gemm_02_gb300 import ncu_record
    from workloads import F8
    peaks, src = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    dense_tf = sms * DENSE_FLOP_PER_CLK_SM * sm_max_mhz * 1e6 / 1e12
    peak_note = "bf16 burst (cuBLAS 8192^3)"
    if w.ab_type in F8:
        # the 8-bit tensor rate: the bf16 peaks times the nominal fp8 / bf16
        # ratio (4.5 / 2.25 PFLOP/s dense); no fp8 peak is measured here
        peak_tf *= 2.0
        dense_tf *= 2.0
        peak_note = "bf16 burst (cuBLAS 8192^3) x 2, the nominal fp8/bf16 ratio"
    algo_bytes = algorithmic_bytes(w)
    if w.flops / algo_bytes >= peak_tf * 1e12 / (peak_bw * 1e9):
        achieved = w.flops / (avg_kernel_ms * 1e-3) / 1e12
        r = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak_tf,
             "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
             "peak_source": f"{src} {peak_note}",
             "peak_dense": round(dense_tf, 1), "frac_of_dense_peak": round(achieved / dense_tf, 4),
             "peak_dense_source": f"{sms} SMs x {DENSE_FLOP_PER_CLK_SM} FLOP/clk x "
                                  f"{sm_max_mhz:.0f} MHz (maximum SM clock)"}
    else:
        achieved = algo_bytes / (avg_kernel_ms * 1e-3) / 1e9
        r = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak_bw,
             "unit": "GB/s", "frac": round(achieved / peak_bw, 4),
             "peak_source": f"{src} HBM copy bandwidth",
             "peak_dense": HBM_NOMINAL_GBS, "frac_of_dense_peak": round(achieved / HBM_NOMINAL_GBS, 4),
             "peak_dense_source": "nominal HBM3e bandwidth"}
    rec = ncu_record.load_record(ROOT, plan, w.name)
    r.update({"traffic": None if rec is None else rec.get("dram_bytes_per_launch"),
              "traffic_record": None if rec is None else
              os.path.relpath(ncu_record.record_path(ROOT, plan, w.name), ROOT),
              "algorithmic_bytes": algo_bytes, "kernel": kernel_name(plan),
              "kernel_ms_mean": round(avg_kernel_ms, 5),
              "kernel_ms_events_mean": round(events_ms, 5),
              "kernel_timing": ("timed region (the step is this one kernel)"
                                if single and avg_kernel_ms < events_ms else
                                "library events around each launch, second pass")})
    if rec is not None and rec.get("dram_bytes_per_launch"):
        r["traffic_over_algorithmic"] = round(rec["dram_bytes_per_launch"] / algo_bytes, 4)
    return r


def measure(pkg, w, args, dev, stream, world, local, sms, keep_inputs: bool = False):
    """Time one workload with the full protocol; returns (fields, inputs, handle)."""
    import torch
    import torch.distributed as dist
    from workloads import TORCH_DTYPE, make_inputs, storage_shape
    inp = make_inputs(w)
    set_bytes = sum(t.numel() * t.element_size() for t in inp.values() if t is not None)
    set_bytes += w.M * w.N * TORCH_DTYPE[w.d_type].itemsize
    nsets = args.nsets or max(2, -(-2 * L2_BYTES // set_bytes))  # a step cycle > 2x L2
    sets = []
    for i in range(nsets):
        A = logical(inp["A"].to(dev), w.layout_a)
        B = logical(inp["B"].to(dev), w.layout_b)
        C = None if inp["C"] is None else logical(inp["C"].to(dev), w.layout_c)
        Ds = torch.empty(storage_shape(w.M, w.N, w.layout_d), dtype=TORCH_DTYPE[w.d_type],
                         device=dev)
        sets.append((A, B, C, logical(Ds, w.layout_d)))
    g = pkg.Gemm.like(*sets[0], mx=w.mx)
    sptr = stream.cuda_stream
    if w.mx:  # E8M0 block scales, shared by the input sets
        from workloads import make_scales
        sc = {k: v.to(dev) for k, v in make_scales(w).items()}

    def step(i):
        A, B, C, D = sets[i % nsets]
        if w.mx:
            rc = pkg.gemm_run_mx(g.handle, A.data_ptr(), sc["SA"].data_ptr(), B.data_ptr(),
                                 sc["SB"].data_ptr(), None if C is None else C.data_ptr(),
                                 D.data_ptr(), sptr)
            if rc != pkg.GEMM_OK:
                raise pkg.GemmError(rc, "gemm_run_mx")
            return
        g.run_ptrs(A.data_ptr(), B.data_ptr(), None if C is None else C.data_ptr(),
                   D.data_ptr(), sptr)

    def check(what):
        st = g.status(stream)
        if st != pkg.GEMM_OK:
            raise RuntimeError(f"{w.name}: {what} failed: {pkg.gemm_strerror(st)}")

    for i in range(args.warmup):
        step(i)
    check("warm-up")

    # ---- the timed region: exactly K steps between a barrier + synchronise
    # and a synchronise.  Only the two events that bracket it: every timing
    # event is a point where the stream drains, which would show up in the
    # step time.
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize(dev)
    check("timed run")
    total_ms = start.elapsed_time(end)
    # ---- the tensor-core kernel alone: the same K steps again, with the
    # library recording an event pair around each of its launches (on this
    # stream).  When a step is that one kernel, the timed region above
    # already gives its duration without the events' own cost.
    g.timing_enable(args.steps)
    for i in range(args.steps):
        step(i)
    torch.cuda.synchronize(dev)
    kernel_ms = g.timing_read(args.steps)
    g.timing_enable(0)
    check("kernel timing run")
    if len(kernel_ms) != args.steps:
        raise RuntimeError(f"kernel timing recorded {len(kernel_ms)} of {args.steps} launches")
    # ---- repeats: R more regions of at least repeat_ms each
    step_guess = max(total_ms / args.steps, 1e-3)
    n_rep = max(args.steps, int(math.ceil(args.repeat_ms / step_guess)))
    rep_ms = []
    for r in range(args.repeats):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        s.record(stream)
        for i in range(n_rep):
            step(i)
        e.record(stream)
        torch.cuda.synchronize(dev)
        rep_ms.append(s.elapsed_time(e) / n_rep)
    check("repeats")
    clk = clocks.stop()

    ms = job_step_ms(total_ms, args.steps, world)
    total_ms = ms * args.steps
    value = job_value(w.flops, ms, world)
    events_ms = statistics.mean(kernel_ms)
    single = launches_per_step(g) == 1
    avg_kernel_ms = min(total_ms / args.steps, events_ms) if single else events_ms
    plan = g.plan()
    roofline = roofline_of(w, plan, avg_kernel_ms, events_ms, single, sms,
                           clk.get("sm_max_mhz") or load_peaks()[0].get("sm_max_mhz", 2070.0))
    med = statistics.median(rep_ms)
    unit = "TOPS" if w.ab_type == pkg.GEMM_I8 else "TFLOPS"
    repeats = {"n": len(rep_ms), "steps_each": n_rep, "median_ms_per_step": round(med, 5),
               "min_ms_per_step": round(min(rep_ms), 5), "max_ms_per_step": round(max(rep_ms), 5),
               "spread": round((max(rep_ms) - min(rep_ms)) / med, 4),
               "median_value": round(job_value(w.flops, med, world), 1), "unit": unit}
    fields = {"metric": metric_name(w), "value": round(value, 1), "unit": unit,
              "ms_per_step": round(ms, 5),
              "config": dict(config_of(w), l2="rotating %d input sets, %.0f MB > L2" %
                             (nsets, nsets * set_bytes / 1e6), plan=plan),
              "roofline": roofline, "clocks": clk, "repeats": repeats,
              "gpu_launches": launches_per_step(g) * args.steps}
    del sets
    return fields, (inp if keep_inputs else None), g


def main():
    args = parse()
    from workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)

    import torch
    import torch.distributed as dist

    import dense_tiled_gemm_02_gb300 as pkg
    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkg.load()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.current_stream(dev)

    from workloads import TYPE_NAME
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    fields, inp, g = measure(pkg, w, args, dev, stream, world, local, sms, keep_inputs=True)
    # ---- end to end through the same handle, host buffers
    e2e = None if args.no_e2e else e2e_measure(pkg, g, w, inp, dev, stream,
                                               max(8, args.steps), world)
    g.close()
    torch.cuda.empty_cache()
    also, also_inputs = [], {}
    for name in also_list(args):
        wa = WORKLOADS[name]
        fa, ia, ga = measure(pkg, wa, args, dev, stream, world, local, sms,
                             keep_inputs=want_cpu and name in CPU_SAMPLED)
        ga.close()
        torch.cuda.empty_cache()
        if ia is not None:
            also_inputs[name] = ia
        also.append(dict(workload=name, **fa))

    line = {"metric": fields["metric"], "value": fields["value"], "unit": fields["unit"],
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": fields["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": TYPE_NAME[w.ab_type],
            "data": "synthetic (seeded, resident in HBM)", "config": fields["config"],
            "roofline": fields["roofline"], "clocks": fields["clocks"],
            "repeats": fields["repeats"], "e2e": e2e, "gpu_launches": fields["gpu_launches"]}
    if also:
        line["also"] = also
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_seconds)
        if world == 1 and not args.no_cpu_matrix:
            line["cpu_baseline"]["matrix"] = cpu_matrix(dict(also_inputs, **{w.name: inp}))
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def kernel_name(plan: str) -> str:
    f = dict(kv.split("=") for kv in plan.split() if "=" in kv)
    if f.get("decode") == "1":
        return "decode_bulk_kernel" if f.get("dbulk") == "1" else "decode_kn_kernel"
    if f.get("native_i8") == "1":
        return "i8_mma_kernel"
    if f.get("pair") == "1":
        return f"tc_gemm_pair_kernel<{f['bn']}, {f['stages']}, {f.get('ksub', '1')}>"
    return f"tc_gemm_kernel<{f['bn']}, {f['stages']}, {f.get('i8x', '0')}>"


def algorithmic_bytes(w) -> int:
    """Compulsory DRAM bytes of one GEMM: A, B, C (when present) and D once."""
    from workloads import TORCH_DTYPE
    es = lambda t: TORCH_DTYPE[t].itemsize
    n = (w.M * w.K + w.K * w.N) * es(w.ab_type) + w.M * w.N * es(w.d_type)
    if w.c_type:
        n += w.M * w.N * es(w.c_type)
    return n


def launches_per_step(g) -> int:
    plan = g.plan()
    if re.search(r"\bdecode=1\b", plan):
        return 1  # the decode kernel finishes D itself
    n = 1
    m = re.search(r"splits=(\d+)", plan)
    csk = re.search(r"\bcsk=(\d+)", plan)
    if m and int(m.group(1)) > 1 and not (csk and int(csk.group(1)) > 1):
        n += 1  # the split-K reduce kernel (none when the splits meet in a cluster)
    flag = {k: int(re.search(k + r"=(\d)", plan).group(1))
            for k in ("repack_a", "repack_b", "stage_c", "stage_d", "i8x")}
    if re.search(r"\bmx=1\b", plan):
        n += 2  # the two scale-packing launches
    if flag["i8x"] or re.search(r"\bnative_i8=1\b", plan):
        # int8 operands are widened (or transposed) by one launch each
        n += flag["repack_a"] + flag["repack_b"]
    elif flag["repack_a"] or flag["repack_b"] or flag["stage_c"]:
        n += 1  # the 16-bit copies before the GEMM share one launch
    return n + flag["stage_d"]


def e2e_measure(pkg, g, w, inp, dev, stream, steps, world):
    """The metric through gemm_run_host_batch: operands in page-locked host
    memory, the K timed steps as one batch of K products, every step's H2D
    copies of A, B, C and D2H copy of D inside the timed region (the library
    overlaps one step's input copies with the previous step's GEMM and output
    copy; a call starts after the work already on its stream, so one product
    per call would serialise the copies)."""
    import torch
    from workloads import TORCH_DTYPE, storage_shape
    host = {k: (None if v is None else v.contiguous().pin_memory()) for k, v in inp.items()}
    shape = storage_shape(w.M, w.N, w.layout_d)
    hD = [torch.empty(shape, dtype=TORCH_DTYPE[w.d_type]).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = hD[0].numel() * hD[0].element_size()
    g.host_io_enable()
    Cs = None if host["C"] is None else [host["C"]]

    def batch(n):
        g.run_host_batch([host["A"]] * n, [host["B"]] * n, None if Cs is None else Cs * n,
                         [hD[i & 1] for i in range(n)], stream)

    batch(3)
    torch.cuda.synchronize(dev)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    batch(steps)
    e.record(stream)
    torch.cuda.synchronize(dev)
    ms = job_step_ms(s.elapsed_time(e), steps, world)
    return {"value": round(job_value(w.flops, ms, world), 1),
            "unit": "TOPS" if w.ab_type == 4 else "TFLOPS", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "api": "gemm_run_host_batch, one call of K products (pinned host operands)"}


if __name__ == "__main__":
    sys.exit(main())
