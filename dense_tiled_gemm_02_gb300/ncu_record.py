"""Machine-written records of Nsight Compute captures, and the source hashes
that say which build a record belongs to.

A record ties one kernel's DRAM traffic, duration and pipe utilisation to
the exact device sources and the plan that produced it, so that the
benchmark reports `roofline.traffic` only for the build and plan it timed
("Tuning Triton" skill page, section 7: verify that the framework really
runs the kernel you measured).

    python -m dense_tiled_gemm_02_gb300.ncu_record \
        --rep prof.ncu-rep [--launches launches.csv] --bench-log plain.log \
        --out profiles/tc_gemm_pair_sq4096_bf16

reads the full capture with ``ncu -i <rep> --page raw --csv --print-units
base``, the optional launch list (``--metrics gpu__time_duration.sum --csv``)
and the plan and workload from the benchmark's JSON line, and writes
``<out>.json``.  Run it on the machine that made the capture, right after
it: the hash is taken from the sources present there.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")

# Device sources of each kernel family: the kernel, the helpers it includes
# and its launch unit.  Host planner changes are caught by comparing the
# plan string instead.
FAMILY_SOURCES = {
    "pair": ("common.h", "ptx.cuh", "tc_gemm.cuh", "tc_gemm2.cuh", "tc_pair_launch.cu"),
    "cta1": ("common.h", "ptx.cuh", "tc_gemm.cuh", "tc_launch.cu"),
    "decode": ("common.h", "ptx.cuh", "decode.cu"),
    "i8mma": ("common.h", "ptx.cuh", "i8_mma.cu"),
    # the auxiliary kernels around a GEMM (split-K reduce, row copies, int8
    # widening); their records are informational, the benchmark reads none
    "aux": ("common.h", "ptx.cuh", "aux_kernels.cu"),
}

# Records of auxiliary kernels: kernel-name pattern -> file-name stem.
AUX_STEMS = {
    "splitk_reduce_kernel": "splitk_reduce",
    "copy_rows16": "copy_rows16",
    "widen_i8": "widen_i8",
}

# Metrics copied into the record (base units): name -> key in the record.
RECORD_METRICS = {
    "gpu__time_duration.sum": "duration_ns",
    "dram__bytes_read.sum": "dram_read_bytes",
    "dram__bytes_write.sum": "dram_write_bytes",
    "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed": "dram_busy_pct",
    "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed": "tensor_pipe_pct_elapsed",
    "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active": "tensor_pipe_pct_active",
    "sm__throughput.avg.pct_of_peak_sustained_elapsed": "sm_throughput_pct",
    "lts__t_sector_hit_rate.pct": "l2_hit_pct",
    "sm__cycles_elapsed.avg.per_second": "sm_clock_hz",
    "launch__registers_per_thread": "registers_per_thread",
    "launch__grid_size": "grid_size",
    "launch__block_size": "block_size",
    "launch__shared_mem_per_block_dynamic": "dynamic_smem_bytes",
}


def family_of(plan: str) -> str:
    """Kernel family of the GEMM kernel a plan string launches."""
    if re.search(r"\bdecode=1\b", plan):
        return "decode"
    if re.search(r"\bnative_i8=1\b", plan):
        return "i8mma"
    return "pair" if re.search(r"\bpair=1\b", plan) else "cta1"


def kernel_stem(plan: str) -> str:
    """File-name stem of the kernel a plan launches (the decode family's two
    forms are two kernels)."""
    fam = family_of(plan)
    if fam == "decode":
        return "decode_bulk" if re.search(r"\bdbulk=1\b", plan) else "decode_kn"
    return {"i8mma": "i8_mma", "pair": "tc_gemm_pair", "cta1": "tc_gemm"}[fam]


def aux_stem(kernel_regex):
    """File-name stem when the captured kernel is an auxiliary one, else None."""
    for pat, stem in AUX_STEMS.items():
        if kernel_regex and pat in kernel_regex:
            return stem
    return None


def source_hash(family: str) -> str:
    """Hash of the device sources of one kernel family."""
    h = hashlib.sha256()
    for name in FAMILY_SOURCES[family]:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def record_path(root: str, plan: str, workload: str) -> str:
    return os.path.join(root, "profiles", f"{kernel_stem(plan)}_{workload}.json")


def load_record(root: str, plan: str, workload: str):
    """The committed record for this plan and workload when it is current
    (same device sources, same plan), else None."""
    try:
        with open(record_path(root, plan, workload)) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_hash") != source_hash(family_of(plan)) or rec.get("plan") != plan:
        return None
    return rec


def _num(s: str):
    s = s.strip().replace(",", "")
    if s in ("", "nan", "n/a"):
        return None
    try:
        return float(s)
    except ValueError:
        return None


def parse_raw_csv(text: str) -> list[dict]:
    """Rows of ``ncu --page raw --csv --print-units base``: one dict per
    captured launch, metric name -> value (numbers as floats)."""
    rows = list(csv.reader(io.StringIO(text)))
    rows = [r for r in rows if r]
    start = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    header = rows[start]
    out = []
    for r in rows[start + 2:]:  # the row after the header holds the units
        if len(r) != len(header):
            continue
        d = {}
        for k, v in zip(header, r):
            n = _num(v)
            d[k] = n if n is not None else v
        out.append(d)
    return out


def parse_launch_list(text: str) -> list[dict]:
    """Per-kernel launches, total time and share from a ``--metrics
    gpu__time_duration.sum --csv`` log (details page, base units)."""
    lines = text.splitlines()
    start = next((i for i, ln in enumerate(lines) if ln.startswith('"ID"')), None)
    if start is None:
        return []
    rd = csv.DictReader(io.StringIO("\n".join(lines[start:])))
    per = {}
    for r in rd:
        if r.get("Metric Name") != "gpu__time_duration.sum":
            continue
        name = r["Kernel Name"].split("(")[0].replace("void ", "").strip()
        unit = (r.get("Metric Unit") or "ns").strip()
        v = _num(r["Metric Value"]) or 0.0
        scale = {"ns": 1e-3, "nsecond": 1e-3, "us": 1.0, "usecond": 1.0, "ms": 1e3,
                 "msecond": 1e3}.get(unit, 1e-3)
        e = per.setdefault(name, [0, 0.0])
        e[0] += 1
        e[1] += v * scale
    total = sum(v[1] for v in per.values()) or 1.0
    return [{"kernel": k, "launches": v[0], "total_us": round(v[1], 2),
             "share": round(v[1] / total, 4)}
            for k, v in sorted(per.items(), key=lambda kv: -kv[1][1])]


def bench_line(path: str) -> dict:
    with open(path) as f:
        for ln in reversed(f.read().strip().splitlines()):
            ln = ln.strip()
            if ln.startswith("{"):
                return json.loads(ln)
    raise ValueError(f"no JSON line in {path}")


def make_record(raw_rows: list[dict], launches: list[dict], line: dict,
                kernel_regex: str | None) -> dict:
    plan = line["config"]["plan"]
    workload = line["config"]["workload"]
    rows = raw_rows
    if kernel_regex:
        rows = [r for r in rows if re.search(kernel_regex, str(r.get("Kernel Name", "")))]
    if not rows:
        raise ValueError("no captured launch matches")
    aux = aux_stem(kernel_regex)
    family = "aux" if aux else family_of(plan)
    rec = {"workload": workload, "plan": plan, "family": family,
           "source_hash": source_hash(family),
           "kernel": str(rows[0].get("Kernel Name", "")).split("(")[0].replace("void ", ""),
           "launches_captured": len(rows)}
    for name, key in RECORD_METRICS.items():
        vals = [r[name] for r in rows if isinstance(r.get(name), float)]
        if vals:
            rec[key] = statistics.mean(vals)
    if "dram_read_bytes" in rec and "dram_write_bytes" in rec:
        rec["dram_bytes_per_launch"] = rec["dram_read_bytes"] + rec["dram_write_bytes"]
        if rec.get("duration_ns"):
            rec["dram_gbs"] = round(rec["dram_bytes_per_launch"] / rec["duration_ns"], 1)
        # (the bench line's algorithmic bytes are the GEMM's, not an
        # auxiliary kernel's)
        algo = None if aux else line.get("roofline", {}).get("algorithmic_bytes")
        if algo:
            rec["algorithmic_bytes"] = algo
            rec["traffic_over_algorithmic"] = round(rec["dram_bytes_per_launch"] / algo, 4)
    if launches:
        rec["launch_list"] = launches
    rec["bench"] = {k: line.get(k) for k in ("value", "unit", "ms_per_step")}
    rec["bench"]["roofline_frac"] = line.get("roofline", {}).get("frac")
    return rec


def markdown(rec: dict) -> str:
    """A short table of the record, for the human-written summary beside it."""
    out = [f"| metric | value |", "|---|---|"]
    for key in ("duration_ns", "sm_clock_hz", "dram_read_bytes", "dram_write_bytes",
                "dram_bytes_per_launch", "dram_gbs", "algorithmic_bytes", "traffic_over_algorithmic",
                "dram_busy_pct", "tensor_pipe_pct_elapsed", "tensor_pipe_pct_active",
                "sm_throughput_pct", "l2_hit_pct", "registers_per_thread", "grid_size",
                "block_size", "dynamic_smem_bytes"):
        if key in rec:
            v = rec[key]
            out.append(f"| {key} | {v:.4g} |" if isinstance(v, float) else f"| {key} | {v} |")
    if rec.get("launch_list"):
        out += ["", "| kernel | launches | total µs | share |", "|---|---|---|---|"]
        out += [f"| {e['kernel']} | {e['launches']} | {e['total_us']} | {100 * e['share']:.1f} % |"
                for e in rec["launch_list"]]
    return "\n".join(out)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--rep", help="ncu report of the full capture (.ncu-rep)")
    ap.add_argument("--raw", help="already exported raw CSV (instead of --rep)")
    ap.add_argument("--launches", help="launch-list CSV log")
    ap.add_argument("--bench-log", required=True, help="log holding the benchmark's JSON line")
    ap.add_argument("--kernel-regex", default=None)
    ap.add_argument("--out", required=True, help="output path without extension")
    a = ap.parse_args(argv)
    if a.raw:
        text = open(a.raw).read()
    else:
        text = subprocess.run(["ncu", "-i", a.rep, "--page", "raw", "--csv", "--print-units",
                               "base"], check=True, capture_output=True, text=True).stdout
    launches = parse_launch_list(open(a.launches).read()) if a.launches else []
    rec = make_record(parse_raw_csv(text), launches, bench_line(a.bench_log), a.kernel_regex)
    with open(a.out + ".json", "w") as f:
        json.dump(rec, f, indent=1, sort_keys=True)
        f.write("\n")
    print(markdown(rec))
    return 0


if __name__ == "__main__":
    sys.exit(main())
