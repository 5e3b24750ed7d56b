"""One Nsight Compute capture of a workload's GEMM kernel, from the plain run
to the committed record.

    python -m dense_tiled_gemm_02_gb300.ncu_capture --workload sq4096_bf16 \
        --kernel-regex tc_gemm_pair_kernel --out-dir out/profiles \
        [--plan native_i8=1] [--skip 3]

For one workload this
  1. runs the benchmark once without ncu (it must exit 0 before ncu runs it),
  2. takes the launch list of the same command (``--metrics
     gpu__time_duration.sum``: one pass, every launch, cold cache and
     serialised, so only the shares are comparable with the benchmark),
  3. captures one launch of the kernel (``--set full``, after ``--skip``
     launches of it) on the same command,
  4. writes ``<out-dir>/<kernel>_<workload>.json`` (ncu_record.make_record:
     DRAM bytes, duration, pipe utilisation, source hash, plan) and a short
     ``.md`` summary with the commands, the table and the launch list.

Every ncu command carries ``--clock-control none``.  The benchmark command is
the short form: three warm-up and three timed steps, one repeat, no CPU
baseline and no end-to-end pass, so that the program holds one workload's
input sets on the device (a few hundred MB to about 1.4 GB) and the captured
launch is the fourth launch of its kernel.
"""
from __future__ import annotations

import argparse
import os
import shlex
import subprocess
import sys
import time

from . import ncu_record

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bench_cmd(workload: str) -> list[str]:
    return [sys.executable, "bench.py", "--workload", workload, "--steps", "3", "--warmup", "3",
            "--repeats", "1", "--repeat-ms", "1", "--also", "none", "--no-cpu-baseline",
            "--no-e2e"]


def run(cmd: list[str], log: str, env: dict) -> int:
    t0 = time.time()
    with open(log, "w") as f:
        rc = subprocess.run(cmd, cwd=ROOT, env=env, stdout=f, stderr=subprocess.STDOUT).returncode
    print(f"[{time.time() - t0:6.1f} s] rc={rc} {' '.join(shlex.quote(c) for c in cmd)}",
          flush=True)
    return rc


def summary(rec: dict, cmds: dict) -> str:
    algo = rec.get("algorithmic_bytes")
    use = (["capture; the JSON beside this file holds the same figures (an auxiliary",
            "kernel of the call: informational, `bench.py` reads no such record)."]
           if rec.get("family") == "aux" else
           ["capture; the JSON beside this file holds the same figures and is what",
            "`bench.py` reads for `roofline.traffic` (only while the kernel family's",
            "device sources hash to `source_hash` and the plan string is the same)."])
    lines = [f"# {rec['kernel']} -- {rec['workload']}", "",
             "Machine-written by `dense_tiled_gemm_02_gb300/ncu_capture.py` from one ncu"] + use + ["",
             f"- plan: `{rec['plan']}`", f"- source_hash ({rec['family']}): `{rec['source_hash']}`"]
    if algo and rec.get("dram_bytes_per_launch"):
        lines.append(f"- DRAM bytes per launch {rec['dram_bytes_per_launch'] / 1e6:.1f} MB against "
                     f"{algo / 1e6:.1f} MB algorithmic: ratio "
                     f"{rec['dram_bytes_per_launch'] / algo:.3f}")
    b = rec.get("bench") or {}
    lines += [f"- plain run of the same command: {b.get('value')} {b.get('unit')}, "
              f"{b.get('ms_per_step')} ms per step (three steps; not a bench figure)", "",
              "Commands (from the repository root, on one GB300):", "", "    " + cmds["plain"],
              "    " + cmds["launches"], "    " + cmds["full"], "", ncu_record.markdown(rec), ""]
    return "\n".join(lines)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", required=True)
    ap.add_argument("--kernel-regex", required=True)
    ap.add_argument("--plan", default="", help="GEMM_FORCE_PLAN for the run (plan keys)")
    ap.add_argument("--skip", type=int, default=3, help="launches of the kernel before the capture")
    ap.add_argument("--max-launches", type=int, default=60, help="launch-list length")
    ap.add_argument("--out-dir", required=True)
    ap.add_argument("--scratch", default=None, help="raw output folder (default: out-dir/raw)")
    a = ap.parse_args(argv)
    os.makedirs(a.out_dir, exist_ok=True)
    scratch = a.scratch or os.path.join(a.out_dir, "raw")
    os.makedirs(scratch, exist_ok=True)
    tag = a.workload + (("_" + a.plan.replace("=", "").replace(" ", "_")) if a.plan else "")
    env = dict(os.environ)
    if a.plan:
        env["GEMM_FORCE_PLAN"] = a.plan
    cmd = bench_cmd(a.workload)
    launches_csv = os.path.join(scratch, tag + ".launches.csv")
    rep = os.path.join(scratch, tag)
    ncu_l = ["ncu", "--metrics", "gpu__time_duration.sum", "--clock-control", "none", "-c",
             str(a.max_launches), "--csv", "--log-file", launches_csv] + cmd
    ncu_f = ["ncu", "--set", "full", "--clock-control", "none", "-k", "regex:" + a.kernel_regex,
             "-s", str(a.skip), "-c", "1", "-f", "-o", rep] + cmd
    plain_log = os.path.join(scratch, tag + ".plain.log")
    if run(cmd, plain_log, env) != 0:
        print("plain run failed; no capture", flush=True)
        return 1
    if run(ncu_l, os.path.join(scratch, tag + ".ncu_launches.log"), env) != 0:
        return 2
    if run(ncu_f, os.path.join(scratch, tag + ".ncu_full.log"), env) != 0:
        return 3
    raw = subprocess.run(["ncu", "-i", rep + ".ncu-rep", "--page", "raw", "--csv",
                          "--print-units", "base"], check=True, capture_output=True,
                         text=True).stdout
    with open(rep + ".raw.csv", "w") as f:
        f.write(raw)
    launches = ncu_record.parse_launch_list(open(launches_csv).read())
    rec = ncu_record.make_record(ncu_record.parse_raw_csv(raw), launches,
                                 ncu_record.bench_line(plain_log), a.kernel_regex)
    if a.plan:
        rec["forced_plan"] = a.plan
    stem = ncu_record.aux_stem(a.kernel_regex) or ncu_record.kernel_stem(rec["plan"])
    if not ncu_record.aux_stem(a.kernel_regex) and stem + "_kernel" not in rec["kernel"]:
        # a GEMM record must hold the plan's GEMM kernel, whatever the regex matched
        print(f"captured {rec['kernel']}, not the plan's {stem}_kernel: no record", flush=True)
        return 4
    out = os.path.join(a.out_dir, f"{stem}_{rec['workload']}")
    import json
    with open(out + ".json", "w") as f:
        json.dump(rec, f, indent=1, sort_keys=True)
        f.write("\n")
    pre = f"GEMM_FORCE_PLAN='{a.plan}' " if a.plan else ""
    cmds = {"plain": pre + " ".join(["python"] + cmd[1:]),
            "launches": pre + " ".join(["ncu"] + ncu_l[1:ncu_l.index("--log-file")] +
                                       ["--log-file", "launches.csv", "python"] + cmd[1:]),
            "full": pre + " ".join(["ncu"] + ncu_f[1:ncu_f.index("-o")] +
                                   ["-o", "prof", "python"] + cmd[1:])}
    with open(out + ".md", "w") as f:
        f.write(summary(rec, cmds))
    print(f"wrote {out}.json", flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
