"""CPU tests of the benchmark's plan-string parsing and roofline arithmetic.

The bench line's kernel name, launch count and algorithmic bytes are read off
the library's plan string (gemm_plan_string); these tests pin that parsing on
plan strings of each kernel family, so that a change of the string's format
cannot silently change what the line reports.
"""
from __future__ import annotations

import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from workloads import WORKLOADS  # noqa: E402

FIELDS = ("decode", "dbulk", "swap", "pair", "bn", "ksub", "stages", "group_m", "splits",
          "kb_per_split", "tail", "grid", "i8x", "a_mn", "b_mn", "repack_a", "repack_b",
          "stage_c", "stage_d", "ws_bytes")


def plan(**kw) -> str:
    """A plan string in the library's format (keys in its order)."""
    vals = dict.fromkeys(FIELDS, 0)
    vals.update(bn=256, stages=6, group_m=8, splits=1, ksub=1, grid=152)
    vals.update(kw)
    return "M=4096 N=4096 K=4096 " + " ".join(f"{k}={vals[k]}" for k in FIELDS)


class _G:
    def __init__(self, s):
        self.s = s

    def plan(self):
        return self.s


def test_kernel_family_and_name():
    p = plan(pair=1)
    assert bench.kernel_family(p) == "pair"
    assert bench.kernel_name(p) == "tc_gemm_pair_kernel<256, 6, 1>"
    p = plan(bn=64, stages=8)
    assert bench.kernel_family(p) == "cta1"
    assert bench.kernel_name(p) == "tc_gemm_kernel<64, 8, 0>"
    p = plan(decode=1, dbulk=1, bn=0, stages=0)
    assert bench.kernel_family(p) == "decode"
    assert bench.kernel_name(p) == "decode_bulk_kernel"
    assert bench.kernel_name(plan(decode=1, dbulk=0)) == "decode_kn_kernel"


def test_launches_per_step():
    assert bench.launches_per_step(_G(plan(pair=1))) == 1
    assert bench.launches_per_step(_G(plan(decode=1, dbulk=1, splits=2))) == 1
    assert bench.launches_per_step(_G(plan(splits=2))) == 2          # GEMM + reduce
    # 16-bit copies before the GEMM share one launch; D's copy is its own
    assert bench.launches_per_step(_G(plan(repack_a=1, repack_b=1, stage_c=1))) == 2
    assert bench.launches_per_step(_G(plan(repack_b=1, stage_d=1))) == 3
    # exact int8: one widening launch per widened operand
    assert bench.launches_per_step(_G(plan(i8x=1, repack_a=1, repack_b=1, pair=1))) == 3


def test_algorithmic_bytes_and_job_value():
    w = WORKLOADS["sq4096_bf16"]
    assert bench.algorithmic_bytes(w) == 4 * 4096 * 4096 * 2
    w = WORKLOADS["sq8192_i8"]
    assert bench.algorithmic_bytes(w) == 2 * 8192 * 8192 + 2 * 8192 * 8192 * 4
    w = WORKLOADS["sq1024_f16"]                                 # C absent
    assert bench.algorithmic_bytes(w) == 3 * 1024 * 1024 * 2
    # 2 M N K flop in 1 ms on one rank: 137.4 TFLOP/s at 4096^3
    assert abs(bench.job_value(2 * 4096 ** 3, 1.0, 1) - 137.438953472) < 1e-9
