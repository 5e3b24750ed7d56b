"""CPU tests of the benchmark's plan-string parsing, roofline arithmetic and
the machine-written ncu records behind `roofline.traffic`.

The bench line's kernel name, launch count and algorithmic bytes are read off
the library's plan string (gemm_plan_string); these tests pin that parsing on
plan strings of each kernel family, so that a change of the string's format
cannot silently change what the line reports.  The ncu record is accepted
only for the device sources and the plan it was captured with.
"""
from __future__ import annotations

import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import json  # noqa: E402

import bench  # noqa: E402
from dense_tiled_gemm_02_gb300 import ncu_record  # noqa: E402
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
    assert ncu_record.family_of(p) == "pair"
    assert bench.kernel_name(p) == "tc_gemm_pair_kernel<256, 6, 1>"
    p = plan(bn=64, stages=8)
    assert ncu_record.family_of(p) == "cta1"
    assert bench.kernel_name(p) == "tc_gemm_kernel<64, 8, 0>"
    p = plan(decode=1, dbulk=1, bn=0, stages=0)
    assert ncu_record.family_of(p) == "decode"
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


def test_family_stems_and_native_int8_plan():
    assert ncu_record.kernel_stem(plan(pair=1)) == "tc_gemm_pair"
    assert ncu_record.kernel_stem(plan(bn=64)) == "tc_gemm"
    assert ncu_record.kernel_stem(plan(decode=1, dbulk=1)) == "decode_bulk"
    assert ncu_record.kernel_stem(plan(decode=1, dbulk=0)) == "decode_kn"
    p = plan(bn=128) + " native_i8=1"
    assert ncu_record.family_of(p) == "i8mma"
    assert bench.kernel_name(p) == "i8_mma_kernel"
    # the split-K reduce kernel is not launched when the splits of a tile add
    # their sums within a cluster
    assert bench.launches_per_step(_G(plan(splits=2) + " csk=2")) == 1
    assert bench.launches_per_step(_G(plan(splits=2) + " csk=0")) == 2


RAW = """"ID","Process ID","Kernel Name","gpu__time_duration.sum","dram__bytes_read.sum","dram__bytes_write.sum","launch__grid_size"
"","","","ns","byte","byte",""
"0","7","void tc_gemm_pair_kernel<256, 6, 1, 0>(CUtensorMap_st, KParams)","90,000","120000000","30000000","152"
"1","7","void splitk_reduce_kernel(KParams, int)","5000","1000","1000","64"
"""

LAUNCHES = """==PROF== Connected to process 1
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","p","h","void tc_gemm_pair_kernel<256, 6, 1, 0>(X)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","s","gpu__time_duration.sum","ns","90000"
"1","1","p","h","void tc_gemm_pair_kernel<256, 6, 1, 0>(X)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","s","gpu__time_duration.sum","us","90"
"2","1","p","h","void splitk_reduce_kernel(X)","1","7","(256, 1, 1)","(64, 1, 1)","0","10.3","s","gpu__time_duration.sum","ns","20000"
"""


def test_ncu_record_parsing_and_acceptance(tmp_path):
    rows = ncu_record.parse_raw_csv(RAW)
    assert len(rows) == 2 and rows[0]["gpu__time_duration.sum"] == 90000.0
    launches = ncu_record.parse_launch_list(LAUNCHES)
    assert launches[0] == {"kernel": "tc_gemm_pair_kernel<256, 6, 1, 0>", "launches": 2,
                           "total_us": 180.0, "share": 0.9}
    p = plan(pair=1)
    line = {"config": {"plan": p, "workload": "sq4096_bf16"}, "value": 1.0,
            "roofline": {"algorithmic_bytes": 134217728, "frac": 0.5}}
    rec = ncu_record.make_record(rows, launches, line, r"tc_gemm_pair")
    assert rec["dram_bytes_per_launch"] == 150000000.0
    assert rec["launches_captured"] == 1
    assert rec["source_hash"] == ncu_record.source_hash("pair")
    assert abs(rec["traffic_over_algorithmic"] - 150000000 / 134217728) < 1e-4
    # accepted only for the same plan and the same device sources
    os.makedirs(tmp_path / "profiles")
    with open(ncu_record.record_path(str(tmp_path), p, "sq4096_bf16"), "w") as f:
        json.dump(rec, f)
    assert ncu_record.load_record(str(tmp_path), p, "sq4096_bf16")["grid_size"] == 152.0
    assert ncu_record.load_record(str(tmp_path), plan(pair=1, group_m=4), "sq4096_bf16") is None
    rec["source_hash"] = "0" * 16
    with open(ncu_record.record_path(str(tmp_path), p, "sq4096_bf16"), "w") as f:
        json.dump(rec, f)
    assert ncu_record.load_record(str(tmp_path), p, "sq4096_bf16") is None


def test_also_list_defaults():
    class A:
        also, workload = "auto", bench.HEADLINE
    assert bench.also_list(A) == ["sq8192_bf16", "sq8192_i8"]
    A.workload = "rag1000_bf16"
    assert bench.also_list(A) == []
    A.also = "none"
    assert bench.also_list(A) == []
    A.also = "sq8192_i8"
    assert bench.also_list(A) == ["sq8192_i8"]


def test_cpu_matrix_small(monkeypatch):
    """The oracle's single-core and all-core timings (here on the 256^3
    workload alone): the whole GEMM when it fits, with its throughput."""
    monkeypatch.setattr(bench, "CPU_MATRIX", ("sq256_f16_f32",))
    monkeypatch.setattr(bench, "CPU_SAMPLED", ())
    out = bench.cpu_matrix({}, budget_s=30.0)
    assert [e["threads"] for e in out][0] == 1
    for e in out:
        assert e["workload"] == "sq256_f16_f32" and not e["extrapolated"]
        assert e["rows"] == 256 and e["value"] > 0


def test_aux_kernel_records_are_named_and_hashed_apart():
    """Records of the auxiliary kernels get their own file stem and are hashed
    over the auxiliary sources, so they never stand in for a GEMM record."""
    assert ncu_record.aux_stem("splitk_reduce_kernel") == "splitk_reduce"
    assert ncu_record.aux_stem("regex:copy_rows16_kernel") == "copy_rows16"
    assert ncu_record.aux_stem("copy_rows16_v_kernel") == "copy_rows16"
    assert ncu_record.aux_stem("widen_i8_x16_kernel") == "widen_i8"
    assert ncu_record.aux_stem("tc_gemm_kernel") is None
    assert ncu_record.source_hash("aux") != ncu_record.source_hash("cta1")
