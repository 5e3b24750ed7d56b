"""Figures the pages print, checked against this repository's conventions."""
from __future__ import annotations

import json
import os

from workloads import F16, WORKLOADS

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "pages_figures.json")


def figures():
    with open(GOLDEN) as f:
        return json.load(f)


def stage_bytes(block_m: int, block_n: int, block_k: int, elem_bytes: int = 2) -> int:
    """Input bytes of one A/B tile pair, the pages' formula."""
    return (block_m + block_n) * block_k * elem_bytes


def test_tile_pair_bytes_formula():
    g = figures()["tile_pair_bytes"]
    assert stage_bytes(g["BLOCK_M"], g["BLOCK_N"], g["BLOCK_K"]) == g["bytes"]
    # the same formula sizes the library's rings: 128 x 256 x 64 tiles, 4 stages
    assert 4 * stage_bytes(128, 256, 64) == 196608 <= 227 * 1024


def test_square_fp16_workload_is_the_slide_example():
    g = figures()["triton_matmul_example"]
    w = WORKLOADS["sq1024_f16"]
    assert (w.M, w.N, w.K) == (g["M"], g["N"], g["K"])
    assert w.ab_type == F16 and w.d_type == F16 and w.c_type is None


def test_key_experiment_throughput_conversion():
    g = figures()["key_experiment_gfx942"]
    M, N, K = g["shape"]
    tflops = 2 * M * N * K / (g["time_us"] * 1e-6) / 1e12
    assert abs(tflops - 393.9) < 0.1
