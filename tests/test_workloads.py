"""CPU tests of the seeded input recipe shared by the oracle and the CUDA path
(workloads.py): what every parity test means by "the same seeded inputs".

* make_inputs is deterministic and uses seeds 1000 * idx + {0: A, 1: B, 2: C};
* uniform[-1, 1] fp16, normal(0, 1) bf16, int8 over [-128, 127] and int32 C
  over [-2^20, 2^20] inclusive, each drawn in the operand's storage order;
* sample_points / sample_rows: deterministic, in range, and the rows include
  the tile edges {0, 127, 128, M - 1} and are distinct.
"""
from __future__ import annotations

import numpy as np
import torch

from workloads import (BF16, COL, F16, I8, ROW, WORKLOADS, Workload, bits_of, draw, make_inputs,
                       sample_points, sample_rows, storage_shape)


def test_inputs_are_deterministic_and_seeded_per_operand():
    w = WORKLOADS["rag1000_bf16"]
    a, b = make_inputs(w), make_inputs(w)
    for k in "ABC":
        assert torch.equal(a[k].view(torch.int16), b[k].view(torch.int16))
    # seeds 1000 * idx + {0, 1, 2}
    assert torch.equal(a["A"], draw((w.M, w.K), w.ab_type, w.dist, 1000 * w.idx + 0))
    assert torch.equal(a["B"], draw((w.K, w.N), w.ab_type, w.dist, 1000 * w.idx + 1))
    assert torch.equal(a["C"], draw((w.M, w.N), w.c_type, w.dist, 1000 * w.idx + 2))
    c = make_inputs(w, seed_offset=1)
    assert not torch.equal(a["A"], c["A"])


def test_storage_order_of_column_major_operands():
    w = WORKLOADS["sq4096_bf16"]  # B column-major
    assert storage_shape(w.K, w.N, w.layout_b) == (w.N, w.K)
    small = Workload("t", 7, 30, 20, 10, BF16, BF16, BF16, "normal", COL, COL, COL, ROW)
    inp = make_inputs(small)
    assert tuple(inp["A"].shape) == (10, 30) and tuple(inp["B"].shape) == (20, 10)
    assert tuple(inp["C"].shape) == (20, 30)


def test_value_distributions():
    u = draw((512, 512), F16, "uniform", 11)
    assert u.dtype == torch.float16 and float(u.min()) >= -1 and float(u.max()) <= 1
    assert abs(float(u.float().mean())) < 0.01 and abs(float(u.float().var()) - 1 / 3) < 0.01
    n = draw((512, 512), BF16, "normal", 12)
    assert n.dtype == torch.bfloat16
    assert abs(float(n.float().mean())) < 0.01 and abs(float(n.float().std()) - 1) < 0.01
    i8 = draw((1024, 1024), I8, "int", 13)
    assert i8.dtype == torch.int8 and int(i8.min()) == -128 and int(i8.max()) == 127
    c = make_inputs(WORKLOADS["sq8192_i8"])["C"]
    assert c.dtype == torch.int32
    assert int(c.min()) == -(2 ** 20) and int(c.max()) == 2 ** 20  # inclusive range, both ends


def test_sampling_rule():
    M = N = 8192
    pi, pj = sample_points(M, N)
    pi2, pj2 = sample_points(M, N)
    assert torch.equal(pi, pi2) and torch.equal(pj, pj2) and pi.numel() == 65536
    assert int(pi.min()) >= 0 and int(pi.max()) < M and int(pj.min()) >= 0 and int(pj.max()) < N
    rows = sample_rows(M)
    assert torch.equal(rows, sample_rows(M)) and rows.numel() == 64
    assert len(set(rows.tolist())) == 64 and set([0, 127, 128, M - 1]) <= set(rows.tolist())
    assert int(rows.min()) >= 0 and int(rows.max()) < M
    small = sample_rows(100, n=10)
    assert set([0, 99]) <= set(small.tolist()) and len(set(small.tolist())) == 10


def test_bits_views():
    x = torch.tensor([1.0, -2.0, 0.5], dtype=torch.bfloat16)
    assert bits_of(x).dtype == np.uint16 and list(bits_of(x)) == [0x3F80, 0xC000, 0x3F00]
    f8 = torch.tensor([1.0, -2.0], dtype=torch.float8_e4m3fn)
    assert bits_of(f8).dtype == np.uint8 and list(bits_of(f8)) == [0x38, 0xC0]
