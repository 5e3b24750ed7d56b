"""The split-K entry point that allocates no device memory.

Callers that cannot allocate at the point of use (code under a framework
whose caching allocator owns all device memory, latency-critical paths that
cannot take cudaMalloc or cudaFree's device-wide synchronisation) call
gemm_run_splitk_noalloc, whose scratch is a static device array shared by
all calls.  These tests call it through the C ABI twice in a row, on
different inputs so that the second call starts from the first call's
leftovers, and check each result against the handle-based entry point
(gemm_create + gemm_run with the same split) and against the oracle, with
the acceptance rule used everywhere else.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import dense_tiled_gemm_02_gb300 as pkg
import oracle
from gpu_helpers import check_rows, forced_plan, logical
from oracle import compare
from workloads import BF16, COL, F16, F32, ROW, TORCH_DTYPE, Workload, make_inputs, storage_shape

pytestmark = pytest.mark.gpu

CASES = [
    # workload, splits
    (Workload("noalloc_a", 61, 1000, 384, 4096, BF16, BF16, BF16, "normal", ROW, COL, ROW, ROW), 4),
    # column-major A: its leading dimension M = 336 keeps rows 16-byte aligned (no repack here)
    (Workload("noalloc_b", 62, 336, 200, 2500, F16, F32, F32, "normal", COL, ROW, ROW, COL), 3),
    # N <= 64: the 128 x 64 tile
    (Workload("noalloc_c", 63, 520, 48, 1024, BF16, BF16, BF16, "normal", ROW, COL, ROW, ROW), 3),
    # N <= 128: the 128 x 128 tile; D rows of 100 bf16 are not 16-byte aligned
    (Workload("noalloc_d", 64, 400, 100, 768, BF16, BF16, BF16, "normal", ROW, COL, ROW, ROW), 2),
    # no split: the kernel writes D itself and the partial-sum area is unused
    (Workload("noalloc_e", 65, 300, 264, 640, F16, F16, F16, "normal", ROW, ROW, ROW, ROW), 1),
]


def _tensors(w, inp, dev):
    A = logical(inp["A"].to(dev), w.layout_a)
    B = logical(inp["B"].to(dev), w.layout_b)
    C = None if inp["C"] is None else logical(inp["C"].to(dev), w.layout_c)
    Ds = torch.zeros(storage_shape(w.M, w.N, w.layout_d), dtype=TORCH_DTYPE[w.d_type], device=dev)
    return A, B, C, Ds


def _desc(w, A, B, C, D):
    la, lda = pkg.layout_of(A)
    lb, ldb = pkg.layout_of(B)
    ld_, ldd = pkg.layout_of(D)
    lc, ldc = pkg.layout_of(C) if C is not None else (ROW, 0)
    return pkg.GemmDesc(w.M, w.N, w.K, w.ab_type, w.c_type or 0, w.d_type, la, lb, lc, ld_,
                        lda, ldb, ldc, ldd)


def _values(w, Ds):
    return logical(Ds, w.layout_d).double().cpu().numpy()


@pytest.mark.parametrize("case", range(len(CASES)))
def test_noalloc_matches_handle_entry_two_calls_in_a_row(case):
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    pkg.load()
    w, splits = CASES[case]
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    orc = oracle.get()
    for call in range(2):
        inp = make_inputs(w, seed_offset=100 * call)
        A, B, C, Dn = _tensors(w, inp, dev)
        rc = pkg.gemm_run_splitk_noalloc(_desc(w, A, B, C, logical(Dn, w.layout_d)), splits,
                                         A.data_ptr(), B.data_ptr(),
                                         None if C is None else C.data_ptr(), Dn.data_ptr(),
                                         stream.cuda_stream)
        assert rc == pkg.GEMM_OK, pkg.gemm_strerror(rc)
        # its status word, read back without allocating
        assert pkg.gemm_noalloc_status(stream.cuda_stream) == pkg.GEMM_OK
        # the handle-based entry point, same split of K
        _, _, _, Do = _tensors(w, inp, dev)
        with forced_plan(f"splits={splits},swap=0"):
            g = pkg.Gemm.like(A, B, C, logical(Do, w.layout_d))
        g.run(A, B, C, logical(Do, w.layout_d), stream)
        assert g.status(stream) == pkg.GEMM_OK
        g.close()
        torch.cuda.synchronize()
        new, old = _values(w, Dn), _values(w, Do)
        # same acceptance rule, with the handle entry's output as the reference
        _, S = orc.gemm_f64_rows(
            w.M, w.N, w.K, *_oracle_inputs(w, inp), ab_type=w.ab_type, c_type=w.c_type or 0,
            a_col=w.layout_a, b_col=w.layout_b, c_col=w.layout_c)
        c_abs = np.abs(logical(inp["C"], w.layout_c).double().numpy())
        rep_vs_old = compare.check_float(orc, new, old, S, c_abs, w.d_type)
        assert rep_vs_old["ok"], f"call {call}: differs from gemm_run: {rep_vs_old}"
        rep = check_rows(w, inp, Dn.cpu())
        assert rep["ok"], f"call {call}: outside the oracle tolerance: {rep}"


def _oracle_inputs(w, inp):
    from workloads import bits_u16
    A = bits_u16(inp["A"])
    B = bits_u16(inp["B"])
    C = inp["C"].numpy() if w.c_type == F32 else bits_u16(inp["C"])
    return A, B, C


def test_noalloc_rejects_partials_beyond_the_scratch():
    pkg.load()
    M = N = 2048  # 2 splits * 2048 * 2048 * 4 bytes = 32 MiB > 16 MiB
    A = torch.zeros(M, 256, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(256, N, dtype=torch.bfloat16, device="cuda")
    D = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    desc = pkg.GemmDesc(M, N, 256, BF16, 0, BF16, ROW, ROW, ROW, ROW, 0, 0, 0, 0)
    rc = pkg.gemm_run_splitk_noalloc(desc, 2, A.data_ptr(), B.data_ptr(), None, D.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == pkg.GEMM_ERR_INVALID_ARG


def test_noalloc_rejects_rows_the_tma_cannot_read():
    """A column-major A with a 666-byte leading dimension is not read in place."""
    pkg.load()
    M, N, K = 333, 200, 256
    A = torch.zeros(K, M, dtype=torch.float16, device="cuda").t()
    B = torch.zeros(K, N, dtype=torch.float16, device="cuda")
    D = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    desc = pkg.GemmDesc(M, N, K, F16, 0, F32, COL, ROW, ROW, ROW, M, N, 0, N)
    rc = pkg.gemm_run_splitk_noalloc(desc, 2, A.data_ptr(), B.data_ptr(), None, D.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == pkg.GEMM_ERR_MISALIGNED
