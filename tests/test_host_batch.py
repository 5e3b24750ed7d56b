"""GPU: the host-buffer entry points (gemm_host_io_enable, gemm_run_host_batch).

Operands start and end in page-locked host memory; the library copies them
in, runs the same plan as gemm_run, and copies D back, with the copies of
consecutive products overlapping.  Each D[i] must equal, bit for bit, what
gemm_run gives on device copies of the same operands with the same handle,
and one of them is also checked against the oracle.
"""
from __future__ import annotations

import pytest
import torch

import dense_tiled_gemm_02_gb300 as pkg
from gpu_helpers import check_rows, logical
from workloads import TORCH_DTYPE, WORKLOADS, make_inputs, sample_rows, storage_shape

pytestmark = pytest.mark.gpu


def _plan_and_device_refs(w, inputs, dev):
    """A handle for w's description and gemm_run's D for each input set."""
    refs = []
    g = None
    for inp in inputs:
        A = logical(inp["A"].to(dev), w.layout_a)
        B = logical(inp["B"].to(dev), w.layout_b)
        C = None if inp["C"] is None else logical(inp["C"].to(dev), w.layout_c)
        Ds = torch.zeros(storage_shape(w.M, w.N, w.layout_d), dtype=TORCH_DTYPE[w.d_type],
                         device=dev)
        D = logical(Ds, w.layout_d)
        if g is None:
            g = pkg.Gemm.like(A, B, C, D)
        g.run(A, B, C, D)
        assert g.status(torch.cuda.current_stream()) == pkg.GEMM_OK
        refs.append(Ds.cpu())
    return g, refs


@pytest.mark.parametrize("name,n", [("sq4096_bf16", 3), ("rag1000_bf16", 5),
                                    ("sq1024_f16", 4), ("skinny8192x128x4096_bf16", 3)])
def test_host_batch_matches_device_run(name, n):
    w = WORKLOADS[name]
    dev = torch.device("cuda")
    inputs = [make_inputs(w, seed_offset=i) for i in range(n)]
    g, refs = _plan_and_device_refs(w, inputs, dev)
    try:
        g.host_io_enable()
        g.host_io_enable()  # a second call is a no-op
        pin = lambda t: None if t is None else t.contiguous().pin_memory()
        As = [pin(inp["A"]) for inp in inputs]
        Bs = [pin(inp["B"]) for inp in inputs]
        Cs = None if w.c_type is None else [pin(inp["C"]) for inp in inputs]
        shape = storage_shape(w.M, w.N, w.layout_d)
        Ds = [torch.full(shape, 7, dtype=TORCH_DTYPE[w.d_type]).pin_memory() for _ in range(n)]
        s = torch.cuda.Stream()
        # two calls on one handle: the device sets alternate across calls too
        g.run_host_batch(As[:2], Bs[:2], None if Cs is None else Cs[:2], Ds[:2], s)
        g.run_host_batch(As[2:], Bs[2:], None if Cs is None else Cs[2:], Ds[2:], s)
        assert g.status(s) == pkg.GEMM_OK
        for i in range(n):
            assert torch.equal(Ds[i].view(torch.uint8), refs[i].view(torch.uint8)), f"product {i}"
        rows = sample_rows(w.M, n=16)
        rep = check_rows(w, inputs[-1], Ds[-1], rows=rows)
        assert rep["ok"], rep["first_failures"]
    finally:
        g.close()


def test_host_batch_without_c_and_argument_errors():
    w = WORKLOADS["rag1000_bf16"]
    dev = torch.device("cuda")
    inp = make_inputs(w)
    inp_noc = dict(inp, C=None)
    g, refs = _plan_and_device_refs(w, [inp_noc], dev)
    try:
        A = inp["A"].contiguous().pin_memory()
        B = inp["B"].contiguous().pin_memory()
        D = torch.empty(storage_shape(w.M, w.N, w.layout_d), dtype=TORCH_DTYPE[w.d_type])
        # not enabled yet
        assert pkg.gemm_run_host_batch(g.handle, [A.data_ptr()], [B.data_ptr()], None,
                                       [D.data_ptr()], None) == pkg.GEMM_ERR_INVALID_ARG
        g.host_io_enable()
        # a null operand is refused before anything is enqueued
        assert pkg.gemm_run_host_batch(g.handle, [A.data_ptr()], [None], None,
                                       [D.data_ptr()], None) == pkg.GEMM_ERR_INVALID_ARG
        # pageable D, a C list whose entry is None (C = 0), and an empty batch
        g.run_host_batch([A], [B], [None], [D])
        g.run_host_batch([], [], None, [])
        assert g.status(torch.cuda.current_stream()) == pkg.GEMM_OK
        assert torch.equal(D.view(torch.uint8), refs[0].view(torch.uint8))
    finally:
        g.close()
