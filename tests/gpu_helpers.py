"""Helpers shared by the GPU parity tests: run the library, ask the oracle."""
from __future__ import annotations

import os
from contextlib import contextmanager

import numpy as np
import torch

import oracle
from oracle import compare
from workloads import F32, I8, I32, ROW, TORCH_DTYPE, Workload, bits_of, bits_u16, storage_shape

TYPE_TORCH = TORCH_DTYPE


def logical(storage: torch.Tensor, layout: int) -> torch.Tensor:
    """Logical (rows x cols) view of an operand stored densely in `layout`."""
    return storage if layout == ROW else storage.t()


@contextmanager
def forced_plan(spec: str | None):
    old = os.environ.get("GEMM_FORCE_PLAN")
    if spec:
        os.environ["GEMM_FORCE_PLAN"] = spec
    try:
        yield
    finally:
        if old is None:
            os.environ.pop("GEMM_FORCE_PLAN", None)
        else:
            os.environ["GEMM_FORCE_PLAN"] = old


def run_gpu(w: Workload, inp: dict, plan: str | None = None, stream=None, D_storage=None):
    """D (host tensor in D's storage order) and the plan string."""
    import dense_tiled_gemm_02_gb300 as pkg
    dev = torch.device("cuda")
    A = logical(inp["A"].to(dev), w.layout_a)
    B = logical(inp["B"].to(dev), w.layout_b)
    C = None if inp["C"] is None else logical(inp["C"].to(dev), w.layout_c)
    if D_storage is None:
        D_storage = torch.full(storage_shape(w.M, w.N, w.layout_d), 0, dtype=TYPE_TORCH[w.d_type],
                               device=dev)
    D = logical(D_storage, w.layout_d)
    with forced_plan(plan):
        g = pkg.Gemm.like(A, B, C, D)
    try:
        g.run(A, B, C, D, stream)
        st = g.status(stream)
        assert st == pkg.GEMM_OK, pkg.gemm_strerror(st)
        return D_storage.cpu(), g.plan()
    finally:
        g.close()


def _oracle_args(w: Workload, inp: dict):
    if w.ab_type == I8:
        A = inp["A"].numpy()
        B = inp["B"].numpy()
        C = None if inp["C"] is None else inp["C"].numpy()
    else:
        A = bits_of(inp["A"])
        B = bits_of(inp["B"])
        C = None
        if inp["C"] is not None:
            C = inp["C"].numpy() if w.c_type == F32 else bits_u16(inp["C"])
    return A, B, C


def d_values(w: Workload, D_storage: torch.Tensor) -> np.ndarray:
    """Logical M x N values of D (fp64 for floats, int64 for int32)."""
    D = logical(D_storage, w.layout_d)
    if w.d_type == I32:
        return D.long().numpy()
    return D.double().numpy()


def c_abs(w: Workload, inp: dict, rows=None) -> np.ndarray:
    if inp["C"] is None:
        shape = (w.M if rows is None else len(rows), w.N)
        return np.zeros(shape)
    C = logical(inp["C"], w.layout_c).double().abs().numpy()
    return C if rows is None else C[np.asarray(rows)]


def check_rows(w: Workload, inp: dict, D_storage: torch.Tensor, rows=None) -> dict:
    """Compare whole rows (all rows when None) of D with the oracle."""
    orc = oracle.get()
    A, B, C = _oracle_args(w, inp)
    Dv = d_values(w, D_storage)
    if rows is not None:
        Dv = Dv[np.asarray(rows)]
    kw = dict(a_col=w.layout_a, b_col=w.layout_b, c_col=w.layout_c, rows=rows)
    if w.ab_type == I8:
        D_ref = orc.gemm_i64_rows(w.M, w.N, w.K, A, B, C, **kw)
        return compare.check_int(Dv, D_ref)
    D_ref, S = orc.gemm_f64_rows(w.M, w.N, w.K, A, B, C, ab_type=w.ab_type,
                                 c_type=w.c_type or 0, **kw)
    return compare.check_float(orc, Dv, D_ref, S, c_abs(w, inp, rows), w.d_type)


def check_points(w: Workload, inp: dict, D_storage: torch.Tensor, pi, pj) -> dict:
    orc = oracle.get()
    A, B, C = _oracle_args(w, inp)
    pi = np.asarray(pi)
    pj = np.asarray(pj)
    Dv = d_values(w, D_storage)[pi, pj]
    kw = dict(a_col=w.layout_a, b_col=w.layout_b, c_col=w.layout_c)
    if w.ab_type == I8:
        D_ref = orc.gemm_i64_points(w.M, w.N, w.K, A, B, C, pi, pj, **kw)
        return compare.check_int(Dv, D_ref)
    D_ref, S = orc.gemm_f64_points(w.M, w.N, w.K, A, B, C, pi, pj, ab_type=w.ab_type,
                                   c_type=w.c_type or 0, **kw)
    Cabs = c_abs(w, inp)[pi, pj] if inp["C"] is not None else np.zeros(pi.size)
    return compare.check_float(orc, Dv, D_ref, S, Cabs, w.d_type)


def run_gpu_mx(w: Workload, inp: dict, sc: dict, plan: str | None = None):
    """D (host, D's storage order) and the plan of a block-scaled run: A and B
    hold E4M3 / E5M2 values, sc["SA"] / sc["SB"] their E8M0 block scales."""
    import dense_tiled_gemm_02_gb300 as pkg
    dev = torch.device("cuda")
    A = logical(inp["A"].to(dev), w.layout_a)
    B = logical(inp["B"].to(dev), w.layout_b)
    C = None if inp["C"] is None else logical(inp["C"].to(dev), w.layout_c)
    D_storage = torch.zeros(storage_shape(w.M, w.N, w.layout_d), dtype=TYPE_TORCH[w.d_type],
                            device=dev)
    D = logical(D_storage, w.layout_d)
    SA, SB = sc["SA"].to(dev), sc["SB"].to(dev)
    with forced_plan(plan):
        g = pkg.Gemm.like(A, B, C, D, mx=True)
    try:
        g.run_mx(A, SA, B, SB, C, D)
        st = g.status()
        assert st == pkg.GEMM_OK, pkg.gemm_strerror(st)
        return D_storage.cpu(), g.plan()
    finally:
        g.close()


def check_rows_mx(w: Workload, inp: dict, sc: dict, D_storage: torch.Tensor, rows=None) -> dict:
    """Compare whole rows of a block-scaled D with the oracle's block-scaled product."""
    orc = oracle.get()
    A, B, C = _oracle_args(w, inp)
    Dv = d_values(w, D_storage)
    if rows is not None:
        Dv = Dv[np.asarray(rows)]
    D_ref, S = orc.gemm_mx_rows(w.M, w.N, w.K, A, B, C, sc["SA"].numpy(), sc["SB"].numpy(),
                                ab_type=w.ab_type, c_type=w.c_type or 0, a_col=w.layout_a,
                                b_col=w.layout_b, c_col=w.layout_c, rows=rows)
    return compare.check_float(orc, Dv, D_ref, S, c_abs(w, inp, rows), w.d_type,
                               s_rel=compare.mx_s_rel(w.K))
