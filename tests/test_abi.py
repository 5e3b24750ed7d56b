"""The C ABI on the CPU: the library builds, loads and exports every symbol
that include/gemm.h declares; host-side validation and the grouped raster
need no GPU."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import dense_tiled_gemm_02_gb300 as pkg
from dense_tiled_gemm_02_gb300 import GemmDesc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols() -> list[str]:
    text = open(os.path.join(ROOT, "include", "gemm.h")).read()
    return re.findall(r"GEMM_API\s+[\w\s\*]+?\b(gemm_\w+)\s*\(", text)


def test_header_declares_the_python_names():
    assert sorted(declared_symbols()) == sorted(pkg.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = pkg.load()
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_strerror_codes():
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert pkg.gemm_strerror(code) != "unknown status"
    assert pkg.gemm_strerror(42) == "unknown status"


def _desc(**kw):
    d = dict(M=64, N=64, K=64, ab_type=pkg.GEMM_BF16, c_type=pkg.GEMM_BF16,
             d_type=pkg.GEMM_BF16, layout_a=0, layout_b=0, layout_c=0, layout_d=0,
             lda=0, ldb=0, ldc=0, ldd=0)
    d.update(kw)
    return GemmDesc(**d)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), pkg.GEMM_ERR_INVALID_ARG),
    (dict(K=-5), pkg.GEMM_ERR_INVALID_ARG),
    (dict(layout_a=2), pkg.GEMM_ERR_INVALID_ARG),
    (dict(lda=10), pkg.GEMM_ERR_INVALID_ARG),           # row-major A needs lda >= K
    (dict(layout_b=1, ldb=63), pkg.GEMM_ERR_INVALID_ARG),
    (dict(ab_type=pkg.GEMM_F32), pkg.GEMM_ERR_UNSUPPORTED),
    (dict(ab_type=pkg.GEMM_I8), pkg.GEMM_ERR_UNSUPPORTED),  # int8 needs int32 D
    (dict(d_type=pkg.GEMM_I32), pkg.GEMM_ERR_UNSUPPORTED),
    (dict(ab_type=pkg.GEMM_I8, c_type=pkg.GEMM_BF16, d_type=pkg.GEMM_I32),
     pkg.GEMM_ERR_UNSUPPORTED),
])
def test_create_rejects_bad_descriptions(kw, code):
    rc, h = pkg.gemm_create(_desc(**kw))
    assert rc == code and h is None


def test_create_without_gpu_reports_no_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = pkg.gemm_create(_desc())
    assert rc == pkg.GEMM_ERR_NO_DEVICE and h is None


def test_null_handles():
    lib = pkg.load()
    assert lib.gemm_destroy(None) == 0
    assert lib.gemm_run(None, None, None, None, None, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_get_status(None, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_plan_string(None, None, 0) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_workspace_bytes(None) == -1
    assert lib.gemm_create(None, None) == pkg.GEMM_ERR_INVALID_ARG


# ------------------------------------------------------------------ grouped raster
@pytest.mark.parametrize("npm,npn,g", [(1, 1, 1), (5, 3, 2), (32, 16, 8), (7, 9, 4), (3, 11, 8),
                                       (16, 1, 8), (1, 16, 8), (64, 64, 1)])
def test_raster_is_a_bijection_with_grouped_columns(npm, npn, g):
    seen = set()
    order = []
    for t in range(npm * npn):
        rc, pm, pn = pkg.gemm_raster_tile(t, npm, npn, g)
        assert rc == 0 and 0 <= pm < npm and 0 <= pn < npn
        seen.add((pm, pn))
        order.append((pm, pn))
    assert len(seen) == npm * npn
    # Within one group, consecutive tiles walk down the group's tile rows
    # first, so each column of B is used by up to GROUP_M tiles in a row.
    for start in range(0, npm * npn, g * npn):
        grp = order[start:start + g * npn]
        rows = {pm for pm, _ in grp}
        size = len(rows)
        assert size == min(g, npm - start // npn)
        for i in range(0, len(grp), size):
            cols = {pn for _, pn in grp[i:i + size]}
            assert len(cols) == 1


def test_raster_rejects_out_of_range():
    assert pkg.gemm_raster_tile(6, 2, 3, 2)[0] == pkg.GEMM_ERR_INVALID_ARG
    assert pkg.gemm_raster_tile(-1, 2, 3, 2)[0] == pkg.GEMM_ERR_INVALID_ARG
    assert pkg.gemm_raster_tile(0, 2, 3, 0)[0] == pkg.GEMM_ERR_INVALID_ARG
