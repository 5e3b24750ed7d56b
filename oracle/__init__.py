"""CPU oracle for D = A*B + C (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does: the CUDA
library in ``dense_tiled_gemm_02_gb300`` shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64 / int64 triple loop,
OpenMP over rows).  This module compiles it on first use with the host C
compiler and exposes it through ctypes over numpy arrays:

* ``gemm_f64_rows`` / ``gemm_f64_points``: fp16/bf16 operands, the sum in fp64,
  plus the sum of absolute products used by the error bound.
* ``gemm_mx_rows``: the block-scaled form of the 8-bit float product (one
  E8M0 power-of-two scale per 32 K elements of each row of A and column of B).
* ``gemm_i64_rows`` / ``gemm_i64_points``: int8 operands, int32 C, int64 sum.
* ``round_bits`` / ``widen_bits``: one correct round-to-nearest-even from fp64
  to fp16/bf16, and the exact inverse widening; ``widen_bits8`` the exact
  widening of the 8-bit float encodings.

Type codes: 1 fp16, 2 bf16, 3 fp32, 4 int8, 5 int32, 6 E4M3, 7 E5M2 (OCP
OFP8).  Layout flags: 0 row-major, 1 column-major.  fp16/bf16 arrays are
passed as their uint16 bit patterns, E4M3/E5M2 arrays as uint8 patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

F16, BF16, F32, I8, I32, E4M3, E5M2 = 1, 2, 3, 4, 5, 6, 7
ROW, COL = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_i64 = ctypes.c_int64
_int = ctypes.c_int
_vp = ctypes.c_void_p


def compile_library(out_path: str = _LIB, mutant: int = 0) -> str:
    """Compile oracle.c into a shared library at ``out_path`` (atomically)."""
    cc = os.environ.get("CC", "cc")
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out_path) or ".")
    os.close(fd)
    cmd = [cc, "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
           f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, out_path)
    except subprocess.CalledProcessError as e:
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed: {' '.join(cmd)}\n{e.stderr}") from e
    return out_path


def _loadable(path: str) -> bool:
    if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        return False
    try:
        ctypes.CDLL(path)
        return True
    except OSError:  # e.g. a library compiled for another architecture
        return False


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_vp)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        self.path = path
        self._lib = lib
        lib.oracle_widen.argtypes = [_vp, _i64, _int, _vp]
        lib.oracle_widen8.argtypes = [_vp, _i64, _int, _vp]
        lib.oracle_round.argtypes = [_vp, _i64, _int, _vp]
        lib.oracle_threads.argtypes = []
        lib.oracle_set_threads.argtypes = [_int]
        lib.oracle_gemm_f64_rows.argtypes = [_i64, _i64, _i64, _int, _int, _int, _int, _int,
                                             _i64, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _vp, _vp]
        lib.oracle_gemm_f64_points.argtypes = [_i64, _i64, _i64, _int, _int, _int, _int, _int,
                                               _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _i64,
                                               _vp, _vp]
        lib.oracle_gemm_mx_rows.argtypes = [_i64, _i64, _i64, _int, _int, _int, _int, _int,
                                            _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp,
                                            _i64, _vp, _vp]
        lib.oracle_gemm_i64_rows.argtypes = [_i64, _i64, _i64, _int, _int, _int,
                                             _i64, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _vp]
        lib.oracle_gemm_i64_points.argtypes = [_i64, _i64, _i64, _int, _int, _int,
                                               _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _i64,
                                               _vp]

    # -- rounding -----------------------------------------------------------
    def round_bits(self, x, t: int) -> np.ndarray:
        """fp64 array -> uint16 encodings of fp16 (t=1) or bf16 (t=2), RNE."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        if self._lib.oracle_round(_ptr(x), x.size, t, _ptr(out)) != 0:
            raise ValueError("bad type")
        return out

    def widen_bits(self, bits, t: int) -> np.ndarray:
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(bits.shape, dtype=np.float64)
        if self._lib.oracle_widen(_ptr(bits), bits.size, t, _ptr(out)) != 0:
            raise ValueError("bad type")
        return out

    def widen_bits8(self, bits, t: int) -> np.ndarray:
        bits = np.ascontiguousarray(bits, dtype=np.uint8)
        out = np.empty(bits.shape, dtype=np.float64)
        if self._lib.oracle_widen8(_ptr(bits), bits.size, t, _ptr(out)) != 0:
            raise ValueError("bad type")
        return out

    def threads(self) -> int:
        return int(self._lib.oracle_threads())

    def set_threads(self, n: int) -> int:
        """Threads of the parallel loops (for timing on one core or all)."""
        return int(self._lib.oracle_set_threads(int(n)))

    # -- floating point -------------------------------------------------------
    def gemm_f64_rows(self, M, N, K, A, B, C, *, ab_type, c_type=BF16, a_col=0, b_col=0,
                      c_col=0, lda=None, ldb=None, ldc=None, rows=None, want_s=True):
        """D (and S = sum |a*b|) for the listed rows (all rows when None)."""
        lda = lda if lda is not None else (M if a_col else K)
        ldb = ldb if ldb is not None else (K if b_col else N)
        ldc = ldc if ldc is not None else (M if c_col else N)
        rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        nr = M if rows_a is None else rows_a.size
        D = np.empty((nr, N), dtype=np.float64)
        S = np.empty((nr, N), dtype=np.float64) if want_s else None
        A = np.ascontiguousarray(A)
        B = np.ascontiguousarray(B)
        C = None if C is None else np.ascontiguousarray(C)
        rc = self._lib.oracle_gemm_f64_rows(M, N, K, ab_type, c_type, a_col, b_col, c_col,
                                            lda, ldb, ldc, _ptr(A), _ptr(B), _ptr(C),
                                            _ptr(rows_a), nr, _ptr(D), _ptr(S))
        if rc != 0:
            raise ValueError(f"oracle_gemm_f64_rows failed ({rc})")
        return D, S

    def gemm_mx_rows(self, M, N, K, A, B, C, SA, SB, *, ab_type, c_type=BF16, a_col=0,
                     b_col=0, c_col=0, lda=None, ldb=None, ldc=None, rows=None):
        """Block-scaled 8-bit float product: D (and S = sum |scaled a * scaled b|)
        for the listed rows.  SA is M x ceil(K/32), SB is N x ceil(K/32), both
        uint8 E8M0 exponents (scale 2^(e-127)) of 32-element K blocks."""
        lda = lda if lda is not None else (M if a_col else K)
        ldb = ldb if ldb is not None else (K if b_col else N)
        ldc = ldc if ldc is not None else (M if c_col else N)
        nb = (K + 31) // 32
        SA = np.ascontiguousarray(SA, dtype=np.uint8)
        SB = np.ascontiguousarray(SB, dtype=np.uint8)
        if SA.shape != (M, nb) or SB.shape != (N, nb):
            raise ValueError(f"scale shapes {SA.shape}, {SB.shape}; want {(M, nb)}, {(N, nb)}")
        rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        nr = M if rows_a is None else rows_a.size
        D = np.empty((nr, N), dtype=np.float64)
        S = np.empty((nr, N), dtype=np.float64)
        A = np.ascontiguousarray(A)
        B = np.ascontiguousarray(B)
        C = None if C is None else np.ascontiguousarray(C)
        rc = self._lib.oracle_gemm_mx_rows(M, N, K, ab_type, c_type, a_col, b_col, c_col,
                                           lda, ldb, ldc, _ptr(A), _ptr(B), _ptr(C), _ptr(SA),
                                           _ptr(SB), _ptr(rows_a), nr, _ptr(D), _ptr(S))
        if rc != 0:
            raise ValueError(f"oracle_gemm_mx_rows failed ({rc})")
        return D, S

    def gemm_f64_points(self, M, N, K, A, B, C, pi, pj, *, ab_type, c_type=BF16, a_col=0,
                        b_col=0, c_col=0, lda=None, ldb=None, ldc=None):
        lda = lda if lda is not None else (M if a_col else K)
        ldb = ldb if ldb is not None else (K if b_col else N)
        ldc = ldc if ldc is not None else (M if c_col else N)
        pi = np.ascontiguousarray(pi, dtype=np.int64)
        pj = np.ascontiguousarray(pj, dtype=np.int64)
        D = np.empty(pi.size, dtype=np.float64)
        S = np.empty(pi.size, dtype=np.float64)
        A = np.ascontiguousarray(A)
        B = np.ascontiguousarray(B)
        C = None if C is None else np.ascontiguousarray(C)
        rc = self._lib.oracle_gemm_f64_points(M, N, K, ab_type, c_type, a_col, b_col, c_col,
                                              lda, ldb, ldc, _ptr(A), _ptr(B), _ptr(C),
                                              _ptr(pi), _ptr(pj), pi.size, _ptr(D), _ptr(S))
        if rc != 0:
            raise ValueError(f"oracle_gemm_f64_points failed ({rc})")
        return D, S

    # -- integer ----------------------------------------------------------------
    def gemm_i64_rows(self, M, N, K, A, B, C, *, a_col=0, b_col=0, c_col=0, lda=None,
                      ldb=None, ldc=None, rows=None):
        lda = lda if lda is not None else (M if a_col else K)
        ldb = ldb if ldb is not None else (K if b_col else N)
        ldc = ldc if ldc is not None else (M if c_col else N)
        rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        nr = M if rows_a is None else rows_a.size
        D = np.empty((nr, N), dtype=np.int64)
        A = np.ascontiguousarray(A, dtype=np.int8)
        B = np.ascontiguousarray(B, dtype=np.int8)
        C = None if C is None else np.ascontiguousarray(C, dtype=np.int32)
        rc = self._lib.oracle_gemm_i64_rows(M, N, K, a_col, b_col, c_col, lda, ldb, ldc,
                                            _ptr(A), _ptr(B), _ptr(C), _ptr(rows_a), nr,
                                            _ptr(D))
        if rc != 0:
            raise ValueError(f"oracle_gemm_i64_rows failed ({rc})")
        return D

    def gemm_i64_points(self, M, N, K, A, B, C, pi, pj, *, a_col=0, b_col=0, c_col=0,
                        lda=None, ldb=None, ldc=None):
        lda = lda if lda is not None else (M if a_col else K)
        ldb = ldb if ldb is not None else (K if b_col else N)
        ldc = ldc if ldc is not None else (M if c_col else N)
        pi = np.ascontiguousarray(pi, dtype=np.int64)
        pj = np.ascontiguousarray(pj, dtype=np.int64)
        D = np.empty(pi.size, dtype=np.int64)
        A = np.ascontiguousarray(A, dtype=np.int8)
        B = np.ascontiguousarray(B, dtype=np.int8)
        C = None if C is None else np.ascontiguousarray(C, dtype=np.int32)
        rc = self._lib.oracle_gemm_i64_points(M, N, K, a_col, b_col, c_col, lda, ldb, ldc,
                                              _ptr(A), _ptr(B), _ptr(C), _ptr(pi), _ptr(pj),
                                              pi.size, _ptr(D))
        if rc != 0:
            raise ValueError(f"oracle_gemm_i64_points failed ({rc})")
        return D


_default: Oracle | None = None


def get() -> Oracle:
    """The default oracle library, compiled on first use when missing or stale."""
    global _default
    if _default is None:
        if not _loadable(_LIB):
            compile_library(_LIB)
        _default = Oracle(_LIB)
    return _default


def build() -> str:
    """Compile the oracle library (used by the package build step)."""
    if not _loadable(_LIB):
        compile_library(_LIB)
    return _LIB
