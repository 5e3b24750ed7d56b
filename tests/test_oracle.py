"""Pins of the CPU oracle against things other than itself (CPU only).

Each ``pin_*`` function raises AssertionError on a mismatch.  The tests run
them on the oracle; ``test_pins_catch_planted_mistakes`` builds the oracle
with one planted mistake at a time (``-DORACLE_MUTANT=n``) and checks that at
least one pin fails for every mistake.

What pins what:
* widening: the standard library's / numpy's IEEE binary16 and binary32
  decoders, over all 65536 encodings; torch's float8 dtypes over all 256
  E4M3 and E5M2 encodings, and the OFP8 specification's named values;
* rounding: every midpoint between neighbouring fp16/bf16 values (ties to
  even) and one double either side, numpy's float64->float16 conversion,
  torch's float32->bfloat16 conversion, and an exact rational search;
* the GEMM: an exact rational evaluation of the definition on every shape in
  {1,2,3}^3 and every layout, closed forms (identity, permutation, rank-1,
  all-ones, linearity), and torch's CPU int64 matmul for int8; for the
  8-bit float types, the exact rational evaluation on tiny shapes and the
  identity and all-ones closed forms; for their block-scaled form, the
  unscaled product at unit scales, the exact rational value of the
  microscaling definition, power-of-two scaling of a row or column, and NaN
  scales.
"""
from __future__ import annotations

import itertools
import os
import random
import tempfile
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact_ref
import oracle
from oracle import BF16, E4M3, E5M2, F16, F32

INF_BITS = {F16: 0x7C00, BF16: 0x7F80}
EMAX1 = {F16: 16, BF16: 128}


def to_storage(X: np.ndarray, col: int) -> np.ndarray:
    return np.ascontiguousarray(X.T if col else X)


def f16_bits(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16_bits_exact(x: np.ndarray) -> np.ndarray:
    """bf16 encodings of values that are exactly representable in bf16."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)
    return (b >> 16).astype(np.uint16)


def bits_of(x, t):
    return f16_bits(x) if t == F16 else bf16_bits_exact(x)


# ----------------------------------------------------------------------------- widening
def pin_widen_exhaustive(orc):
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref16 = allb.view(np.float16).astype(np.float64)
    with np.errstate(invalid="ignore"):
        refbf = (allb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t, ref in ((F16, ref16), (BF16, refbf)):
        got = orc.widen_bits(allb, t)
        same = (got == ref) | (np.isnan(got) & np.isnan(ref))
        assert same.all(), f"widen type {t}: first bad encoding {np.argmax(~same):#06x}"


# 8-bit floats (OCP OFP8): torch's float8 dtypes decode every encoding, and
# the specification's named values are checked by their closed forms.
FP8_TORCH = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def fp8_bits(x, t) -> np.ndarray:
    """Encodings of values exactly representable in the 8-bit type t."""
    xt = torch.as_tensor(np.asarray(x, dtype=np.float32))
    b = xt.to(FP8_TORCH[t])
    assert torch.equal(b.float(), xt), "value not representable"
    return b.view(torch.uint8).numpy()


def pin_widen_fp8(orc):
    allb = np.arange(256, dtype=np.uint8)
    for t, dt in FP8_TORCH.items():
        ref = torch.from_numpy(allb).view(dt).to(torch.float64).numpy()
        got = orc.widen_bits8(allb, t)
        same = (got == ref) | (np.isnan(got) & np.isnan(ref))
        assert same.all(), f"widen type {t}: first bad encoding {np.argmax(~same):#04x}"
    e4 = orc.widen_bits8(np.array([0x7E, 0x7F, 0xFE, 0x01, 0x08, 0x38, 0x78], np.uint8), E4M3)
    assert e4[0] == 448.0 and np.isnan(e4[1]) and e4[2] == -448.0
    assert e4[3] == 2.0 ** -9 and e4[4] == 2.0 ** -6 and e4[5] == 1.0 and e4[6] == 256.0
    e5 = orc.widen_bits8(np.array([0x7B, 0x7C, 0x7D, 0x01, 0x04, 0x3C], np.uint8), E5M2)
    assert e5[0] == 57344.0 and e5[1] == np.inf and np.isnan(e5[2])
    assert e5[3] == 2.0 ** -16 and e5[4] == 2.0 ** -14 and e5[5] == 1.0


def _rand_fp8(rng, shape, t):
    """Random finite encodings of t (normal and subnormal alike) and their
    values as decoded by torch."""
    codes = rng.integers(0, 256, size=shape).astype(np.uint8)
    vals = torch.from_numpy(codes).view(FP8_TORCH[t]).to(torch.float64).numpy()
    # finite, and |v| < 2^8, so that the exact sums of the tiny shapes below
    # still fit fp64's 53 bits (the test compares for equality)
    bad = ~np.isfinite(vals) | (np.abs(vals) >= 256.0)
    codes[bad] = codes[bad] & 0x83  # exponent field cleared: a finite (subnormal) code
    vals = torch.from_numpy(codes).view(FP8_TORCH[t]).to(torch.float64).numpy()
    assert np.isfinite(vals).all()
    return vals, codes


def pin_fp8_gemm(orc):
    rng = np.random.default_rng(17)
    for t in (E4M3, E5M2):
        for (M, N, K), (a_col, b_col) in itertools.product(
                [(1, 1, 1), (2, 3, 1), (3, 2, 5), (4, 4, 17)], itertools.product((0, 1), repeat=2)):
            A, Ab = _rand_fp8(rng, (M, K), t)
            B, Bb = _rand_fp8(rng, (K, N), t)
            C = (rng.integers(-64, 64, size=(M, N)) / 16).astype(np.float32)
            D, S = orc.gemm_f64_rows(M, N, K, to_storage(Ab, a_col), to_storage(Bb, b_col), C,
                                     ab_type=t, c_type=F32, a_col=a_col, b_col=b_col)
            Af = [[exact_ref.decode(int(v), t) for v in r] for r in Ab]
            Bf = [[exact_ref.decode(int(v), t) for v in r] for r in Bb]
            Cf = [[Fraction(float(v)) for v in r] for r in C]
            ex = exact_ref.exact_gemm(Af, Bf, Cf)
            for i in range(M):
                for j in range(N):
                    assert Fraction(float(D[i, j])) == ex[i][j], (t, M, N, K, i, j)
                    assert Fraction(float(S[i, j])) == sum(abs(Af[i][k] * Bf[k][j])
                                                           for k in range(K))
        # identity: D = B + C; all ones: D = K + C
        n, N = 24, 20
        B, Bb = _rand_fp8(rng, (n, N), t)
        C = rng.standard_normal((n, N)).astype(np.float32)
        D, _ = orc.gemm_f64_rows(n, N, n, fp8_bits(np.eye(n), t), Bb, C, ab_type=t, c_type=F32)
        assert np.array_equal(D, B + C.astype(np.float64))
        for K in (1, 9, 300):
            D, S = orc.gemm_f64_rows(3, 2, K, fp8_bits(np.ones((3, K)), t),
                                     fp8_bits(np.ones((K, 2)), t), None, ab_type=t)
            assert np.all(D == K) and np.all(S == K)


def _mx_exact(Ab, Bb, SA, SB, C, t):
    """Exact rational value and magnitude sum of the block-scaled product from
    the microscaling definition: element (i, k) of A is 2^(SA[i, k//32] - 127)
    times its 8-bit float value, element (k, j) of B 2^(SB[j, k//32] - 127)
    times its value (decoded by exact_ref, independently of the oracle)."""
    M, K = Ab.shape
    N = Bb.shape[1]
    x = lambda e: Fraction(2) ** (int(e) - 127)
    A = [[x(SA[i, k // 32]) * exact_ref.decode(int(Ab[i, k]), t) for k in range(K)]
         for i in range(M)]
    B = [[x(SB[j, k // 32]) * exact_ref.decode(int(Bb[k, j]), t) for j in range(N)]
         for k in range(K)]
    D = [[sum((A[i][k] * B[k][j] for k in range(K)), Fraction(0)) +
          (Fraction(float(C[i, j])) if C is not None else 0) for j in range(N)] for i in range(M)]
    S = [[sum((abs(A[i][k] * B[k][j]) for k in range(K)), Fraction(0)) for j in range(N)]
         for i in range(M)]
    return D, S


def pin_mx_gemm(orc):
    """Block-scaled 8-bit float product.  (1) With every scale 2^0 (exponent
    127) it is the unscaled product, bit for bit; (2) on tiny shapes with
    random scales and K across block boundaries it matches the exact rational
    value of the microscaling definition within fp64's summation bound;
    (3) raising all of a row's (a column's) scales by t multiplies that row
    (column) of D - C by 2^t exactly; (4) a NaN scale (exponent 255) makes
    its row NaN."""
    rng = np.random.default_rng(29)
    for t in (E4M3, E5M2):
        # (1) unit scales reduce to the unscaled product
        for (M, N, K), (a_col, b_col) in itertools.product(
                [(3, 5, 1), (4, 3, 33), (2, 6, 70), (5, 4, 96)], itertools.product((0, 1), repeat=2)):
            _, Ab = _rand_fp8(rng, (M, K), t)
            _, Bb = _rand_fp8(rng, (K, N), t)
            C = (rng.integers(-64, 64, size=(M, N)) / 16).astype(np.float32)
            nb = (K + 31) // 32
            one_a = np.full((M, nb), 127, np.uint8)
            one_b = np.full((N, nb), 127, np.uint8)
            a, b = to_storage(Ab, a_col), to_storage(Bb, b_col)
            D, S = orc.gemm_mx_rows(M, N, K, a, b, C, one_a, one_b, ab_type=t, c_type=F32,
                                    a_col=a_col, b_col=b_col)
            D0, S0 = orc.gemm_f64_rows(M, N, K, a, b, C, ab_type=t, c_type=F32, a_col=a_col,
                                       b_col=b_col)
            assert np.array_equal(D, D0) and np.array_equal(S, S0), (t, M, N, K)
        # (2) exact rational value, random scales
        for (M, N, K), (a_col, b_col) in itertools.product(
                [(1, 1, 1), (2, 3, 31), (3, 2, 32), (2, 2, 33), (3, 3, 70)],
                itertools.product((0, 1), repeat=2)):
            _, Ab = _rand_fp8(rng, (M, K), t)
            _, Bb = _rand_fp8(rng, (K, N), t)
            C = (rng.integers(-64, 64, size=(M, N)) / 16).astype(np.float32)
            nb = (K + 31) // 32
            SA = rng.integers(118, 137, size=(M, nb)).astype(np.uint8)
            SB = rng.integers(118, 137, size=(N, nb)).astype(np.uint8)
            D, S = orc.gemm_mx_rows(M, N, K, to_storage(Ab, a_col), to_storage(Bb, b_col), C,
                                    SA, SB, ab_type=t, c_type=F32, a_col=a_col, b_col=b_col)
            ex, exs = _mx_exact(Ab, Bb, SA, SB, C, t)
            for i in range(M):
                for j in range(N):
                    bound = Fraction(K + 1, 2 ** 52) * (exs[i][j] + abs(Fraction(float(C[i, j]))))
                    assert abs(Fraction(float(D[i, j])) - ex[i][j]) <= bound, (t, M, N, K, i, j)
                    assert abs(Fraction(float(S[i, j])) - exs[i][j]) <= bound, (t, M, N, K, i, j)
        # (3) a row's / a column's scales raised by t2: that row / column times 2^t2
        M, N, K = 4, 5, 100
        _, Ab = _rand_fp8(rng, (M, K), t)
        _, Bb = _rand_fp8(rng, (K, N), t)
        SA = rng.integers(120, 135, size=(M, 4)).astype(np.uint8)
        SB = rng.integers(120, 135, size=(N, 4)).astype(np.uint8)
        D, _ = orc.gemm_mx_rows(M, N, K, Ab, Bb, None, SA, SB, ab_type=t)
        SA2 = SA.copy()
        SA2[2] += 3
        D2, _ = orc.gemm_mx_rows(M, N, K, Ab, Bb, None, SA2, SB, ab_type=t)
        assert np.array_equal(D2[2], D[2] * 8) and np.array_equal(np.delete(D2, 2, 0),
                                                                  np.delete(D, 2, 0))
        SB2 = SB.copy()
        SB2[4] -= 2
        D3, _ = orc.gemm_mx_rows(M, N, K, Ab, Bb, None, SA, SB2, ab_type=t)
        assert np.array_equal(D3[:, 4], D[:, 4] / 4) and np.array_equal(D3[:, :4], D[:, :4])
        # (4) a NaN scale poisons its row (every column reads that block)
        SA3 = SA.copy()
        SA3[1, 3] = 255
        D4, _ = orc.gemm_mx_rows(M, N, K, Ab, Bb, None, SA3, SB, ab_type=t)
        assert np.isnan(D4[1]).all() and np.array_equal(np.delete(D4, 1, 0), np.delete(D, 1, 0))


# ----------------------------------------------------------------------------- rounding
def pin_round_midpoints(orc):
    for t in (F16, BF16):
        b = np.arange(INF_BITS[t], dtype=np.uint32).astype(np.uint16)
        lo = orc.widen_bits(b, t)
        hi = np.empty_like(lo)
        hi[:-1] = lo[1:]
        hi[-1] = 2.0 ** EMAX1[t]                # the successor of the largest finite value
        mid = (lo + hi) / 2                     # exact in fp64
        up = np.nextafter(mid, np.inf)
        down = np.nextafter(mid, 0.0)
        exp_mid = np.where(b % 2 == 0, b, b + 1).astype(np.uint16)
        assert np.array_equal(orc.round_bits(lo, t), b), f"type {t}: values not fixed points"
        assert np.array_equal(orc.round_bits(mid, t), exp_mid), f"type {t}: ties not to even"
        assert np.array_equal(orc.round_bits(up, t), (b + 1).astype(np.uint16)), f"type {t}: above tie"
        assert np.array_equal(orc.round_bits(down, t), b), f"type {t}: below tie"
        assert np.array_equal(orc.round_bits(-mid, t), exp_mid | np.uint16(0x8000)), "sign"


def pin_round_vs_libraries(orc):
    rng = np.random.default_rng(7)
    # log-uniform magnitudes spanning fp16 subnormals to beyond fp16 overflow
    mag = np.exp2(rng.uniform(-30, 17, 200_000))
    x = mag * rng.choice([-1.0, 1.0], mag.size)
    with np.errstate(over="ignore"):
        ref16 = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(orc.round_bits(x, F16), ref16), "fp16 rounding differs from numpy"
    # bf16: values exactly representable in fp32 (torch rounds fp32 -> bf16 with RNE)
    x32 = (np.exp2(rng.uniform(-140, 127, 200_000)) * rng.choice([-1.0, 1.0], 200_000)).astype(
        np.float32)
    refbf = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.round_bits(x32.astype(np.float64), BF16), refbf), \
        "bf16 rounding differs from torch"


def pin_round_vs_exact(orc):
    rng = random.Random(11)
    xs = []
    for _ in range(3000):
        e = rng.uniform(-140, 130)
        xs.append(rng.choice([-1, 1]) * 2.0 ** e * rng.uniform(1, 2))
    xs += [0.0, -0.0, 65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]
    x = np.array(xs)
    for t in (F16, BF16):
        got = orc.round_bits(x, t)
        for v, g in zip(xs, got):
            want = exact_ref.round_exact(Fraction(v), t)
            if v == 0.0:
                want = 0x8000 if str(v).startswith("-") else 0
            assert int(g) == want, f"type {t}: round({v!r}) = {int(g):#06x}, want {want:#06x}"


# ----------------------------------------------------------------------------- GEMM
def _rand_values(rng, shape, t, small_int=False):
    if small_int:
        return rng.integers(-2, 3, shape).astype(np.float64)
    v = rng.standard_normal(shape)
    if t == F16:
        return v.astype(np.float16).astype(np.float64)
    return torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()


def pin_brute_force_tiny(orc):
    rng = np.random.default_rng(3)
    cases = 0
    for M, N, K in itertools.product((1, 2, 3), repeat=3):
        for a_col, b_col, c_col in itertools.product((0, 1), repeat=3):
            t = F16 if (M + N + K + a_col) % 2 else BF16
            small = (M * N * K) % 3 == 0
            A = _rand_values(rng, (M, K), t, small)
            B = _rand_values(rng, (K, N), t, small)
            C = _rand_values(rng, (M, N), t, small)
            Af, Bf, Cf = ([[Fraction(float(v)) for v in r] for r in X] for X in (A, B, C))
            exact = exact_gemm_f = exact_ref.exact_gemm(Af, Bf, Cf)
            D, S = orc.gemm_f64_rows(M, N, K, to_storage(bits_of(A, t), a_col),
                                     to_storage(bits_of(B, t), b_col),
                                     to_storage(bits_of(C, t), c_col), ab_type=t, c_type=t,
                                     a_col=a_col, b_col=b_col, c_col=c_col)
            for i in range(M):
                for j in range(N):
                    assert Fraction(float(D[i, j])) == exact_gemm_f[i][j], (M, N, K, i, j)
                    s = sum(abs(Af[i][k] * Bf[k][j]) for k in range(K))
                    assert Fraction(float(S[i, j])) == s
            for out_t in (F16, BF16):
                got = orc.round_bits(D, out_t)
                for i in range(M):
                    for j in range(N):
                        assert int(got[i, j]) == exact_ref.round_exact(exact[i][j], out_t)
            cases += 1
    # exhaustive 1x1x1 over small integers, C in fp32 and absent
    for a, b, c in itertools.product((-2, -1, 0, 1, 2), repeat=3):
        D, _ = orc.gemm_f64_rows(1, 1, 1, f16_bits(np.array([[a]])), f16_bits(np.array([[b]])),
                                 np.array([[c]], np.float32), ab_type=F16, c_type=F32)
        assert D[0, 0] == a * b + c
        D0, _ = orc.gemm_f64_rows(1, 1, 1, f16_bits(np.array([[a]])),
                                  f16_bits(np.array([[b]])), None, ab_type=F16)
        assert D0[0, 0] == a * b
    assert cases == 27 * 8


def pin_closed_forms(orc):
    rng = np.random.default_rng(5)
    t = BF16
    n, N = 48, 40
    B = _rand_values(rng, (n, N), t)
    C = _rand_values(rng, (n, N), t)
    # identity: D = B + C exactly, S = |B|
    I = np.eye(n)
    for a_col, b_col in itertools.product((0, 1), repeat=2):
        D, S = orc.gemm_f64_rows(n, N, n, to_storage(bits_of(I, t), a_col),
                                 to_storage(bits_of(B, t), b_col), bits_of(C, t), ab_type=t,
                                 c_type=t, a_col=a_col, b_col=b_col)
        assert np.array_equal(D, B + C) and np.array_equal(S, np.abs(B))
    # permutation: D = P B + C, a row shuffle
    perm = rng.permutation(n)
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1.0
    for a_col in (0, 1):
        D, _ = orc.gemm_f64_rows(n, N, n, to_storage(bits_of(P, t), a_col), bits_of(B, t),
                                 bits_of(C, t), ab_type=t, c_type=t, a_col=a_col)
        assert np.array_equal(D, B[perm] + C)
    # rank 1 (K = 1): D = a b^T + C, exact in fp64
    a = _rand_values(rng, (n, 1), t)
    b = _rand_values(rng, (1, N), t)
    D, _ = orc.gemm_f64_rows(n, N, 1, bits_of(a, t), bits_of(b, t), bits_of(C, t), ab_type=t,
                             c_type=t)
    assert np.array_equal(D, a @ b + C)
    # all ones: D = K + C
    for K in (1, 7, 64, 1000):
        ones_a, ones_b = np.ones((5, K)), np.ones((K, 6))
        Cs = _rand_values(rng, (5, 6), t)
        D, S = orc.gemm_f64_rows(5, 6, K, bits_of(ones_a, t), bits_of(ones_b, t), bits_of(Cs, t),
                                 ab_type=t, c_type=t)
        assert np.array_equal(D, K + Cs) and np.all(S == K)
    # linearity on small integers (exact): f(A,B,C) = f(A,B,0) + C and additivity in A
    A1 = _rand_values(rng, (n, 33), t, True)
    A2 = _rand_values(rng, (n, 33), t, True)
    Bi = _rand_values(rng, (33, N), t, True)
    Ci = _rand_values(rng, (n, N), t, True)
    f = lambda A_, C_: orc.gemm_f64_rows(n, N, 33, bits_of(A_, t), bits_of(Bi, t),
                                         None if C_ is None else bits_of(C_, t), ab_type=t,
                                         c_type=t)[0]
    assert np.array_equal(f(A1, Ci), f(A1, None) + Ci)
    assert np.array_equal(f(A1 + A2, None), f(A1, None) + f(A2, None))
    # empty K: D = C
    D, S = orc.gemm_f64_rows(n, N, 0, np.zeros((n, 0), np.uint16), np.zeros((0, N), np.uint16),
                             bits_of(C, t), ab_type=t, c_type=t)
    assert np.array_equal(D, C) and np.all(S == 0)


def pin_views_agree(orc):
    """Rows, points and storage orders give the same numbers (same k order)."""
    rng = np.random.default_rng(9)
    t, M, N, K = F16, 37, 29, 53
    A = _rand_values(rng, (M, K), t)
    B = _rand_values(rng, (K, N), t)
    C = rng.standard_normal((M, N)).astype(np.float32)
    D, S = orc.gemm_f64_rows(M, N, K, bits_of(A, t), bits_of(B, t), C, ab_type=t, c_type=F32)
    # numpy fp64 matmul as a cross-check of the whole array (rounding order differs)
    np.testing.assert_allclose(D, A @ B + C, rtol=0, atol=1e-12 * (np.abs(A) @ np.abs(B)).max())
    for a_col, b_col, c_col in itertools.product((0, 1), repeat=3):
        D2, _ = orc.gemm_f64_rows(M, N, K, to_storage(bits_of(A, t), a_col),
                                  to_storage(bits_of(B, t), b_col), to_storage(C, c_col),
                                  ab_type=t, c_type=F32, a_col=a_col, b_col=b_col, c_col=c_col)
        assert np.array_equal(D, D2)
    rows = np.array([0, 36, 5, 5, 17])
    Dr, Sr = orc.gemm_f64_rows(M, N, K, bits_of(A, t), bits_of(B, t), C, ab_type=t, c_type=F32,
                               rows=rows)
    assert np.array_equal(Dr, D[rows]) and np.array_equal(Sr, S[rows])
    pi, pj = rng.integers(0, M, 300), rng.integers(0, N, 300)
    Dp, Sp = orc.gemm_f64_points(M, N, K, bits_of(A, t), bits_of(B, t), C, pi, pj, ab_type=t,
                                 c_type=F32)
    assert np.array_equal(Dp, D[pi, pj]) and np.array_equal(Sp, S[pi, pj])
    # a square problem (the 8192^3 checks sample points of one): (i, j) is not (j, i)
    n = 31
    A = _rand_values(rng, (n, K), t)
    B = _rand_values(rng, (K, n), t)
    D, _ = orc.gemm_f64_rows(n, n, K, bits_of(A, t), bits_of(B, t), None, ab_type=t)
    pi, pj = rng.integers(0, n, 300), rng.integers(0, n, 300)
    Dp, _ = orc.gemm_f64_points(n, n, K, bits_of(A, t), bits_of(B, t), None, pi, pj, ab_type=t)
    assert np.array_equal(Dp, D[pi, pj])


def pin_int8(orc):
    g = torch.Generator().manual_seed(21)
    M, N, K = 23, 19, 301
    A = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
    B = torch.randint(-128, 128, (K, N), generator=g, dtype=torch.int8)
    C = torch.randint(-(2 ** 20), 2 ** 20 + 1, (M, N), generator=g, dtype=torch.int32)
    ref = (A.long() @ B.long() + C.long()).numpy()
    for a_col, b_col, c_col in itertools.product((0, 1), repeat=3):
        D = orc.gemm_i64_rows(M, N, K, to_storage(A.numpy(), a_col), to_storage(B.numpy(), b_col),
                              to_storage(C.numpy(), c_col), a_col=a_col, b_col=b_col, c_col=c_col)
        assert np.array_equal(D, ref), (a_col, b_col, c_col)
    pi, pj = np.array([0, 22, 7]), np.array([18, 0, 9])
    Dp = orc.gemm_i64_points(M, N, K, A.numpy(), B.numpy(), C.numpy(), pi, pj)
    assert np.array_equal(Dp, ref[pi, pj])
    # square: points (i, j) and (j, i) differ
    Aq, Bq = A[:19], B
    refq = (Aq.long() @ Bq.long()).numpy()
    pi, pj = np.array([0, 18, 3, 7]), np.array([18, 0, 11, 2])
    Dq = orc.gemm_i64_points(19, 19, K, Aq.contiguous().numpy(), Bq.numpy(), None, pi, pj)
    assert np.array_equal(Dq, refq[pi, pj])
    D0 = orc.gemm_i64_rows(M, N, K, A.numpy(), B.numpy(), None)
    assert np.array_equal(D0, (A.long() @ B.long()).numpy())
    # worst case: all -128, K = 8192 -> 2^27 + C
    K = 8192
    Aw = np.full((3, K), -128, np.int8)
    Bw = np.full((K, 4), -128, np.int8)
    Cw = np.array([[2 ** 20, -(2 ** 20), 0, 1]] * 3, np.int32)
    D = orc.gemm_i64_rows(3, 4, K, Aw, Bw, Cw)
    assert np.array_equal(D, 2 ** 27 + Cw.astype(np.int64))


PINS = [pin_widen_exhaustive, pin_round_midpoints, pin_round_vs_libraries, pin_round_vs_exact,
        pin_brute_force_tiny, pin_closed_forms, pin_views_agree, pin_int8, pin_widen_fp8,
        pin_fp8_gemm, pin_mx_gemm]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(orc, pin):
    pin(orc)


def test_numpy_f16_conversion_is_direct_rne():
    """The numpy conversion used as a pin rounds fp64 directly (no fp32 step)."""
    # 1 + 2^-11 + 2^-40 is above the fp16 tie at 1 + 2^-11; via fp32 it would
    # become the tie itself and round down to 1.0.
    x = np.array([1 + 2.0 ** -11 + 2.0 ** -40])
    assert x.astype(np.float16)[0] == np.float16(1 + 2.0 ** -10)
    assert exact_ref.round_exact(Fraction(float(x[0])), F16) == 0x3C01


def test_oracle_threads(orc):
    assert orc.threads() >= 1


@pytest.mark.parametrize("mutant", range(1, 19))
def test_pins_catch_planted_mistakes(mutant):
    with tempfile.TemporaryDirectory() as d:
        path = oracle.compile_library(os.path.join(d, f"liboracle_m{mutant}.so"), mutant=mutant)
        bad = oracle.Oracle(path)
        failed = []
        for pin in PINS:
            try:
                pin(bad)
            except Exception:  # an assertion, or garbage values the pin cannot even read
                failed.append(pin.__name__)
        assert failed, f"no pin caught planted mistake {mutant}"
