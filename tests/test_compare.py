"""CPU tests of the acceptance rule (oracle/compare.py) that every GPU parity
test applies: that it accepts what the rule allows and rejects the rest, so a
green parity run means what it says.

* spacing(): for every finite fp16 / bf16 encoding, the distance from the
  value to the next encoding away from zero, computed here from the oracle's
  exact widening of neighbouring encodings (the spacing of the binade of
  |y|, the subnormal spacing below the normal range);
* check_float(): exact and one-ulp results pass with no slack used; two ulps
  off fail where S and C are zero; the fp32 bound 2e-6 * S + 2^-24 * |C| is
  applied at its edge; NaN and infinity always fail; a transposed result
  fails; the slack count reports the elements that needed the fp32 bound;
* check_int(): equality only.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from oracle import BF16, F16, F32, compare

INF_BITS = {F16: 0x7C00, BF16: 0x7F80}


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("t", [F16, BF16])
def test_spacing_is_the_gap_to_the_next_encoding(orc, t):
    bits = np.arange(INF_BITS[t], dtype=np.uint32).astype(np.uint16)  # +0 .. largest finite
    vals = orc.widen_bits(bits, t)
    nxt = np.empty_like(vals)
    nxt[:-1] = vals[1:]
    nxt[-1] = vals[-1] + (vals[-1] - vals[-2])  # the largest finite value keeps its binade's gap
    assert np.array_equal(compare.spacing(bits, t), nxt - vals)
    # negative encodings have the spacing of their magnitude
    neg = (bits.astype(np.uint32) | 0x8000).astype(np.uint16)
    assert np.array_equal(compare.spacing(neg, t), nxt - vals)


def _ref(orc, t, n=4000, seed=0):
    rng = np.random.default_rng(seed)
    D_ref = rng.standard_normal(n) * np.exp2(rng.integers(-20, 12, n))
    bits = orc.round_bits(D_ref, t)
    return D_ref, orc.widen_bits(bits, t), compare.spacing(bits, t)


@pytest.mark.parametrize("t", [F16, BF16])
def test_narrow_output_rule(orc, t):
    D_ref, rnd, ulp = _ref(orc, t)
    zero = np.zeros_like(D_ref)
    rep = compare.check_float(orc, rnd, D_ref, zero, zero, t)
    assert rep["ok"] and rep["n_needed_slack"] == 0 and rep["max_err_over_bound"] == 0
    # one ulp away (either side) is within "one output ulp of the correctly rounded value"
    for sgn in (1, -1):
        rep = compare.check_float(orc, rnd + sgn * ulp, D_ref, zero, zero, t)
        assert rep["ok"] and rep["n_needed_slack"] == 0
    # two ulps away fails everywhere when S and C give no slack
    rep = compare.check_float(orc, rnd + 2 * ulp, D_ref, zero, zero, t)
    assert not rep["ok"] and rep["n_fail"] == D_ref.size
    # ... and passes where the fp32 bound covers the extra ulp, counted as slack
    S = np.full_like(D_ref, 0.0)
    S[::2] = ulp[::2] / 2e-6                   # 2e-6 * S = one more ulp on even elements
    rep = compare.check_float(orc, rnd + 2 * ulp, D_ref, S, zero, t)
    assert rep["n_fail"] == D_ref.size - D_ref[::2].size
    assert rep["n_needed_slack"] == D_ref[::2].size
    # |C| * 2^-24 slack works the same way
    Cabs = np.ldexp(ulp, 24)
    rep = compare.check_float(orc, rnd + 2 * ulp, D_ref, zero, Cabs, t)
    assert rep["ok"] and rep["n_needed_slack"] == D_ref.size


def test_fp32_output_rule(orc):
    rng = np.random.default_rng(3)
    n = 3000
    D_ref = rng.standard_normal(n) * 50
    S = np.abs(D_ref) * 10 + rng.random(n) * 100
    Cabs = rng.random(n) * 1e3
    bound = 2e-6 * S + np.ldexp(Cabs, -24)
    inside = D_ref + bound * 0.999
    rep = compare.check_float(orc, inside, D_ref, S, Cabs, F32)
    assert rep["ok"] and rep["max_err_over_bound"] < 1
    outside = D_ref - bound * 1.001
    rep = compare.check_float(orc, outside, D_ref, S, Cabs, F32)
    assert rep["n_fail"] == n


@pytest.mark.parametrize("t", [F16, BF16, F32])
def test_non_finite_results_fail(orc, t):
    D_ref = np.array([1.0, -2.5, 3.0e-3])
    S = np.full(3, 1e30)  # a huge bound must not excuse a non-finite value
    D = np.array([np.nan, np.inf, -np.inf])
    rep = compare.check_float(orc, D, D_ref, S, np.zeros(3), t)
    assert rep["n_fail"] == 3


@pytest.mark.parametrize("t", [BF16, F32])
def test_transposed_result_fails(orc, t):
    """A GEMM result computed with a transposed operand is far outside the rule."""
    rng = np.random.default_rng(5)
    n, K = 48, 64
    A = rng.integers(-8, 8, (n, K)).astype(np.float64) / 8
    B = rng.integers(-8, 8, (K, n)).astype(np.float64) / 8
    D_ref = A @ B
    S = np.abs(A) @ np.abs(B)
    wrong = D_ref.T  # the product stored transposed
    rep = compare.check_float(orc, wrong, D_ref, S, np.zeros_like(S), t)
    assert not rep["ok"] and rep["n_fail"] > n * n // 2
    rep = compare.check_float(orc, D_ref, D_ref, S, np.zeros_like(S), t)
    assert rep["ok"]


def test_int_rule():
    D_ref = np.array([[0, -7, 2 ** 27 + 5]], dtype=np.int64)
    assert compare.check_int(D_ref.astype(np.int32), D_ref)["ok"]
    D = D_ref.copy()
    D[0, 2] += 1
    rep = compare.check_int(D, D_ref)
    assert not rep["ok"] and rep["n_fail"] == 1 and rep["first_failures"][0][0] == (0, 2)


def test_block_scaled_coefficient():
    """max(2e-6, ceil(K/32) * 2^-23): the default below K = 544, one fp32 ulp
    of the running sum per 32-element block above it."""
    assert compare.mx_s_rel(32) == 2e-6
    assert compare.mx_s_rel(512) == 2e-6
    assert compare.mx_s_rel(8192) == 256 * 2.0 ** -23
    assert compare.mx_s_rel(8193) == 257 * 2.0 ** -23
    D_ref = np.array([1000.0])
    S = np.array([1000.0])
    over = 1000.0 - 1.5 * 256 * 2.0 ** -23 * 1000.0  # outside 2e-6 S, inside the wider bound
    assert not compare.check_float(None, np.array([over]), D_ref, S, np.zeros(1), F32)["ok"]
    assert compare.check_float(None, np.array([over]), D_ref, S, np.zeros(1), F32,
                               s_rel=compare.mx_s_rel(8192 * 2))["ok"]
