"""Acceptance rule for a computed D against the oracle (test infrastructure).

Floating point (the sum accumulated in fp32 by the library, in fp64 here):

* fp32 output:   |D - D_ref| <= 2e-6 * S + 2^-24 * |C|
* fp16/bf16 out: |D - rnd(D_ref)| <= ulp(rnd(D_ref)) + 2e-6 * S + 2^-24 * |C|

where S[i,j] = sum_k |A[i,k] * B[k,j]|, rnd is one round-to-nearest-even of
the fp64 value to the output type and ulp(y) is the spacing of the output
format at |y| (the subnormal spacing for tiny values).  The first term of the
narrow-output rule is "within one output ulp of the correctly rounded value";
the other two are the fp32 bound, which only matter where |D| is small next
to S (cancellation), and the report counts how many elements needed them.

Block-scaled 8-bit floats (the scaled product whose tolerance the pages do
not state): the same rule with the S coefficient widened to
max(2e-6, ceil(K / 32) * 2^-23).  The tensor core adds the scaled partial of
each 32-element K block into an fp32 accumulator, and each of those ceil(K/32)
additions may be off by up to one fp32 ulp of the running sum, so by at most
2^-23 * S (the additions measured on the GPU round toward zero: every result
outside the narrower bound lies on the small-magnitude side of the exact
value).  ``mx_s_rel(K)`` gives the coefficient.

Integer: D must equal the int64 oracle value exactly.
"""
from __future__ import annotations

import numpy as np

from . import F16, BF16, F32

_FMT = {F16: (10, 15), BF16: (7, 127)}  # (fraction bits, bias)


def spacing(bits: np.ndarray, t: int) -> np.ndarray:
    """Spacing of format t at |y| for encodings y (finite values)."""
    frac_bits, bias = _FMT[t]
    e = (bits.astype(np.int64) >> frac_bits) & ((1 << (15 - frac_bits)) - 1)
    e = np.maximum(e, 1)
    return np.ldexp(1.0, (e - bias - frac_bits).astype(np.int64))


def mx_s_rel(K: int) -> float:
    """S coefficient of the block-scaled rule: max(2e-6, ceil(K/32) * 2^-23)."""
    return max(2e-6, -(-K // 32) * 2.0 ** -23)


def check_float(oracle, D, D_ref, S, C_abs, out_type: int, max_report: int = 8,
                s_rel: float = 2e-6) -> dict:
    """Compare computed values D (fp64 view of the output) with the oracle.

    D, D_ref, S, C_abs are same-shape fp64 arrays (C_abs = |C| or zeros).
    s_rel is the coefficient of S (2e-6, or mx_s_rel(K) for the block-scaled
    product).  Returns a report dict; ``report["ok"]`` is the verdict.
    """
    D = np.asarray(D, dtype=np.float64)
    D_ref = np.asarray(D_ref, dtype=np.float64)
    slack = s_rel * np.asarray(S, dtype=np.float64) + np.ldexp(np.asarray(C_abs, np.float64), -24)
    if out_type == F32:
        err = np.abs(D - D_ref)
        bound = slack
        strict = np.zeros(D.shape, dtype=bool)
        target = D_ref
    else:
        ref_bits = oracle.round_bits(D_ref, out_type)
        target = oracle.widen_bits(ref_bits, out_type)
        ulp = spacing(ref_bits, out_type)
        err = np.abs(D - target)
        strict = err <= ulp
        bound = ulp + slack
    finite = np.isfinite(D)
    bad = ~(finite & (err <= bound))
    idx = np.argwhere(bad)[:max_report]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    return {
        "ok": not bool(bad.any()),
        "n": int(D.size),
        "n_fail": int(bad.sum()),
        "n_needed_slack": int((~bad & ~strict).sum()) if out_type != F32 else 0,
        "max_err_over_bound": float(np.nanmax(ratio)) if D.size else 0.0,
        "first_failures": [
            (tuple(int(v) for v in i), float(D[tuple(i)]), float(target[tuple(i)]),
             float(bound[tuple(i)])) for i in idx
        ],
    }


def check_int(D, D_ref, max_report: int = 8) -> dict:
    D = np.asarray(D, dtype=np.int64)
    D_ref = np.asarray(D_ref, dtype=np.int64)
    bad = D != D_ref
    idx = np.argwhere(bad)[:max_report]
    return {
        "ok": not bool(bad.any()),
        "n": int(D.size),
        "n_fail": int(bad.sum()),
        "first_failures": [(tuple(int(v) for v in i), int(D[tuple(i)]), int(D_ref[tuple(i)]))
                           for i in idx],
    }
