"""Exact rational reference for tiny GEMMs (an independent pin of the oracle).

Pure Python over ``fractions.Fraction``; it shares nothing with the C oracle:

* decoding uses the standard library's IEEE binary16 codec (``struct`` 'e')
  and, for bfloat16, the binary32 codec on the bits shifted into the upper
  half of a float; the 8-bit float types (E4M3, E5M2) are decoded by
  torch's own float8 dtypes;
* rounding to fp16/bf16 is a nearest-neighbour search over the sorted table
  of every non-negative encoding (ties go to the even encoding; the encoding
  after the largest finite value is infinity, with value 2^(emax+1), which
  makes overflow follow IEEE 754 without a special case);
* the GEMM is the definition D[i,j] = C[i,j] + sum_k A[i,k] B[k,j], exact.
"""
from __future__ import annotations

import bisect
import struct
from fractions import Fraction
from functools import lru_cache

F16, BF16, F32, E4M3, E5M2 = 1, 2, 3, 6, 7


def _decode8(bits: int, t: int) -> float:
    import torch
    dt = torch.float8_e4m3fn if t == E4M3 else torch.float8_e5m2
    return float(torch.tensor([bits], dtype=torch.uint8).view(dt).float()[0])


def decode(bits: int, t: int) -> Fraction | float:
    if t == F16:
        v = struct.unpack("<e", struct.pack("<H", bits))[0]
    elif t == BF16:
        v = struct.unpack("<f", struct.pack("<I", bits << 16))[0]
    elif t in (E4M3, E5M2):
        v = _decode8(bits, t)
    else:
        raise ValueError(t)
    if v != v or v in (float("inf"), float("-inf")):
        return v
    return Fraction(v)


@lru_cache(maxsize=None)
def _table(t: int):
    inf_bits = 0x7C00 if t == F16 else 0x7F80
    vals = [decode(b, t) for b in range(inf_bits)]
    inf_val = Fraction(2) ** (16 if t == F16 else 128)
    return vals + [inf_val], inf_bits


def round_exact(q: Fraction, t: int) -> int:
    """Encoding of the value of format t nearest to q (ties to even)."""
    vals, inf_bits = _table(t)
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    if a >= vals[-1]:
        return sign | inf_bits
    hi = bisect.bisect_left(vals, a)        # vals[hi] >= a
    if vals[hi] == a:
        return sign | hi
    lo = hi - 1
    dl, dh = a - vals[lo], vals[hi] - a
    if dl < dh:
        pick = lo
    elif dh < dl:
        pick = hi
    else:
        pick = lo if lo % 2 == 0 else hi
    return sign | pick


def exact_gemm(A, B, C):
    """A: M x K, B: K x N, C: M x N (or None); lists of Fractions."""
    M = len(A)
    K = len(B)
    N = len(B[0]) if K else (len(C[0]) if C else 0)
    out = []
    for i in range(M):
        row = []
        for j in range(N):
            s = sum((A[i][k] * B[k][j] for k in range(K)), Fraction(0))
            if C is not None:
                s += C[i][j]
            row.append(s)
        out.append(row)
    return out
