"""Seeded synthetic workloads for D = A*B + C (shared by tests and bench).

This module only draws inputs; it holds none of the GEMM's arithmetic.  The
CUDA library and the CPU oracle both read the very same host buffers.

Every operand is drawn on the CPU with ``torch.Generator`` in its own storage
order (a column-major operand is drawn as the row-major array of its
transpose; the entries are i.i.d., so nothing depends on that choice):

* uniform[-1, 1]: fp32 ``rand * 2 - 1`` rounded once to fp16
* normal(0, 1):   fp32 ``randn`` rounded once to bf16
* int8:           ``randint(-128, 128)``; int32 C: ``randint(-2**20, 2**20 + 1)``
* E4M3 / E5M2 operands (8-bit floats): fp32 ``randn`` rounded once by
  torch's float8 conversion (nearest even; |x| < 448 always fits)

Seeds: ``seed = 1000 * idx + {0: A, 1: B, 2: C}`` with the workload index
below.  The shapes and distributions are the ones the pages' workloads use
(the square Triton example at 1024^3 with 32x32x32 blocks, the 4096^3 bf16
tuning table, ragged/skinny shapes, and an 8192^3 int8 case).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

F16, BF16, F32, I8, I32, E4M3, E5M2 = 1, 2, 3, 4, 5, 6, 7
ROW, COL = 0, 1
F8 = (E4M3, E5M2)

TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32,
               I8: torch.int8, I32: torch.int32, E4M3: torch.float8_e4m3fn,
               E5M2: torch.float8_e5m2}
TYPE_NAME = {F16: "f16", BF16: "bf16", F32: "f32", I8: "i8", I32: "i32", E4M3: "e4m3",
             E5M2: "e5m2"}


@dataclass(frozen=True)
class Workload:
    name: str
    idx: int
    M: int
    N: int
    K: int
    ab_type: int
    c_type: int | None      # None: C = 0 (not read)
    d_type: int
    dist: str               # "uniform" | "normal" | "int"
    layout_a: int = ROW
    layout_b: int = ROW
    layout_c: int = ROW
    layout_d: int = ROW
    mx: bool = False        # 8-bit float operands with E8M0 scales per 32-element K block
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    "sq256_f16_f32": Workload("sq256_f16_f32", 1, 256, 256, 256, F16, F16, F32, "uniform"),
    "sq1024_f16": Workload("sq1024_f16", 2, 1024, 1024, 1024, F16, None, F16, "uniform"),
    "sq4096_bf16": Workload("sq4096_bf16", 3, 4096, 4096, 4096, BF16, BF16, BF16, "normal",
                            layout_b=COL),
    "sq8192_bf16": Workload("sq8192_bf16", 31, 8192, 8192, 8192, BF16, BF16, BF16, "normal",
                            layout_b=COL),
    # 8192^3 with a row-major (N-contiguous) B: the operand layout of the
    # int8 workload, for comparing the kernels' two B majors at one size
    "sq8192_bf16_browB": Workload("sq8192_bf16_browB", 32, 8192, 8192, 8192, BF16, BF16, BF16,
                                  "normal"),
    "rag1000_bf16": Workload("rag1000_bf16", 41, 1000, 1000, 1000, BF16, BF16, BF16, "normal"),
    "skinny64x8192x8192_bf16": Workload("skinny64x8192x8192_bf16", 42, 64, 8192, 8192, BF16,
                                        BF16, BF16, "normal"),
    "skinny8192x128x4096_bf16": Workload("skinny8192x128x4096_bf16", 43, 8192, 128, 4096, BF16,
                                         BF16, BF16, "normal"),
    "rag4095x4097x4099_bf16": Workload("rag4095x4097x4099_bf16", 44, 4095, 4097, 4099, BF16,
                                       BF16, BF16, "normal"),
    "sq8192_i8": Workload("sq8192_i8", 5, 8192, 8192, 8192, I8, I32, I32, "int"),
    # 8-bit float operands (K-major A and B, as the kind::f8f6f4 path reads
    # them), bf16 C and D
    "sq4096_e4m3": Workload("sq4096_e4m3", 51, 4096, 4096, 4096, E4M3, BF16, BF16, "normal",
                            layout_b=COL),
    "sq8192_e4m3": Workload("sq8192_e4m3", 52, 8192, 8192, 8192, E4M3, BF16, BF16, "normal",
                            layout_b=COL),
    # the same with E8M0 block scales (make_scales: 2^-7 .. 2^7 per block)
    "sq4096_mxe4m3": Workload("sq4096_mxe4m3", 53, 4096, 4096, 4096, E4M3, BF16, BF16, "normal",
                              layout_b=COL, mx=True),
    "sq8192_mxe4m3": Workload("sq8192_mxe4m3", 54, 8192, 8192, 8192, E4M3, BF16, BF16, "normal",
                              layout_b=COL, mx=True),
    # decode regime (M <= 16, N = K = 4096), with B K-contiguous (a weight
    # stored N x K) and N-contiguous
    "decode1x4096x4096_bf16": Workload("decode1x4096x4096_bf16", 61, 1, 4096, 4096, BF16, BF16,
                                       BF16, "normal", layout_b=COL),
    "decode16x4096x4096_bf16": Workload("decode16x4096x4096_bf16", 62, 16, 4096, 4096, BF16,
                                        BF16, BF16, "normal", layout_b=COL),
    "decode1x4096x4096_bf16_brow": Workload("decode1x4096x4096_bf16_brow", 63, 1, 4096, 4096,
                                            BF16, BF16, BF16, "normal"),
    "decode16x4096x4096_bf16_brow": Workload("decode16x4096x4096_bf16_brow", 64, 16, 4096, 4096,
                                             BF16, BF16, BF16, "normal"),
}


def storage_shape(rows: int, cols: int, layout: int) -> tuple[int, int]:
    """Shape of the dense row-major array that stores a rows x cols operand."""
    return (rows, cols) if layout == ROW else (cols, rows)


def draw(shape, dtype_code: int, dist: str, seed: int, c_operand: bool = False) -> torch.Tensor:
    """One operand, drawn on the CPU in storage order."""
    g = torch.Generator().manual_seed(seed)
    if dist == "uniform":
        return (torch.rand(shape, generator=g, dtype=torch.float32) * 2 - 1).to(
            TORCH_DTYPE[dtype_code])
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32).to(TORCH_DTYPE[dtype_code])
    if dist == "int":
        if c_operand:
            return torch.randint(-(2 ** 20), 2 ** 20 + 1, shape, generator=g, dtype=torch.int32)
        return torch.randint(-128, 128, shape, generator=g, dtype=torch.int8)
    raise ValueError(dist)


def make_inputs(w: Workload, seed_offset: int = 0) -> dict:
    """Host tensors A, B, C (C may be None), each dense in its storage order."""
    base = 1000 * w.idx + seed_offset
    A = draw(storage_shape(w.M, w.K, w.layout_a), w.ab_type, w.dist, base + 0)
    B = draw(storage_shape(w.K, w.N, w.layout_b), w.ab_type, w.dist, base + 1)
    C = None
    if w.c_type is not None:
        C = draw(storage_shape(w.M, w.N, w.layout_c), w.c_type, w.dist, base + 2, c_operand=True)
    return {"A": A, "B": B, "C": C}


def draw_scales(rows: int, K: int, seed: int, lo: int = 120, hi: int = 134) -> torch.Tensor:
    """E8M0 exponents (uint8) of the 32-element K blocks of `rows` rows (rows
    of A, or columns of B): rows x ceil(K / 32), i.i.d. uniform integers in
    [lo, hi] (scales 2^-7 .. 2^7 by default)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (rows, (K + 31) // 32), generator=g,
                         dtype=torch.int32).to(torch.uint8)


def make_scales(w: Workload, seed_offset: int = 0) -> dict:
    """Seeded E8M0 block scales of a block-scaled workload: SA for the rows of
    A, SB for the columns of B (seeds 1000 idx + 3 and + 4)."""
    base = 1000 * w.idx + seed_offset
    return {"SA": draw_scales(w.M, w.K, base + 3), "SB": draw_scales(w.N, w.K, base + 4)}


def sample_points(M: int, N: int, n: int = 65536, seed: int = 0x5EED):
    """Seeded (i, j) pairs, uniform with replacement."""
    g = torch.Generator().manual_seed(seed)
    pi = torch.randint(0, M, (n,), generator=g, dtype=torch.int64)
    pj = torch.randint(0, N, (n,), generator=g, dtype=torch.int64)
    return pi, pj


def sample_rows(M: int, n: int = 64, seed: int = 0x5EED + 1):
    """Tile-edge rows {0, 127, 128, M-1} plus distinct seeded rows, n in all."""
    fixed = [r for r in (0, 127, 128, M - 1) if 0 <= r < M]
    fixed = sorted(set(fixed))
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(M, generator=g).tolist()
    rest = [r for r in perm if r not in fixed][: max(0, n - len(fixed))]
    return torch.tensor(fixed + rest, dtype=torch.int64)


def bits_of(t: torch.Tensor):
    """Bit patterns of a 16-bit (uint16) or 8-bit float (uint8) CPU tensor,
    the oracle's input form."""
    if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return t.contiguous().view(torch.uint8).numpy()
    return bits_u16(t)


def bits_u16(t: torch.Tensor):
    """uint16 numpy view of an fp16/bf16 CPU tensor (the oracle's input form)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")
