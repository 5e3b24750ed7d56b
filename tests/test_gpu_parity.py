"""GPU parity: the CUDA library through its C ABI against the CPU oracle.

Floating point uses the acceptance rule of oracle/compare.py (one output ulp
of the correctly rounded fp64 value, plus the fp32 accumulation bound where
the sum cancels); fp32 output uses the fp32 bound alone; int8 is bit-exact.
Closed forms (identity / permutation operands) are checked bit for bit,
which exposes any transposed or mis-swizzled operand tile.
"""
from __future__ import annotations

import itertools

import numpy as np
import pytest
import torch

import dense_tiled_gemm_02_gb300 as pkg
from gpu_helpers import (check_points, check_rows, check_rows_mx, forced_plan, logical, run_gpu,
                         run_gpu_mx)
from workloads import (BF16, COL, E4M3, E5M2, F16, F32, I8, I32, ROW, TORCH_DTYPE, WORKLOADS,
                       Workload, draw, draw_scales,
                       make_inputs, make_scales, sample_points, sample_rows, storage_shape)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkg.load()


def _assert_ok(rep, what):
    assert rep["ok"], f"{what}: {rep['n_fail']} of {rep['n']} outside tolerance; first {rep['first_failures']}"


# ------------------------------------------------------------------ closed forms, bit-exact
PERM_PLANS = ([(bn, 0, 1) for bn in (64, 128, 256)] + [(bn, 1, 1) for bn in (128, 256)]
              + [(bn, 1, 2) for bn in (128, 256)])


@pytest.mark.parametrize("bn,pair,ksub", PERM_PLANS,
                         ids=[f"bn{b}-pair{p}-ksub{k}" for b, p, k in PERM_PLANS])
@pytest.mark.parametrize("a_col,b_col", list(itertools.product((ROW, COL), repeat=2)))
@pytest.mark.parametrize("swap", [0, 1])
def test_permutation_is_exact(bn, pair, ksub, a_col, b_col, swap):
    """A = P (a permutation): D = P B exactly, for every operand layout and
    both the single-CTA and the CTA-pair kernels."""
    M = K = 320
    N = 384
    g = torch.Generator().manual_seed(bn * 7 + a_col * 3 + b_col + 11 * swap)
    perm = torch.randperm(M, generator=g)
    P = torch.zeros(M, K, dtype=torch.bfloat16)
    P[torch.arange(M), perm] = 1
    B = torch.randn(K, N, generator=g).to(torch.bfloat16)
    w = Workload("perm", 0, M, N, K, BF16, None, BF16, "normal", a_col, b_col, ROW, ROW)
    inp = {"A": P if a_col == ROW else P.t().contiguous(),
           "B": B if b_col == ROW else B.t().contiguous(), "C": None}
    D, plan = run_gpu(w, inp, plan=f"bn={bn},swap={swap},pair={pair},ksub={ksub}")
    assert torch.equal(D.view(torch.int16), B[perm].view(torch.int16)), plan


@pytest.mark.parametrize("bn", [64, 128, 256])
def test_identity_plus_c(bn):
    """A = I: D = rnd(B + C); checked against the oracle (one rounding)."""
    M = K = 256
    N = 320
    g = torch.Generator().manual_seed(5 + bn)
    I = torch.eye(M, K).to(torch.float16)
    B = torch.randn(K, N, generator=g).to(torch.float16)
    C = torch.randn(M, N, generator=g).to(torch.float16)
    w = Workload("ident", 0, M, N, K, F16, F16, F16, "normal")
    inp = {"A": I, "B": B, "C": C}
    D, plan = run_gpu(w, inp, plan=f"bn={bn}")
    _assert_ok(check_rows(w, inp, D), plan)


# ------------------------------------------------------------------ the small configs, every element
@pytest.mark.parametrize("name", ["sq256_f16_f32", "sq1024_f16", "rag1000_bf16"])
@pytest.mark.parametrize("plan", [None, "bn=64", "bn=128", "bn=256", "bn=128,splits=3",
                                  "bn=64,group=1", "bn=128,swap=1", "pair=1,bn=256",
                                  "pair=1,bn=128", "pair=1,bn=256,grid=28",
                                  "pair=1,bn=256,grid=28,tail=0", "pair=1,bn=256,splits=2",
                                  "pair=1,bn=128,swap=1", "pair=1,bn=256,ksub=2",
                                  "pair=1,bn=256,ksub=2,splits=3", "pair=1,bn=128,ksub=2",
                                  # stream-K runs over a few clusters
                                  "pair=1,bn=128,grid=20", "pair=1,bn=256,ksub=2,grid=22",
                                  # single-CTA stream-K, shared tiles finished in the kernel
                                  "pair=0,bn=128,sk=1", "pair=0,bn=64,sk=1",
                                  "pair=0,bn=256,sk=1,grid=37", "pair=0,bn=64,sk=1,swap=1",
                                  # K slices loaded in groups of 2 and 4
                                  "pair=0,bn=64,kgroup=2", "pair=0,bn=128,kgroup=4,splits=3",
                                  "pair=0,bn=64,kgroup=4,sk=1"])
def test_small_config(name, plan):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    D, p = run_gpu(w, inp, plan=plan)
    _assert_ok(check_rows(w, inp, D), f"{name} [{p}]")


SHAPES = [
    # (M, N, K, layout_a, layout_b, layout_c, layout_d, ab, c, d)
    (1, 1, 1, ROW, ROW, ROW, ROW, BF16, BF16, BF16),
    (1, 1, 17, ROW, COL, ROW, ROW, F16, F16, F32),
    (129, 257, 65, ROW, ROW, ROW, ROW, BF16, BF16, BF16),
    (129, 257, 65, COL, COL, COL, COL, F16, F32, F16),
    (7, 300, 1000, ROW, ROW, ROW, ROW, BF16, BF16, BF16),
    (513, 77, 129, COL, ROW, ROW, COL, BF16, None, F32),
    (300, 520, 200, ROW, COL, ROW, ROW, BF16, BF16, BF16),
    (64, 2048, 4096, ROW, ROW, ROW, ROW, BF16, BF16, BF16),
    (1000, 96, 3000, ROW, COL, COL, ROW, F16, F16, F16),
    (255, 255, 255, ROW, ROW, ROW, ROW, BF16, BF16, BF16),
    # split-K with workspace rows that are not 16-byte multiples
    (1000, 90, 4096, ROW, ROW, ROW, ROW, BF16, BF16, BF16),
    (999, 130, 2000, ROW, COL, ROW, ROW, F16, F32, F32),
]


@pytest.mark.parametrize("plan", [None, "pair=1,bn=256", "pair=1,bn=128", "pair=1,bn=256,ksub=2",
                                  "pair=0,bn=128,sk=1", "pair=0,bn=64,sk=1,grid=150",
                                  "pair=0,bn=64,kgroup=2", "pair=0,bn=128,lsu=1",
                                  "pair=0,bn=256,lsu=1,swap=0"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"{s[0]}x{s[1]}x{s[2]}-{s[3]}{s[4]}{s[5]}{s[6]}"
                                               for s in SHAPES])
def test_ragged_shapes(shape, plan):
    M, N, K, la, lb, lc, ld, ab, ct, dt = shape
    w = Workload("shape", 7, M, N, K, ab, ct, dt, "normal", la, lb, lc, ld)
    inp = make_inputs(w, seed_offset=M + N + K)
    D, p = run_gpu(w, inp, plan=plan)
    _assert_ok(check_rows(w, inp, D), f"{shape} [{p}]")


@pytest.mark.parametrize("plan", [None, "pair=0", "pair=1,bn=256", "pair=1,bn=128", "pair=1,bn=256,ksub=2",
                                  "pair=0,bn=128,sk=1"])
def test_unaligned_c_d_rows_and_aliased(plan):
    """16-bit C and D rows that are not 16-byte aligned go through aligned
    workspace copies (stage_c / stage_d in the plan); D may alias C there."""
    M, N, K = 390, 301, 200
    w = Workload("stage", 10, M, N, K, BF16, BF16, BF16, "normal")
    inp = make_inputs(w)
    A, B = inp["A"].cuda(), inp["B"].cuda()
    CD = inp["C"].cuda().clone()  # C in, D out, same buffer (ld = 301)
    with forced_plan(plan):
        g = pkg.Gemm.like(A, B, CD, CD)
    plan_str = g.plan()
    assert "stage_c=1" in plan_str and "stage_d=1" in plan_str, plan_str
    g.run(A, B, CD, CD)
    assert g.status() == pkg.GEMM_OK
    g.close()
    _assert_ok(check_rows(w, inp, CD.cpu()), f"aliased [{plan_str}]")


def _placed(t: torch.Tensor, ld: int, off: int, fill: float) -> tuple[torch.Tensor, torch.Tensor]:
    """A device view of the rows x cols tensor t at column offset off of a
    (rows + 2) x ld buffer filled with `fill` (row 0 and the last row are
    guard rows); returns (view, buffer)."""
    rows, cols = t.shape
    buf = torch.full((rows + 2, ld), fill, dtype=t.dtype, device="cuda")
    view = buf[1:1 + rows, off:off + cols]
    view.copy_(t.cuda())
    return view, buf


# (M, N, K, type, C (ld, offset) or None, D (ld, offset)): rows off 16 bytes
# through the stride (odd ld) or the base (offset 1 with an aligned ld), for
# C alone, D alone and both, and aligned rows padded past an N that is not
# a multiple of 8; ragged tiles in M and N.
ROWS_CASES = [
    (600, 700, 300, BF16, (701, 0), (704, 0)),      # C rows off, D by TMA
    (600, 700, 300, BF16, (704, 0), (703, 0)),      # C by vectors, D rows off
    (600, 700, 300, F16, (705, 3), (709, 5)),       # both off, f16
    (513, 515, 130, BF16, (528, 1), (528, 1)),      # aligned ld, base off by one element
    (520, 300, 64, F16, None, (301, 0)),            # no C, D rows off
    (257, 1000, 520, BF16, (1001, 0), (1001, 0)),   # stream-K tail, both off
]


@pytest.mark.parametrize("plan", ["pair=1,bn=256", "pair=1,bn=128", "pair=1,bn=256,tail=1,grid=8"])
@pytest.mark.parametrize("case", ROWS_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}-{i}"
                                                  for i, c in enumerate(ROWS_CASES)])
def test_pair_c_d_placements(case, plan):
    """C and D placed in padded buffers, rows aligned or not: every element
    against the oracle, and nothing written outside D's view (the pair
    kernel's TMA store, its by-rows store of the chunk crossing N, and the
    staged copies)."""
    M, N, K, t, cspec, dspec = case
    w = Workload("rows", 12, M, N, K, t, t if cspec else None, t, "normal")
    inp = make_inputs(w, seed_offset=M + N)
    A, B = inp["A"].cuda(), inp["B"].cuda()
    C = None
    if cspec:
        C, _ = _placed(inp["C"], cspec[0], cspec[1], 0.0)
    D, dbuf = _placed(torch.zeros(M, N, dtype=TORCH_DTYPE[t]), dspec[0], dspec[1], 768.0)
    dbuf.fill_(768.0)  # exact in bf16 and fp16
    with forced_plan(plan):
        g = pkg.Gemm.like(A, B, C, D)
    plan_str = g.plan()
    assert "pair=1" in plan_str, plan_str
    g.run(A, B, C, D)
    assert g.status() == pkg.GEMM_OK
    g.close()
    host = dbuf.cpu()
    mask = torch.ones_like(host, dtype=torch.bool)
    mask[1:1 + M, dspec[1]:dspec[1] + N] = False
    assert torch.all(host[mask] == 768.0), f"write outside D [{plan_str}]"
    _assert_ok(check_rows(w, inp, D.cpu().contiguous()), f"{case} [{plan_str}]")


@pytest.mark.parametrize("plan", [None, "pair=0,bn=128", "pair=0,bn=64", "pair=1,bn=256",
                                  "pair=1,bn=128"])
@pytest.mark.parametrize("lb", [ROW, COL], ids=["Brow", "Bcol"])
def test_padding_never_read_or_written(plan, lb):
    """Operands read in place (rows 16-byte aligned) whose rows are padded
    past K or N with NaN: the padding must not reach D (the TMA loads and the
    C loads stop at K and N), and D's own padding past N keeps its sentinel."""
    M, N, K = 300, 260, 203  # K and N not multiples of 8; leading dimensions are
    w = Workload("pad", 13, M, N, K, BF16, BF16, BF16, "normal", ROW, lb)
    inp = make_inputs(w)
    nan = float("nan")
    A, _ = _placed(inp["A"], 208, 0, nan)
    Bs, _ = _placed(inp["B"], 208 if lb == COL else 264, 0, nan)
    B = Bs.t() if lb == COL else Bs
    C, _ = _placed(inp["C"], 264, 0, nan)
    D, dbuf = _placed(torch.zeros(M, N, dtype=torch.bfloat16), 264, 0, 768.0)
    dbuf.fill_(768.0)
    with forced_plan(plan):
        g = pkg.Gemm.like(A, B, C, D)
    plan_str = g.plan()
    assert "repack_a=0" in plan_str and "repack_b=0" in plan_str, plan_str
    g.run(A, B, C, D)
    assert g.status() == pkg.GEMM_OK
    g.close()
    host = dbuf.cpu()
    mask = torch.ones_like(host, dtype=torch.bool)
    mask[1:1 + M, :N] = False
    assert torch.all(host[mask] == 768.0), f"write outside D [{plan_str}]"
    _assert_ok(check_rows(w, inp, D.cpu().contiguous()), f"padded [{plan_str}]")


@pytest.mark.parametrize("plan", ["pair=0,bn=128,lsu=1", "pair=0,bn=256,lsu=1"])
@pytest.mark.parametrize("la,lb", [(ROW, ROW), (ROW, COL), (COL, ROW), (COL, COL)],
                         ids=["ArowBrow", "ArowBcol", "AcolBrow", "AcolBcol"])
def test_producer_warps_read_unaligned_rows(plan, la, lb):
    """Operands whose rows sit off the 16-byte grid (odd leading dimensions,
    bases one element past an aligned address) read in place by the kernel's
    producer warps, both majors of A and B; the rows are padded with NaN
    before and after, which must never reach D."""
    M, N, K = 300, 260, 203
    w = Workload("lsu", 15, M, N, K, BF16, BF16, BF16, "normal", la, lb)
    inp = make_inputs(w, seed_offset=la * 2 + lb)
    nan = float("nan")
    As, _ = _placed(inp["A"], 205 if la == ROW else 303, 1, nan)
    Bs, _ = _placed(inp["B"], 263 if lb == ROW else 205, 1, nan)
    A = As.t() if la == COL else As
    B = Bs.t() if lb == COL else Bs
    C, _ = _placed(inp["C"], 264, 0, nan)
    D, dbuf = _placed(torch.zeros(M, N, dtype=torch.bfloat16), 264, 0, 768.0)
    dbuf.fill_(768.0)
    with forced_plan(plan):
        g = pkg.Gemm.like(A, B, C, D)
    plan_str = g.plan()
    assert "lsu_a=1" in plan_str and "lsu_b=1" in plan_str, plan_str
    assert "repack_a=0" in plan_str and "repack_b=0" in plan_str, plan_str
    g.run(A, B, C, D)
    assert g.status() == pkg.GEMM_OK
    g.close()
    host = dbuf.cpu()
    mask = torch.ones_like(host, dtype=torch.bool)
    mask[1:1 + M, :N] = False
    assert torch.all(host[mask] == 768.0), f"write outside D [{plan_str}]"
    _assert_ok(check_rows(w, inp, D.cpu().contiguous()), f"producer warps [{plan_str}]")


def test_k_zero_gives_c():
    w = Workload("k0", 8, 130, 70, 0, BF16, F16, F32, "normal")
    inp = make_inputs(w)
    D, _ = run_gpu(w, inp)
    assert torch.equal(D, inp["C"].float())


@pytest.mark.parametrize("M,N,K,b_col", [(0, 100, 2048, ROW), (1, 0, 4096, COL), (0, 0, 0, ROW),
                                         (3, 0, 300, COL), (0, 4096, 4096, COL)])
def test_empty_output(M, N, K, b_col):
    """M or N zero: planning succeeds (the decode and split-K planners are
    not reached), gemm_run and the host-buffer batch return at once, the
    status is clean, and the next handle on the context works."""
    dev = torch.device("cuda")
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=dev)
    Bs = torch.zeros((N, K) if b_col else (K, N), dtype=torch.bfloat16, device=dev)
    B = Bs.t() if b_col else Bs
    C = torch.zeros(M, N, dtype=torch.bfloat16, device=dev)
    D = torch.zeros(M, N, dtype=torch.bfloat16, device=dev)
    desc = pkg.GemmDesc(M, N, K, pkg.GEMM_BF16, pkg.GEMM_BF16, pkg.GEMM_BF16, pkg.GEMM_ROW_MAJOR,
                        b_col, pkg.GEMM_ROW_MAJOR, pkg.GEMM_ROW_MAJOR, max(K, 1),
                        max(K, 1) if b_col else max(N, 1), max(N, 1), max(N, 1))
    g = pkg.Gemm(desc)
    try:
        assert pkg.gemm_workspace_bytes(g.handle) == 0, g.plan()
        assert pkg.gemm_run(g.handle, A.data_ptr(), B.data_ptr(), C.data_ptr(), D.data_ptr(),
                            None) == pkg.GEMM_OK
        assert pkg.gemm_run(g.handle, None, None, None, None, None) == pkg.GEMM_OK
        g.host_io_enable()
        assert pkg.gemm_run_host_batch(g.handle, [None], [None], None, [None], None) == pkg.GEMM_OK
        assert g.status(torch.cuda.current_stream()) == pkg.GEMM_OK
    finally:
        g.close()
    w = WORKLOADS["rag1000_bf16"]
    inp = make_inputs(w)
    Dn, p = run_gpu(w, inp)
    _assert_ok(check_rows(w, inp, Dn, rows=[0, 999]), p)


def test_guard_bands_untouched():
    """D written into a larger buffer (ldd > N, extra rows): canaries survive."""
    M, N, K = 200, 300, 130
    w = Workload("guard", 9, M, N, K, BF16, BF16, BF16, "normal")
    inp = make_inputs(w)
    big = torch.full((M + 9, N + 40), 12345.0, dtype=torch.bfloat16, device="cuda")
    view = big[3:3 + M, 8:8 + N]
    import dense_tiled_gemm_02_gb300 as g_
    A, B, C = inp["A"].cuda(), inp["B"].cuda(), inp["C"].cuda()
    g = g_.Gemm.like(A, B, C, view)
    g.run(A, B, C, view)
    assert g.status() == 0
    g.close()
    host = big.cpu()
    mask = torch.ones_like(host, dtype=torch.bool)
    mask[3:3 + M, 8:8 + N] = False
    assert torch.all(host[mask] == 12345.0)
    _assert_ok(check_rows(w, inp, host[3:3 + M, 8:8 + N].contiguous()), "guard")


def test_side_stream_and_reuse():
    """One handle, two runs on a side stream with different buffers."""
    w = WORKLOADS["rag1000_bf16"]
    s = torch.cuda.Stream()
    for off in (0, 1):
        inp = make_inputs(w, seed_offset=off)
        with torch.cuda.stream(s):
            D, _ = run_gpu(w, inp, stream=s)
        _assert_ok(check_rows(w, inp, D), f"stream run {off}")


def test_kernel_timing_hook():
    """gemm_timing_enable/read: one duration per recorded run, each inside the
    whole call's events (the split-K reduce of this plan falls outside it),
    and the result of the timed runs unchanged."""
    w = WORKLOADS["skinny8192x128x4096_bf16"]
    inp = make_inputs(w)
    dev = torch.device("cuda")
    A, B, C = (logical(inp[k].to(dev), l) for k, l in
               (("A", w.layout_a), ("B", w.layout_b), ("C", w.layout_c)))
    D_storage = torch.empty(storage_shape(w.M, w.N, w.layout_d), dtype=torch.bfloat16,
                            device=dev)
    D = logical(D_storage, w.layout_d)
    g = pkg.Gemm.like(A, B, C, D)
    s = torch.cuda.current_stream()
    n = 3
    g.timing_enable(n)
    outer = []
    for _ in range(n + 1):  # one run more than recorded
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        g.run(A, B, C, D, s)
        e1.record(s)
        outer.append((e0, e1))
    torch.cuda.synchronize()
    ms = g.timing_read(8)
    assert g.status(s) == pkg.GEMM_OK
    assert len(ms) == n
    for k, (e0, e1) in zip(ms, outer):
        assert 0.0 < k <= e0.elapsed_time(e1) * 1.001 + 1e-3
    g.timing_enable(0)
    assert g.timing_read(8) == []
    _assert_ok(check_rows(w, inp, D_storage.cpu(), rows=[0, 127, 128, 4097, w.M - 1]),
               "timed run")
    g.close()


# The measured rows of the selection table (csrc/plan_table.h) are the plans
# these workloads get.
TABLE_ROWS = {
    "sq4096_bf16": "pair=1 bn=256 ksub=1",
    "sq8192_bf16": "pair=1 bn=256 ksub=1",
    "sq8192_i8": "pair=1 bn=256 ksub=1",
    "sq4096_e4m3": "pair=1 bn=224 ksub=1",
    "skinny64x8192x8192_bf16": "swap=0 pair=0 bn=128 ksub=1 stages=5",
    "skinny8192x128x4096_bf16": "swap=0 pair=0 bn=128 ksub=1 stages=5",
    "rag1000_bf16": "swap=0 pair=0 bn=64",
    "decode16x4096x4096_bf16": "swap=1 pair=0 bn=64",
    "decode16x4096x4096_bf16_brow": "swap=1 pair=0 bn=64",
    "decode1x4096x4096_bf16_brow": "swap=1 pair=0 bn=64",
    "sq1024_f16": "swap=0 pair=0 bn=64",
}


@pytest.mark.parametrize("name", sorted(TABLE_ROWS))
def test_plan_table_rows_engage(name):
    w = WORKLOADS[name]
    dev = torch.device("cuda")
    A = torch.empty(storage_shape(w.M, w.K, w.layout_a), dtype=TORCH_DTYPE[w.ab_type], device=dev)
    B = torch.empty(storage_shape(w.K, w.N, w.layout_b), dtype=TORCH_DTYPE[w.ab_type], device=dev)
    D = torch.empty(storage_shape(w.M, w.N, w.layout_d), dtype=TORCH_DTYPE[w.d_type], device=dev)
    C = None if w.c_type is None else torch.empty(storage_shape(w.M, w.N, w.layout_c),
                                                  dtype=TORCH_DTYPE[w.c_type], device=dev)
    g = pkg.Gemm.like(logical(A, w.layout_a), logical(B, w.layout_b),
                      None if C is None else logical(C, w.layout_c), logical(D, w.layout_d))
    plan = g.plan()
    g.close()
    assert TABLE_ROWS[name] in plan, plan
    want_splits = {"skinny64x8192x8192_bf16": 2, "skinny8192x128x4096_bf16": 2,
                   "decode16x4096x4096_bf16": 4, "decode16x4096x4096_bf16_brow": 4,
                   "decode1x4096x4096_bf16_brow": 4}.get(name, 1)
    assert f" splits={want_splits} " in plan, plan
    if name.startswith("skinny"):
        assert f"csk={want_splits}" in plan, plan


# ------------------------------------------------------------------ full-size configs
FULL = [("sq4096_bf16", None), ("sq4096_bf16", "pair=1,bn=256,tail=0"), ("sq4096_e4m3", None),
        ("sq4096_bf16", "pair=0,bn=256"), ("skinny64x8192x8192_bf16", None),
        ("skinny8192x128x4096_bf16", None), ("rag4095x4097x4099_bf16", None),
        ("rag4095x4097x4099_bf16", "pair=1,bn=256"), ("sq4096_bf16", "pair=1,bn=256,ksub=2"),
        ("rag4095x4097x4099_bf16", "pair=1,bn=256,ksub=2"),
        ("skinny64x8192x8192_bf16", "pair=0,bn=128,sk=1"),
        ("skinny64x8192x8192_bf16", "pair=0,bn=64,sk=1,swap=1"),
        ("skinny8192x128x4096_bf16", "pair=0,bn=128,sk=1"),
        ("skinny8192x128x4096_bf16", "pair=0,bn=64,sk=1"),
        ("skinny8192x128x4096_bf16", "pair=0,bn=64,kgroup=4"),
        ("skinny8192x128x4096_bf16", "pair=0,bn=64,splits=1"),
        ("sq4096_bf16", "pair=1,bn=224"), ("sq4096_bf16", "pair=1,bn=224,tail=1"),
        ("rag4095x4097x4099_bf16", "pair=1,bn=224"), ("sq4096_e4m3", "pair=1,bn=224"),
        ("skinny64x8192x8192_bf16", "pair=0,bn=128,splits=2,csk=0"),
        ("skinny64x8192x8192_bf16", "pair=0,bn=128,splits=2,kgroup=2"),
        ("rag4095x4097x4099_bf16", "pair=0,bn=256,lsu=1"),
        ("rag4095x4097x4099_bf16", "pair=0,bn=128,lsu=1"),
        ("skinny8192x128x4096_bf16", "pair=0,bn=128,splits=2,csk=1"),
        ("skinny64x8192x8192_bf16", "pair=0,bn=128,splits=2,csk=1"),
        ("decode16x4096x4096_bf16", "decode=0,pair=0,bn=64,splits=4,csk=1"),
        ("decode1x4096x4096_bf16_brow", "decode=0,pair=0,bn=64,splits=4,csk=1")]


@pytest.mark.parametrize("name,plan", FULL, ids=[f"{n}-{p}" for n, p in FULL])
def test_full_config_every_element(name, plan):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    D, p = run_gpu(w, inp, plan=plan)
    rep = check_rows(w, inp, D)
    _assert_ok(rep, f"{name} [{p}]")
    print(f"{name}: {rep['n']} elements ok, {rep['n_needed_slack']} needed the fp32 slack [{p}]")


@pytest.mark.parametrize("name,plan", [("sq8192_bf16", None), ("sq8192_i8", None),
                                       ("sq8192_i8", "pair=0"), ("sq8192_i8", "native_i8=1"),
                                       ("sq8192_i8", "i8chunk=960"),
                                       ("sq8192_e4m3", None)])
def test_8192_sampled(name, plan):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    D, p = run_gpu(w, inp, plan=plan)
    pi, pj = sample_points(w.M, w.N)
    _assert_ok(check_points(w, inp, D, pi.numpy(), pj.numpy()), f"{name} points [{p}]")
    rows = sample_rows(w.M).numpy()
    _assert_ok(check_rows(w, inp, D, rows=rows), f"{name} rows [{p}]")


# ------------------------------------------------------------------ 8-bit float operands
# (M, N, K, C type or None, D type); A row-major, B column-major (K-major).
F8_CASES = [
    (128, 128, 128, BF16, BF16),
    (300, 520, 200, BF16, BF16),    # rows of 200 bytes: copied to 128-byte workspace rows
    (129, 257, 72, None, F32),
    (1000, 1000, 1000, F16, F16),
    (513, 770, 4096, F32, BF16),
    (64, 2048, 4096, BF16, BF16),   # skinny
    (3, 512, 1024, BF16, F32),      # below the decode kernel's types: the tensor path
]
F8_PLANS = [None, "pair=0,bn=64", "pair=0,bn=128", "pair=0,bn=256", "pair=1,bn=256",
            "pair=1,bn=128", "pair=1,bn=256,ksub=2", "pair=1,bn=256,grid=8,tail=1",
            "pair=0,bn=128,splits=3"]


@pytest.mark.parametrize("plan", F8_PLANS)
@pytest.mark.parametrize("t", [E4M3, E5M2], ids=["e4m3", "e5m2"])
@pytest.mark.parametrize("case", F8_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}" for c in F8_CASES])
def test_fp8_every_element(case, t, plan):
    """kind::f8f6f4 on both kernels (split-K, stream-K, two K slices a stage)
    against the oracle's exact widening of the OFP8 encodings."""
    M, N, K, ct, dt = case
    w = Workload("f8", 14, M, N, K, t, ct, dt, "normal", ROW, COL)
    inp = make_inputs(w, seed_offset=M + K)
    D, p = run_gpu(w, inp, plan=plan)
    _assert_ok(check_rows(w, inp, D), f"{case} {t} [{p}]")


def test_fp8_special_values():
    """E4M3's largest finite (448), subnormals and signed zeros pass through
    unchanged: A = diag of specials, B = I, so D = A exactly."""
    vals = torch.tensor([448.0, -448.0, 2.0 ** -9, -(2.0 ** -9), 2.0 ** -6, 0.0, -0.0, 1.0],
                        dtype=torch.float32)
    n = 128
    A = torch.zeros(n, n, dtype=torch.float32)
    A[torch.arange(n), torch.arange(n)] = vals.repeat(n // vals.numel())
    w = Workload("f8s", 15, n, n, n, E4M3, None, F32, "normal", ROW, COL)
    inp = {"A": A.to(torch.float8_e4m3fn), "B": torch.eye(n).to(torch.float8_e4m3fn).t()
           .contiguous(), "C": None}
    D, p = run_gpu(w, inp)
    assert torch.equal(D, torch.diag(vals.repeat(n // vals.numel()))), p


@pytest.mark.parametrize("name", ["decode1x4096x4096_bf16", "decode16x4096x4096_bf16",
                                  "decode1x4096x4096_bf16_brow", "decode16x4096x4096_bf16_brow"])
def test_decode_shapes_every_element(name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    D, p = run_gpu(w, inp)
    _assert_ok(check_rows(w, inp, D), f"{name} [{p}]")


DECODE_CASES = [
    # (M, N, K, layout_a, ab, c, d, layout_d, B element offset)
    (3, 1000, 1032, ROW, BF16, BF16, BF16, ROW, 0),
    (4, 777, 4096, COL, F16, F32, F32, ROW, 0),
    (2, 512, 264, ROW, BF16, None, BF16, COL, 0),
    (1, 4096, 4096, ROW, BF16, BF16, BF16, ROW, 1),   # B not 16-byte aligned: 2-byte loads
    (1, 333, 2312, ROW, F16, F16, F16, ROW, 0),       # K slices not a multiple of 4 steps
    (4, 64, 8192, ROW, BF16, BF16, BF16, ROW, 0),
    (4, 4096, 4096, ROW, BF16, BF16, BF16, ROW, 0),   # bulk form: 8-column stages, reused
    (1, 8192, 4096, ROW, BF16, None, BF16, ROW, 0),   # bulk form: two waves of blocks
    (2, 4096, 2048, ROW, F16, F16, F32, COL, 0),      # bulk form: a slot per column, fp32 D
]


@pytest.mark.parametrize("plan", [None, "decode=0", "dbulk=1", "dbulk=0", "dmma=1"])
@pytest.mark.parametrize("case", DECODE_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}-off{c[8]}"
                                                   for c in DECODE_CASES])
def test_decode_kernel(case, plan):
    """M <= 4 with a K-contiguous B takes the decode kernel (with decode=0,
    the tensor-core path; dbulk=1 / dbulk=0 force its bulk-copy form on or
    off, the form falling back to the split-K one at run time when A or B is
    off the 16-byte grid); every element against the oracle."""
    M, N, K, la, ab, ct, dt, ld, off = case
    w = Workload("dec", 65, M, N, K, ab, ct, dt, "normal", la, COL, ROW, ld)
    inp = make_inputs(w)
    dev = torch.device("cuda")
    A = logical(inp["A"].to(dev), la)
    flat = torch.zeros(N * K + 8, dtype=inp["B"].dtype, device=dev)
    flat[off:off + N * K] = inp["B"].to(dev).reshape(-1)
    B = flat[off:off + N * K].view(N, K).t()          # K x N, column-major, ldb = K
    C = None if inp["C"] is None else inp["C"].to(dev)
    D_storage = torch.zeros(storage_shape(M, N, ld), dtype=TORCH_DTYPE[dt], device=dev)
    D = logical(D_storage, ld)
    with forced_plan(plan):
        g = pkg.Gemm.like(A, B, C, D)
    p = g.plan()
    assert ("decode=1" in p) == (plan != "decode=0"), p
    k_rows = la == ROW or M == 1  # A's rows K-contiguous (ld a multiple of 8 here)
    if plan == "dbulk=1" and k_rows and K <= 4096:  # A and two stages of B fit
        assert "dbulk=1" in p, p
    if plan == "dbulk=0" or not k_rows:
        assert "dbulk=0" in p, p
    if plan == "decode=0" and off:
        # the tensor-core path reads B with TMA: a B base off the 16-byte grid
        # with 16-byte aligned rows has no workspace copy and is rejected
        with pytest.raises(pkg.GemmError) as e:
            g.run(A, B, C, D)
        assert e.value.code == pkg.GEMM_ERR_MISALIGNED
        g.close()
        return
    g.run(A, B, C, D)
    assert g.status() == pkg.GEMM_OK
    g.close()
    _assert_ok(check_rows(w, inp, D_storage.cpu()), f"{case} [{p}]")


# The tensor-core decode form (mma.sync, up to 16 rows, B in either layout):
# (M, N, K, layout_a, ab, c, d, layout_d, B element offset, layout_b).
DMMA_CASES = [
    (1, 4096, 4096, ROW, BF16, BF16, BF16, ROW, 0, ROW),
    (16, 4096, 4096, ROW, BF16, BF16, BF16, ROW, 0, ROW),
    (5, 1000, 1000, COL, F16, F32, F16, ROW, 0, ROW),    # K ends inside a 16-row step
    (9, 777, 333, ROW, BF16, None, F32, COL, 0, ROW),    # N off the 8-column grid: 2-byte loads
    (16, 264, 2050, ROW, BF16, BF16, BF16, ROW, 1, ROW),  # B off the 16-byte grid
    (8, 136, 24, ROW, F16, F16, F16, ROW, 0, ROW),       # one short K slice
    (7, 4096, 512, ROW, F16, F16, F16, ROW, 0, COL),
    (16, 1000, 4104, COL, BF16, F32, BF16, COL, 0, COL),  # K not a multiple of 128
    (12, 130, 8192, ROW, BF16, BF16, BF16, ROW, 1, COL),  # B off the 16-byte grid, few columns
    (3, 4096, 4096, ROW, BF16, BF16, BF16, ROW, 0, COL),  # forced below 5 rows
    (16, 8, 64, ROW, BF16, BF16, BF16, ROW, 0, COL),
]


# every case with the form forced, the aligned ones also with the default plan
DMMA_RUNS = [(c, "dmma=1") for c in DMMA_CASES] + [(c, None) for c in DMMA_CASES if c[8] == 0]


@pytest.mark.parametrize("case,plan", DMMA_RUNS,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}-{'kc' if c[9] == COL else 'nc'}-off{c[8]}-{p}"
                              for c, p in DMMA_RUNS])
def test_decode_mma_form(case, plan):
    """The warp-level tensor-core decode form (up to 16 rows, B of either
    layout; taken when asked for with dmma=1, else these shapes run on the
    tcgen05 path or, at most 4 rows against a K-contiguous B, the CUDA-core
    decode forms); every element against the oracle."""
    M, N, K, la, ab, ct, dt, ld, off, lb = case
    w = Workload("dmma", 66, M, N, K, ab, ct, dt, "normal", la, lb, ROW, ld)
    inp = make_inputs(w)
    dev = torch.device("cuda")
    A = logical(inp["A"].to(dev), la)
    flat = torch.zeros(N * K + 8, dtype=inp["B"].dtype, device=dev)
    flat[off:off + N * K] = inp["B"].to(dev).reshape(-1)
    B = logical(flat[off:off + N * K].view(storage_shape(K, N, lb)), lb)
    C = None if inp["C"] is None else inp["C"].to(dev)
    D_storage = torch.zeros(storage_shape(M, N, ld), dtype=TORCH_DTYPE[dt], device=dev)
    D = logical(D_storage, ld)
    with forced_plan(plan):
        g = pkg.Gemm.like(A, B, C, D)
    p = g.plan()
    assert ("dmma=1" in p) == (plan == "dmma=1"), p
    g.run(A, B, C, D)
    assert g.status() == pkg.GEMM_OK
    g.close()
    _assert_ok(check_rows(w, inp, D_storage.cpu()), f"{case} [{p}]")


def test_decode_bulk_form_engages_at_4096_columns():
    w = WORKLOADS["decode1x4096x4096_bf16"]
    dev = torch.device("cuda")
    inp = make_inputs(w)
    A = logical(inp["A"].to(dev), w.layout_a)
    B = logical(inp["B"].to(dev), w.layout_b)
    D = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    g = pkg.Gemm.like(A, B, None, D)
    try:
        assert "decode=1 dbulk=1" in g.plan(), g.plan()
    finally:
        g.close()


# ------------------------------------------------------------------ block-scaled 8-bit floats
# (M, N, K, C type or None, D type); A row-major, B column-major.  K not a
# multiple of 32 (a short last block with its own scale), of 128 (a ring
# stage of four blocks), ragged tiles, rows that are copied to workspace.
MX_CASES = [
    (128, 128, 128, BF16, BF16),
    (300, 520, 200, BF16, BF16),
    (129, 257, 72, None, F32),
    (1000, 1000, 1000, F16, BF16),  # scales up to 2^14: |D| beyond fp16's range
    (513, 770, 4096, F32, BF16),
    (256, 384, 8192, BF16, F32),
    (64, 136, 4000, BF16, BF16),
]


@pytest.mark.parametrize("t", [E4M3, E5M2], ids=["e4m3", "e5m2"])
@pytest.mark.parametrize("case", MX_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}" for c in MX_CASES])
def test_mx_every_element(case, t):
    """kind::mxf8f6f4: every element against the oracle's block-scaled
    product (each element times 2^(e - 127) of its 32-element K block)."""
    M, N, K, ct, dt = case
    w = Workload("mx", 16, M, N, K, t, ct, dt, "normal", ROW, COL)
    inp = make_inputs(w, seed_offset=M + K)
    sc = make_scales(w, seed_offset=M + K)
    D, p = run_gpu_mx(w, inp, sc)
    assert " mx=1" in p, p
    _assert_ok(check_rows_mx(w, inp, sc, D), f"mx {case} [{p}]")


def test_mx_8192_sampled_rows():
    """The block-scaled 8192^3 workload: 64 sampled rows (the sampling rule's
    rows) against the oracle."""
    w = WORKLOADS["sq8192_mxe4m3"]
    inp = make_inputs(w)
    sc = make_scales(w)
    D, p = run_gpu_mx(w, inp, sc)
    rows = sample_rows(w.M).numpy()
    _assert_ok(check_rows_mx(w, inp, sc, D, rows=rows), f"sq8192_mxe4m3 rows [{p}]")


def test_mx_scales_reach_the_right_rows_and_blocks():
    """All-ones operands: D[m, n] = sum over K blocks of 32 (or the short last
    block's length) x 2^(ea(m, b) + eb(n, b) - 254), exact in fp32, so a scale
    read from the wrong row, column or block shows up exactly."""
    M, N, K = 256, 128, 300
    w = Workload("mx1", 17, M, N, K, E4M3, None, F32, "normal", ROW, COL)
    inp = {"A": torch.ones(M, K).to(torch.float8_e4m3fn),
           "B": torch.ones(N, K).to(torch.float8_e4m3fn), "C": None}
    sc = {"SA": draw_scales(M, K, 71, 124, 130), "SB": draw_scales(N, K, 72, 124, 130)}
    D, p = run_gpu_mx(w, inp, sc)
    ea = sc["SA"].double() - 127
    eb = sc["SB"].double() - 127
    width = torch.tensor([min(32, K - 32 * b) for b in range((K + 31) // 32)], dtype=torch.float64)
    want = torch.einsum("mb,nb,b->mn", torch.exp2(ea), torch.exp2(eb), width)
    assert torch.equal(D.double(), want), p


# ------------------------------------------------------------------ exact int8
# i8chunk: K of one exact fp32 pass; 960 is the longest whose partial sums
# stay below 2^24 (the all -128 case below reaches 960 * 2^14 per pass)
I8_PLANS = [None, "pair=1,ksub=1", "pair=1,ksub=2", "native_i8=1", "native_i8=1,group=1",
            "pair=1,i8chunk=960", "pair=1,ksub=2,i8chunk=768", "pair=0,i8chunk=960"]


@pytest.mark.parametrize("plan", I8_PLANS)
@pytest.mark.parametrize("shape", [(300, 200, 1500, ROW, ROW), (129, 257, 2049, COL, COL),
                                   (64, 384, 600, ROW, COL), (520, 640, 4160, ROW, ROW)])
def test_int8_exact_small(shape, plan):
    """Exact int8 on both kernels; K spans several 512-wide chunks and ends
    in a partial one."""
    M, N, K, la, lb = shape
    w = Workload("i8", 51, M, N, K, I8, I32, I32, "int", la, lb)
    inp = make_inputs(w)
    D, p = run_gpu(w, inp, plan=plan)
    if plan and "i8chunk" in plan:
        assert plan.split("i8chunk=")[1].split(",")[0] in p.split("i8chunk=")[1], p
    _assert_ok(check_rows(w, inp, D), f"int8 {shape} [{p}]")


I8_SK_CASES = [
    (520, 640, 4160, "pair=1,tail=1,grid=8", -1),     # 9 tiles, 4 clusters: equal runs
    (520, 640, 4160, "pair=1,tail=1,grid=12", 0),     # 9 tiles, 6 clusters: pair chains
    (1024, 1536, 2048, "pair=1,tail=1,grid=20", 2),   # 24 tiles, 10 clusters: both chains
    (1024, 1536, 2048, "pair=1,tail=1,grid=20,ksub=2,i8chunk=512", 2),
]


@pytest.mark.parametrize("case", I8_SK_CASES, ids=[c[3] for c in I8_SK_CASES])
def test_int8_stream_k(case):
    """Exact int8 with stream-K pieces (int32 partials between clusters):
    every element of the sampled rows exact, and the same bits as round-robin
    whole tiles."""
    M, N, K, plan, n3 = case
    w = Workload("i8sk", 54, M, N, K, I8, I32, I32, "int")
    inp = make_inputs(w)
    D, p = run_gpu(w, inp, plan=plan)
    assert "i8x=1" in p and f"skchain={n3}" in p and "tail=0" not in p, p
    _assert_ok(check_rows(w, inp, D), f"int8 stream-K [{p}]")
    D0, p0 = run_gpu(w, inp, plan=plan.replace("tail=1", "tail=0"))
    assert "tail=0" in p0, p0
    assert torch.equal(D, D0), (p, p0)


@pytest.mark.parametrize("plan", I8_PLANS)
def test_int8_without_c(plan):
    """C absent: D = A*B exactly (the pair kernel stages D alone)."""
    M, N, K = 520, 640, 2112
    w = Workload("i8n", 53, M, N, K, I8, None, I32, "int")
    inp = make_inputs(w)
    D, p = run_gpu(w, inp, plan=plan)
    _assert_ok(check_rows(w, inp, D), f"int8 no C [{p}]")


@pytest.mark.parametrize("plan", I8_PLANS)
@pytest.mark.parametrize("fill", [-128, 127])
def test_int8_extremes(fill, plan):
    """All entries at one extreme, K = 8192: |sum| = 2^27 (or 127^2 * 8192)."""
    M, N, K = 256, 256, 8192
    A = torch.full((M, K), fill, dtype=torch.int8)
    B = torch.full((K, N), -128 if fill == -128 else 127, dtype=torch.int8)
    C = torch.randint(-(2 ** 20), 2 ** 20 + 1, (M, N), generator=torch.Generator().manual_seed(3),
                      dtype=torch.int32)
    w = Workload("i8x", 52, M, N, K, I8, I32, I32, "int")
    inp = {"A": A, "B": B, "C": C}
    D, p = run_gpu(w, inp, plan=plan)
    want = (A[0, 0].long() * B[0, 0].long() * K) + C.long()
    assert torch.equal(D.long(), want), p


@pytest.mark.parametrize("shape", [(1000, 1000, 1000, ROW, ROW, ROW),
                                   (255, 129, 4097, COL, COL, COL),
                                   (130, 70, 33, ROW, COL, ROW),
                                   (64, 520, 160, COL, ROW, COL)])
def test_native_int8_every_element(shape):
    """The integer mma.sync kernel: every element bit-exact, for operands read
    in place (row-major A, column-major B) and copied K-contiguous first, with
    ragged tiles in M, N and K, and column-major C and D."""
    M, N, K, la, lb, lcd = shape
    w = Workload("i8n", 54, M, N, K, I8, I32, I32, "int", la, lb, lcd, lcd)
    inp = make_inputs(w, seed_offset=M)
    D, p = run_gpu(w, inp, plan="native_i8=1")
    assert "native_i8=1" in p and f"repack_a={int(la != ROW or K % 16 != 0)}" in p, p
    _assert_ok(check_rows(w, inp, D), f"native int8 {shape} [{p}]")


# ------------------------------------------------------------------ failure detection
@pytest.mark.parametrize("plan", ["pair=0", "pair=1,bn=128"])
def test_bounded_wait_reports_timeout_and_context_survives(plan):
    """A stage that is never filled: the consumer's wait expires after the
    short limit, every role exits, the status word says so, and the next
    GEMM on the same context is correct."""
    from gpu_helpers import forced_plan
    w = WORKLOADS["rag1000_bf16"]
    inp = make_inputs(w)
    A, B, C = (inp[k].cuda() for k in "ABC")
    D = torch.empty(w.M, w.N, dtype=torch.bfloat16, device="cuda")
    with forced_plan(plan):
        g = pkg.Gemm.like(A, B, C, D)
    assert ("pair=1" in g.plan()) == plan.startswith("pair=1"), g.plan()
    assert pkg.gemm_debug_set(g.handle, pkg.GEMM_DEBUG_SKIP_FIRST_FILL, 50_000_000) == 0
    g.run(A, B, C, D)
    assert g.status() == pkg.GEMM_ERR_DEVICE_TIMEOUT
    assert pkg.gemm_debug_set(g.handle, 0, 0) == 0
    g.run(A, B, C, D)
    assert g.status() == pkg.GEMM_OK
    g.close()
    _assert_ok(check_rows(w, inp, D.cpu()), "after timeout")


def test_decode_bulk_wait_reports_timeout_and_context_survives():
    """The decode kernel's bulk-copy form with its first ring stage never
    filled: the consumers' waits expire, the producer waits for the copies it
    did issue, the status word reports the timeout, and the next call on the
    same handle is correct."""
    w = WORKLOADS["decode1x4096x4096_bf16"]
    inp = make_inputs(w)
    dev = torch.device("cuda")
    A = logical(inp["A"].to(dev), w.layout_a)
    B = logical(inp["B"].to(dev), w.layout_b)
    C = logical(inp["C"].to(dev), w.layout_c)
    D = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    g = pkg.Gemm.like(A, B, C, D)
    assert "dbulk=1" in g.plan(), g.plan()
    assert pkg.gemm_debug_set(g.handle, pkg.GEMM_DEBUG_SKIP_FIRST_FILL, 50_000_000) == 0
    g.run(A, B, C, D)
    assert g.status() == pkg.GEMM_ERR_DEVICE_TIMEOUT
    assert pkg.gemm_debug_set(g.handle, 0, 0) == 0
    g.run(A, B, C, D)
    assert g.status() == pkg.GEMM_OK
    g.close()
    _assert_ok(check_rows(w, inp, D.cpu()), "after timeout")


# Split-K over clusters (csk): (M, N, K, layouts A/B/C/D, types C/D, bn, splits)
CSK_CASES = [
    (1000, 520, 2000, ROW, ROW, ROW, ROW, BF16, BF16, 128, 2),
    (300, 200, 4100, ROW, COL, ROW, ROW, None, F32, 64, 3),      # 3 CTAs in a cluster of up to 4
    (129, 64, 8192, COL, ROW, COL, COL, F16, F16, 64, 4),       # column-major C and D
    (64, 1000, 4096, ROW, COL, ROW, ROW, BF16, BF16, 64, 4),    # swapped (long N on the M side)
    (256, 256, 128, ROW, ROW, ROW, ROW, BF16, BF16, 128, 2),    # one K slice per split
    # rows below M in one 64-row half of the tile only (one half moves)
    (64, 512, 2048, ROW, ROW, ROW, ROW, BF16, BF16, 128, 2),
    (40, 200, 1500, ROW, ROW, ROW, ROW, F16, F16, 64, 3),       # ranks owning 1, 1, 0 slices
    (170, 320, 2500, ROW, ROW, COL, ROW, BF16, BF16, 64, 4),     # C column-major, 4 ranks
]


@pytest.mark.parametrize("case", CSK_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}-s{c[10]}" for c in CSK_CASES])
def test_cluster_split_k(case):
    """The splits of a tile add their sums through the shared memory of
    their cluster; every element against the oracle, no reduce launch."""
    M, N, K, la, lb, lc, ld, ct, dt, bn, s = case
    ab = F16 if ct == F16 else BF16
    w = Workload("csk", 68, M, N, K, ab, ct, dt, "normal", la, lb, lc, ld)
    inp = make_inputs(w)
    D, p = run_gpu(w, inp, plan=f"pair=0,bn={bn},splits={s},csk=1,decode=0")
    assert f"csk={s}" in p and f"splits={s}" in p, p
    _assert_ok(check_rows(w, inp, D), f"csk {case} [{p}]")


@pytest.mark.parametrize("case", CSK_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}-s{c[10]}" for c in CSK_CASES])
def test_cluster_split_k_matches_reduce_launch(case):
    """Both split-K forms add the splits' fp32 sums in split order and then
    C: the cluster exchange gives the same bits as the partials-and-reduce
    form with the same splits."""
    M, N, K, la, lb, lc, ld, ct, dt, bn, s = case
    ab = F16 if ct == F16 else BF16
    w = Workload("csk", 69, M, N, K, ab, ct, dt, "normal", la, lb, lc, ld)
    inp = make_inputs(w)
    D1, p1 = run_gpu(w, inp, plan=f"pair=0,bn={bn},splits={s},csk=1,decode=0")
    D0, p0 = run_gpu(w, inp, plan=f"pair=0,bn={bn},splits={s},csk=0,decode=0")
    assert f"csk={s}" in p1 and "csk=0" in p0, (p1, p0)
    assert torch.equal(D1.view(torch.uint8), D0.view(torch.uint8)), (case, p1)


# Pair kernel epilogue with C by TMA into the staging buffers: several units
# per cluster (few clusters forced by grid=), stream-K pieces, N off the
# 16-byte grid, no C, and a C of another type (the register path).
PAIR_EPI_CASES = [
    (1000, 1000, 1000, BF16, BF16, "pair=1,bn=256,grid=4"),
    (1000, 1003, 1000, BF16, BF16, "pair=1,bn=256,grid=6,tail=1"),
    (777, 1030, 520, F16, F16, "pair=1,bn=256,grid=6,tail=1"),
    (1000, 1000, 1000, None, BF16, "pair=1,bn=256,grid=4"),
    (1000, 1000, 1000, F32, BF16, "pair=1,bn=256,grid=4"),
    (1024, 768, 2048, BF16, BF16, "pair=1,bn=128,grid=4,tail=1"),
    (1024, 768, 2048, BF16, BF16, "pair=1,bn=256,grid=4,ksub=2"),
    # 224-wide tiles (B K-major: 112 rows per CTA): seven 32-column slices,
    # the last 64-column chunk half
    (1000, 1000, 1000, BF16, BF16, "pair=1,bn=224,grid=4,lb=col"),
    (1000, 1003, 1000, BF16, BF16, "pair=1,bn=224,grid=6,tail=1,lb=col"),
    (777, 1030, 520, F16, F16, "pair=1,bn=224,grid=6,tail=1,lb=col"),
    (1000, 1000, 1000, None, BF16, "pair=1,bn=224,grid=4,lb=col"),
    (1000, 1000, 1000, F32, F32, "pair=1,bn=224,grid=4,lb=col"),
    (512, 448, 512, BF16, BF16, "pair=1,bn=224,lb=col"),
]


@pytest.mark.parametrize("case", PAIR_EPI_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}-{c[5]}"
                                                      for c in PAIR_EPI_CASES])
def test_pair_epilogue_c_by_tma(case):
    M, N, K, ct, dt, plan = case
    ab = F16 if dt == F16 else BF16
    lb = COL if plan.endswith(",lb=col") else ROW  # (lb= is the test's, not a plan key)
    plan = plan.replace(",lb=col", "")
    w = Workload("pepi", 69, M, N, K, ab, ct, dt, "normal", ROW, lb)
    inp = make_inputs(w)
    D, p = run_gpu(w, inp, plan=plan)
    assert "pair=1" in p and ("bn=224" in p) == ("bn=224" in plan), p
    _assert_ok(check_rows(w, inp, D), f"{case} [{p}]")


# Pair kernel stream-K with the chained run layout (4C/3 <= S <= 3C/2 of the
# partial last wave's tiles over C clusters, forced by grid=): pairs of runs
# only, triples only, both; ragged K; row-major B; C of another type.
CHAIN_CASES = [
    (512, 1280, 1024, ROW, BF16, BF16, 8, 0),      # C = 4, S = 6: two pairs
    (512, 1792, 1000, COL, BF16, BF16, 12, 2),     # C = 6, S = 8: two triples
    (1024, 1536, 1024, COL, F16, F16, 20, 2),      # C = 10, S = 14: two of each
    (1024, 1536, 2048, ROW, F32, BF16, 20, 2),
]


@pytest.mark.parametrize("case", CHAIN_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}-g{c[6]}"
                                                   for c in CHAIN_CASES])
def test_pair_stream_k_chained_runs(case):
    """Every element against the oracle with the chained stream-K runs and,
    forced back (skpat=0), with the equal runs."""
    M, N, K, lb, ct, dt, grid, n3 = case
    ab = F16 if dt == F16 or ct == F16 else BF16
    w = Workload("chain", 70, M, N, K, ab, ct, dt, "normal", ROW, lb)
    inp = make_inputs(w)
    D, p = run_gpu(w, inp, plan=f"pair=1,bn=256,tail=1,grid={grid}")
    assert f"skchain={n3}" in p, p
    _assert_ok(check_rows(w, inp, D), f"{case} [{p}]")
    D0, p0 = run_gpu(w, inp, plan=f"pair=1,bn=256,tail=1,grid={grid},skpat=0")
    assert "skchain=-1" in p0 and "tail=0" not in p0, p0
    _assert_ok(check_rows(w, inp, D0), f"{case} [{p0}]")


def test_timeline_hook_stamps_in_order():
    """gemm_trace_set: every CTA of the single-CTA kernel stamps its events in
    causal order; with the hook off the buffer is left alone."""
    import re
    w = Workload("tl", 67, 1000, 520, 700, BF16, BF16, BF16, "normal")
    inp = make_inputs(w)
    dev = torch.device("cuda")
    A, B, C = inp["A"].to(dev), inp["B"].to(dev), inp["C"].to(dev)
    D = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    with forced_plan("pair=0,bn=64"):
        g = pkg.Gemm.like(A, B, C, D)
    grid = int(re.search(r"grid=(\d+)", g.plan()).group(1))
    buf = torch.zeros(grid * pkg.GEMM_TRACE_EVENTS, dtype=torch.int64, device=dev)
    assert pkg.gemm_trace_set(g.handle, buf.data_ptr()) == pkg.GEMM_OK
    g.run(A, B, C, D)
    assert g.status() == pkg.GEMM_OK
    t = buf.view(grid, pkg.GEMM_TRACE_EVENTS).cpu()[:, :8]  # 8 on: split-K and pair kernel only
    assert (t > 0).all()
    # each thread's own stamps are in order (0-2 thread 0, 3-4 the MMA
    # thread, 5-7 the first epilogue thread)
    for a, b in ((0, 1), (1, 2), (3, 4), (5, 6), (6, 7)):
        assert (t[:, b] >= t[:, a]).all(), (a, b, t)
    assert pkg.gemm_trace_set(g.handle, None) == pkg.GEMM_OK
    buf.zero_()
    g.run(A, B, C, D)
    assert g.status() == pkg.GEMM_OK
    assert int(buf.abs().sum()) == 0
    g.close()
    _assert_ok(check_rows(w, inp, D.cpu()), "timeline run")
