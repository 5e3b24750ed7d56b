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
    # 8-bit float operands: K-major A and B only, 16/32-bit float C and D
    (dict(ab_type=pkg.GEMM_E4M3), pkg.GEMM_ERR_UNSUPPORTED),           # B row-major
    (dict(ab_type=pkg.GEMM_E5M2, layout_a=1, layout_b=1), pkg.GEMM_ERR_UNSUPPORTED),
    (dict(ab_type=pkg.GEMM_E4M3, layout_b=1, d_type=pkg.GEMM_I32), pkg.GEMM_ERR_UNSUPPORTED),
    (dict(ab_type=pkg.GEMM_E4M3, layout_b=1, d_type=pkg.GEMM_E4M3), pkg.GEMM_ERR_UNSUPPORTED),
    (dict(ab_type=pkg.GEMM_E5M2, layout_b=1, c_type=pkg.GEMM_I32), pkg.GEMM_ERR_UNSUPPORTED),
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
    # a valid 8-bit float description passes validation and reaches the device check
    rc, h = pkg.gemm_create(_desc(ab_type=pkg.GEMM_E4M3, layout_b=1, d_type=pkg.GEMM_F32))
    assert rc == pkg.GEMM_ERR_NO_DEVICE and h is None


def test_null_handles():
    lib = pkg.load()
    assert lib.gemm_destroy(None) == 0
    assert lib.gemm_run(None, None, None, None, None, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_get_status(None, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_plan_string(None, None, 0) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_workspace_bytes(None) == -1
    assert lib.gemm_create(None, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_host_io_enable(None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_run_host_batch(None, 0, None, None, None, None, None) == \
        pkg.GEMM_ERR_INVALID_ARG


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


def _grouped_tile(t, num_pid_m, num_pid_n, group_m):
    """The grouped mapping of the FlagGems "Hygon optimization" page, section
    "Grouped scheduling: improve L2 data reuse", written out step by step:
    a group spans GROUP_M tile rows and every tile column; the tile's group
    is t // (GROUP_M * num_pid_n); the last group is clamped to the tile rows
    that remain; inside a group the row index runs fastest."""
    num_pid_in_group = group_m * num_pid_n
    group_id = t // num_pid_in_group
    first_pid_m = group_id * group_m
    group_size_m = min(num_pid_m - first_pid_m, group_m)
    pid_m = first_pid_m + (t % num_pid_in_group) % group_size_m
    pid_n = (t % num_pid_in_group) // group_size_m
    return pid_m, pid_n


@pytest.mark.parametrize("npm,npn,g", [(1, 1, 1), (5, 3, 2), (32, 16, 8), (7, 9, 4), (3, 11, 8),
                                       (16, 1, 8), (1, 16, 8), (64, 64, 1), (33, 17, 8),
                                       (16, 16, 8), (13, 5, 16), (12, 40, 5)])
def test_raster_equals_the_grouped_formula(npm, npn, g):
    """Tile for tile, the library's order is the page's formula (a reordered
    walk that is still grouped would pass the bijection test above)."""
    for t in range(npm * npn):
        rc, pm, pn = pkg.gemm_raster_tile(t, npm, npn, g)
        assert rc == 0 and (pm, pn) == _grouped_tile(t, npm, npn, g), (t, pm, pn)


def test_raster_rejects_out_of_range():
    assert pkg.gemm_raster_tile(6, 2, 3, 2)[0] == pkg.GEMM_ERR_INVALID_ARG
    assert pkg.gemm_raster_tile(-1, 2, 3, 2)[0] == pkg.GEMM_ERR_INVALID_ARG
    assert pkg.gemm_raster_tile(0, 2, 3, 0)[0] == pkg.GEMM_ERR_INVALID_ARG


# ------------------------------------------------------------------ pair-kernel work schedule
def _schedule(tm, tn, group, nkb, ksub, clusters, sk):
    return [pkg.gemm_pair_schedule(tm, tn, group, nkb, ksub, clusters, sk, c)
            for c in range(clusters)]


SCHEDULES = [
    # (tiles_m, tiles_n, group_m, num_kb, ksub, clusters)
    (16, 16, 8, 64, 1, 76),     # 4096^3 at 256x256 on 152 SMs
    (32, 32, 8, 128, 1, 76),    # 8192^3
    (16, 17, 8, 65, 1, 76),     # 4095 x 4097 x 4099
    (16, 16, 8, 64, 2, 76),     # two K slices per stage
    (16, 16, 8, 66, 2, 74),
    (5, 31, 4, 3, 1, 76),       # short K: runs of a few stages
    (7, 11, 8, 2, 1, 76),       # 77 tiles: one full wave and one tile
    (10, 16, 8, 9, 1, 76),
    (4, 4, 2, 64, 1, 16),       # tiles a multiple of the clusters: no stream-K
    (3, 5, 8, 40, 1, 76),       # fewer tiles than clusters: no stream-K
]


@pytest.mark.parametrize("sk", [False, True])
@pytest.mark.parametrize("tm,tn,group,nkb,ksub,clusters", SCHEDULES)
def test_pair_schedule_covers_every_tile_stage_once(tm, tn, group, nkb, ksub, clusters, sk):
    """Every (tile, K slice) is computed by exactly one unit; a shared tile
    has exactly one piece that leaves its partial (slot = its cluster) and
    one that adds that slot's partial and finishes it; the runs of stream-K
    are balanced to one stage."""
    sched = _schedule(tm, tn, group, nkb, ksub, clusters, sk)
    seen = {}
    pieces = {}
    for cid, units in enumerate(sched):
        for (r, c, kb0, kb1, shared, part, slot) in units:
            assert 0 <= r < tm and 0 <= c < tn and 0 <= kb0 < kb1 <= nkb
            assert kb0 % ksub == 0 and (kb1 % ksub == 0 or kb1 == nkb)
            for k in range(kb0, kb1):
                assert (r, c, k) not in seen, ((r, c, k), seen.get((r, c, k)), cid)
                seen[(r, c, k)] = cid
            pieces.setdefault((r, c), []).append((cid, kb0, kb1, shared, part, slot))
    assert len(seen) == tm * tn * nkb
    for tile, ps in pieces.items():
        if len(ps) == 1:
            cid, kb0, kb1, shared, part, slot = ps[0]
            assert (kb0, kb1, shared) == (0, nkb, 0)
            continue
        assert sk and len(ps) == 2, (tile, ps)
        first, second = sorted(ps, key=lambda x: x[1])
        # the K head belongs to the cluster whose run ends there: it finishes
        assert first[1] == 0 and first[3:5] == (1, 0)
        assert second[2] == nkb and second[3:5] == (1, 1)
        assert second[5] == second[0] and first[5] == second[0] == first[0] + 1
    tiles = tm * tn
    if sk and tiles >= clusters and tiles % clusters and nkb % ksub == 0 and nkb // ksub >= 2:
        # every cluster has the same number of full-wave tiles, and the
        # stream-K runs are equal to one stage
        work = [sum(u[3] - u[2] for u in units) for units in sched]
        assert max(work) - min(work) <= ksub
        waves = tiles // clusters
        # after the full-wave tiles: the piece that leaves a partial first (it
        # waits for nothing), then the piece that finishes a shared tile, so
        # every wait is for the first piece of another run, and at most one
        # whole tile follows it (tensor memory holds two accumulators)
        for cid, units in enumerate(sched):
            waits = [i for i, u in enumerate(units) if u[4] and u[5] == 0]
            leaves = [i for i, u in enumerate(units) if u[4] and u[5] == 1]
            assert len(waits) <= 1 and len(leaves) <= 1
            assert all(i == waves - 1 for i in leaves)
            assert all(i == waves - 1 + len(leaves) for i in waits)
            if waits:
                assert len(units) - 1 - waits[0] <= 1
    else:
        assert all(u[4] == 0 for units in sched for u in units)


@pytest.mark.parametrize("tm,tn,group,nkb,ksub,clusters", SCHEDULES)
def test_pair_schedule_chained_runs(tm, tn, group, nkb, ksub, clusters):
    """The kernel's default stream-K layout: every (tile, K slice) once, a
    shared tile split between the end of one run (it finishes) and the start
    of the next (it leaves its partial), every run of at most two pieces
    where the chained layout applies (4C/3 <= S <= 3C/2 stream-K tiles),
    with run lengths of 4/3 or 3/2 tiles; otherwise the equal runs."""
    sched = _schedule(tm, tn, group, nkb, ksub, clusters, 2)
    seen = set()
    pieces = {}
    for cid, units in enumerate(sched):
        for (r, c, kb0, kb1, shared, part, slot) in units:
            for k in range(kb0, kb1):
                assert (r, c, k) not in seen
                seen.add((r, c, k))
            pieces.setdefault((r, c), []).append((cid, kb0, kb1, shared, part, slot))
    assert len(seen) == tm * tn * nkb
    for tile, ps in pieces.items():
        if len(ps) == 2:
            first, second = sorted(ps, key=lambda x: x[1])
            assert first[1] == 0 and first[3:5] == (1, 0) and second[2] == nkb
            assert second[3:5] == (1, 1) and first[5] == second[5] == second[0] == first[0] + 1
        else:
            assert len(ps) == 1 and ps[0][1:4] == (0, nkb, 0)
    tiles, nks = tm * tn, nkb // ksub
    waves = tiles // clusters if tiles >= clusters else 0
    S = tiles - (waves - 1) * clusters
    chained = (tiles >= clusters and tiles % clusters and nkb % ksub == 0 and nks >= 8
               and 3 * S >= 4 * clusters and 2 * S <= 3 * clusters)
    equal = _schedule(tm, tn, group, nkb, ksub, clusters, 1)
    if not chained:
        assert sched == equal
        return
    n3 = 3 * clusters - 2 * S
    for cid, units in enumerate(sched):
        sk_units = units[waves - 1:]
        assert all(u[2] == 0 and u[3] == nkb and u[4] == 0 for u in units[:waves - 1])
        shared = [u for u in sk_units if u[4]]
        assert len(sk_units) <= 2 and len(shared) <= 2
        work = sum(u[3] - u[2] for u in sk_units) // ksub
        want = (4 * nks) / 3 if cid < 3 * n3 else (3 * nks) / 2
        assert abs(work - want) < 1, (cid, work, want)
        # the wait (if any) comes first or after the leaving piece, and at most
        # one unit follows it, as in the equal layout
        waits = [i for i, u in enumerate(units) if u[4] and u[5] == 0]
        leaves = [i for i, u in enumerate(units) if u[4] and u[5] == 1]
        assert all(i == waves - 1 for i in leaves)
        assert all(i == waves - 1 + len(leaves) for i in waits)


# ------------------------------------------------------------------ decode ring
def test_decode_ring_fits_and_never_lets_a_warp_run_a_phase_ahead():
    """The bulk-copy decode form's ring, over every row count, K (multiples
    of 8 up to 20 000) and columns per block: a block's shared memory stays
    within the 227 KB a CTA may have, stage fills stay below the mbarrier's
    transaction limit, and either every column has a slot of its own or the
    stages are eight columns wide (one per consumer warp), so that a warp's
    parity waits see every phase in turn."""
    n_taken = 0
    for M in (1, 2, 3, 4):
        mm = 1 if M == 1 else 2 if M == 2 else 4
        for K in range(8, 20001, 8):
            for cpb in (1, 2, 3, 5, 8, 9, 16, 17, 25, 27, 31, 32):
                stages, cps, smem = pkg.gemm_decode_ring(M, K, cpb)
                assert stages >= 0
                if not (stages * cps >= cpb or stages >= 2):
                    continue  # the planner keeps the split-K form
                n_taken += 1
                assert smem == 256 + mm * 2 * K + stages * cps * 2 * K
                assert smem <= 227 * 1024, (M, K, cpb, stages, cps)
                assert 1 <= stages <= 12
                assert stages * cps >= cpb or cps == 8, (M, K, cpb, stages, cps)
                assert cps * 2 * K < 1 << 20 and M * 2 * K < 1 << 20
    assert n_taken > 50_000
    # the 4096-column decode shape: 27 columns per block, one slot each
    assert pkg.gemm_decode_ring(1, 4096, 27)[:2] == (9, 3)


def test_decode_ring_rejects_bad_arguments():
    for args in ((0, 4096, 27), (5, 4096, 27), (1, 0, 27), (1, 4096, 0), (1, 4096, 33)):
        assert pkg.gemm_decode_ring(*args)[0] == pkg.GEMM_ERR_INVALID_ARG


# ------------------------------------------------------------------ single-CTA kernel work schedule
CTA_SCHEDULES = [  # tiles_m, tiles_n, group, num_kb, splits, grid, stream_k
    (64, 1, 8, 64, 1, 152, True),     # (8192, 128, 4096) at 128 x 128 tiles
    (1, 64, 8, 128, 1, 152, True),    # (64, 8192, 8192)
    (8, 16, 8, 16, 1, 152, True),     # 1000^3 at 128 x 64 tiles
    (3, 5, 2, 7, 1, 100, True),       # at most one CTA per iteration
    (3, 5, 2, 7, 1, 105, True),       # exactly one iteration per CTA
    (2, 2, 8, 4, 1, 5, True),         # runs longer than a tile
    (10, 10, 4, 2, 1, 152, True),     # 200 iterations over 152 CTAs
    (4, 4, 8, 10, 3, 20, False),      # round-robin split-K
    (5, 3, 2, 9, 1, 7, False),        # round-robin, several waves
]


@pytest.mark.parametrize("tm,tn,g,nkb,splits,grid,sk", CTA_SCHEDULES)
def test_cta_schedule_covers_every_slice_once(tm, tn, g, nkb, splits, grid, sk):
    """Every (tile, K slice) is computed exactly once; a tile's pieces are
    ranked in K order and all know how many there are; the finishing piece
    (rank 0) is the last unit of its CTA, every other piece is the first
    unit of its CTA (so it waits for nothing) and writes that CTA's slot,
    and the finishing CTA looks for each rank at the CTA that holds it."""
    seen = {}
    pieces = {}
    slots = set()
    for c in range(grid):
        units = pkg.gemm_cta_schedule(tm, tn, g, nkb, splits, grid, sk, c)
        if sk:
            assert len(units) >= 1  # no CTA is left without work
        for i, (t, pm, pn, kb0, kb1, n, j, ws, pc) in enumerate(units):
            assert 0 <= t < tm * tn and 0 <= kb0 < kb1 <= nkb
            rc, em, en = pkg.gemm_raster_tile(t, tm, tn, min(g, tm))
            assert rc == 0 and (em, en) == (pm, pn)
            for kb in range(kb0, kb1):
                assert (t, kb) not in seen
                seen[(t, kb)] = c
            pieces.setdefault(t, []).append((kb0, kb1, n, j, ws, pc, c))
            if n > 1:
                assert pc == c
                if j == 0:
                    assert ws == -1 and i == len(units) - 1
                else:
                    assert ws == c and i == 0 and ws not in slots
                    slots.add(ws)
            else:
                assert ws == -1 and pc == -1
    assert len(seen) == tm * tn * nkb
    for t, ps in pieces.items():
        ps.sort()
        n = len(ps)
        if not sk:
            continue
        for j, (kb0, kb1, n_, j_, ws, pc, c) in enumerate(ps):
            assert n_ == n and j_ == j
        assert ps[0][0] == 0 and ps[-1][1] == nkb
        assert all(ps[i][1] == ps[i + 1][0] for i in range(n - 1))


def test_cta_schedule_rejects_bad_arguments():
    assert pkg.load().gemm_cta_schedule(2, 2, 8, 4, 1, 17, 1, 0, 0, None) == \
        pkg.GEMM_ERR_INVALID_ARG  # more CTAs than iterations
    assert pkg.load().gemm_cta_schedule(2, 2, 8, 4, 1, 4, 1, 4, 0, None) == \
        pkg.GEMM_ERR_INVALID_ARG
