"""CPU model check of the barrier protocol of the decode kernel's bulk-copy form.

The kernel (csrc/decode.cu, decode_bulk_kernel) hands ring stages between one
copy thread and eight consumer warps with mbarriers and parity waits:

* group j of cps columns goes to stage s = j % S in round r = j // S; before
  refilling a stage (j >= S) the copy thread waits for phase r - 1 of the
  stage's "empty" barrier, then arms phase r of its "full" barrier, which
  completes when the group's copies land;
* warp w reads the block's columns w, w + 8, ...: for column c in group j it
  waits for phase r of full[s], reads, and arrives on empty[s] (cps arrivals
  complete a phase).

A parity wait is only sound while the barrier is within one phase of the one
awaited: try_wait.parity(r & 1) reports phase r complete whenever the count of
completed phases differs in parity from r, so a count of r - 1 would pass too
early and a count of r + 2 would never pass.  This test replays the protocol
under random interleavings (copies landing at arbitrary times, warps and the
copy thread advancing in any order) for every ring shape the library plans
(taken from gemm_decode_ring, the compiled planner), and checks at every step
that (1) every waiter's barrier stays within {r, r + 1} completed phases,
(2) a stage is never refilled while a column of its previous group is unread,
(3) every column is read exactly once, after its copy landed, and (4) the
run never deadlocks.
"""
from __future__ import annotations

import random

import pytest

import dense_tiled_gemm_02_gb300 as pkg

WARPS = 8


def _replay(S: int, cps: int, ncols: int, rng: random.Random) -> None:
    groups = (ncols + cps - 1) // cps
    full_done = [0] * S      # completed phases of full[s]
    empty_done = [0] * S     # completed phases of empty[s]
    empty_arr = {}           # (s, round) -> arrivals so far
    in_flight = []           # groups issued whose copies have not landed
    landed = set()
    read = set()             # columns read
    nxt = 0                  # copy thread: next group
    cols = [list(range(w, ncols, WARPS)) for w in range(WARPS)]
    pos = [0] * WARPS

    def stage_round(j):
        return j % S, j // S

    while True:
        moves = []
        # the copy thread
        if nxt < groups:
            s, r = stage_round(nxt)
            if nxt >= S:
                c = empty_done[s]
                assert c in (r - 1, r), ("copy thread parity wait off by a phase", S, cps, ncols)
                if c >= r:
                    moves.append(("issue", None))
            else:
                moves.append(("issue", None))
        # copies landing, in any order
        for j in in_flight:
            moves.append(("land", j))
        # consumer warps
        for w in range(WARPS):
            if pos[w] < len(cols[w]):
                col = cols[w][pos[w]]
                s, r = stage_round(col // cps)
                c = full_done[s]
                assert c in (r, r + 1), ("consumer parity wait off by a phase", S, cps, ncols, w)
                if c >= r + 1:
                    moves.append(("read", w))
        if not moves:
            break
        kind, arg = rng.choice(moves)
        if kind == "issue":
            j = nxt
            s, r = stage_round(j)
            if j >= S:  # the previous group in this stage is fully read
                prev = j - S
                for col in range(prev * cps, min(ncols, prev * cps + cps)):
                    assert col in read, ("stage refilled before it was read", S, cps, ncols, j)
            in_flight.append(j)
            nxt += 1
        elif kind == "land":
            in_flight.remove(arg)
            s, r = stage_round(arg)
            assert full_done[s] == r, "full phases complete out of order"
            full_done[s] = r + 1
            landed.add(arg)
        else:
            w = arg
            col = cols[w][pos[w]]
            j = col // cps
            assert j in landed and col not in read
            read.add(col)
            pos[w] += 1
            s, r = stage_round(j)
            empty_arr[(s, r)] = empty_arr.get((s, r), 0) + 1
            if empty_arr[(s, r)] == cps:
                assert empty_done[s] == r, "empty phases complete out of order"
                empty_done[s] = r + 1
    assert nxt == groups and not in_flight, ("deadlock", S, cps, ncols)
    assert read == set(range(ncols)), ("deadlock or lost column", S, cps, ncols)


def _ring_shapes():
    shapes = set()
    for M in (1, 2, 3, 4):
        for K in (8, 264, 1032, 2048, 4096, 6144, 8192, 12288, 16384):
            for cpb in range(1, 33):
                stages, cps, _ = pkg.gemm_decode_ring(M, K, cpb)
                if stages * cps >= cpb or stages >= 2:  # the planner takes the form
                    shapes.add((stages, cps, cpb))
    return sorted(shapes)


def test_protocol_holds_for_every_planned_ring():
    shapes = _ring_shapes()
    assert (9, 3, 27) in shapes and (3, 8, 27) in shapes  # the 4096-column shapes
    rng = random.Random(2026)
    for S, cps, cpb in shapes:
        # a full block and the shorter last blocks of a grid
        for ncols in sorted({cpb, max(1, cpb - 1), max(1, cpb // 2), 1}):
            for _ in range(12):
                _replay(S, cps, ncols, rng)


@pytest.mark.parametrize("S,cps,ncols", [(2, 2, 9), (3, 4, 27), (2, 1, 5)])
def test_model_catches_a_phase_ahead_wait(S, cps, ncols):
    """The check is not vacuous: narrow stages with stage reuse (the shapes the
    planner avoids) let a warp that skipped a round wait a phase ahead."""
    with pytest.raises(AssertionError, match="parity wait off by a phase"):
        rng = random.Random(7)
        for _ in range(200):
            _replay(S, cps, ncols, rng)
