"""The work split of the decode-attention kernel, restated on the CPU (no GPU).

The block kernel lays the fixed 64-position blocks of every (sequence, KV head)
pair end to end (N blocks), gives grid block c of C the run
[c*N/C, (c+1)*N/C), and stores the partial state of pair p computed by grid
block c in slot c + p; the merge finds the grid blocks covering pair p with
cta_of(s) = ((s+1)*C - 1) / N. These tests check the arithmetic that argument
rests on: every fixed block lies in exactly one run, cta_of names it, the
covering blocks of a pair are exactly those from cta_of(first) to
cta_of(last) with a non-empty run, and no two (block, pair) pieces share a
slot, so the workspace of C_max + B*Hkv slots suffices.
"""
import numpy as np
import pytest

POS = 64


def nblocks(n):
    return (n + POS - 1) // POS


def runs(N, C):
    return [(c * N // C, (c + 1) * N // C) for c in range(C)]


def cta_of(s, N, C):
    return ((s + 1) * C - 1) // N


def pieces(lens, Hkv, C):
    """(grid block, pair) for every piece of work, by walking the runs."""
    starts, p = [], 0
    for b, n in enumerate(lens):
        for g in range(Hkv):
            starts.append((p, b * Hkv + g, nblocks(n)))
            p += nblocks(n)
    N = p
    owner = {}
    for c, (lo, hi) in enumerate(runs(N, C)):
        for s in range(lo, hi):
            pair = next(pr for st, pr, nb in starts if st <= s < st + nb)
            owner.setdefault((c, pair), []).append(s)
    return N, starts, owner


CASES = [((32768,), 2, 152), ((100,), 2, 152), ((1,), 2, 152), ((0, 130, 4097), 2, 152),
         ((4096, 32768, 1, 17000, 65536, 8191, 777, 20000), 2, 152), ((64, 64, 64), 1, 3),
         (tuple(np.random.default_rng(7).integers(0, 700, size=37)), 2, 152), ((5000,), 4, 7)]


@pytest.mark.parametrize("lens,Hkv,C", CASES)
def test_runs_partition_and_slots_are_unique(lens, Hkv, C):
    lens = [int(x) for x in lens]
    N, starts, owner = pieces(lens, Hkv, C)
    R = runs(N, C)
    # every fixed block in exactly one run, and cta_of names that run
    seen = np.zeros(N, dtype=int)
    for c, (lo, hi) in enumerate(R):
        seen[lo:hi] += 1
        for s in range(lo, hi):
            assert cta_of(s, N, C) == c
    assert np.all(seen == 1)
    # slots c + pair never collide, and stay below C + B*Hkv
    slots = [c + pair for (c, pair) in owner]
    assert len(slots) == len(set(slots))
    assert max(slots, default=0) < C + len(lens) * Hkv
    # the covering blocks of each pair: cta_of(first) .. cta_of(last), non-empty runs only
    for st, pair, nb in starts:
        want = sorted(c for (c, pr) in owner if pr == pair)
        if nb == 0:
            assert want == []
            continue
        c0, c1 = cta_of(st, N, C), cta_of(st + nb - 1, N, C)
        got = [c for c in range(c0, c1 + 1) if R[c][0] != R[c][1]]
        assert got == want, (pair, got, want)
