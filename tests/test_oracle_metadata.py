"""Pins for the split-KV schedule restatement and its invariant checker (CPU)."""
import numpy as np
import pytest

from oracle import metadata as M


def _rand_seqlens(rng, B, lo, hi, zero_frac=0.0):
    L = rng.integers(lo, hi + 1, size=B)
    if zero_frac:
        L[rng.random(B) < zero_frac] = 0
    return [int(x) for x in L]


@pytest.mark.parametrize("B,parts,lo,hi,zf", [
    (1, 1, 1, 100, 0.0), (2, 76, 100, 257, 0.0), (64, 76, 1, 8192, 0.0),
    (128, 38, 4096, 4096, 0.0), (256, 76, 2048, 16384, 0.0), (7, 3, 0, 300, 0.3),
    (300, 152, 0, 5000, 0.2), (5, 200, 1, 64, 0.0), (33, 1, 1, 1000, 0.1),
])
def test_schedule_meets_invariants(B, parts, lo, hi, zf):
    rng = np.random.default_rng(B * 1000 + parts)
    L = _rand_seqlens(rng, B, lo, hi, zf)
    md, ns = M.schedule(L, parts)
    M.check_metadata(L, md, ns)
    nb = M.n_blocks(L)
    W = sum(n + M.FIXED_COST for n in nb if n > 0)
    T = max(1, -(-(W + (parts - 1) * M.FIXED_COST) // parts))
    assert M.max_part_load(L, md) <= T


def test_skewed_long_sequence_is_split_and_balanced():
    L = [131072] + [1024] * 31
    md, ns = M.schedule(L, 76)
    M.check_metadata(L, md, ns)
    nb = M.n_blocks(L)
    W = sum(n + M.FIXED_COST for n in nb)
    T = -(-(W + 75 * M.FIXED_COST) // 76)
    assert ns[1] - ns[0] > 20                # the long sequence spans many parts
    assert M.max_part_load(L, md) <= T       # no part, the last included, exceeds T


def test_all_empty_sequences():
    L = [0, 0, 0]
    md, ns = M.schedule(L, 4)
    M.check_metadata(L, md, ns)
    assert list(ns) == [0, 0, 0, 0]
    assert (md[:, 5] == 0).all()


def test_single_part_takes_everything_unsplit():
    L = [5, 700, 64, 65]
    md, ns = M.schedule(L, 1)
    M.check_metadata(L, md, ns)
    assert list(ns) == [0, 1, 2, 3, 4]
    assert md[0, 5] == sum(M.n_blocks(L))


def _expect_fail(L, md, ns):
    with pytest.raises(AssertionError):
        M.check_metadata(L, md, ns)


def test_checker_rejects_planted_mistakes():
    L = [100, 1000, 3, 640]
    md, ns = M.schedule(L, 5)
    M.check_metadata(L, md, ns)
    # a part that stops one block early leaves a block uncovered
    bad = md.copy()
    p = next(p for p in range(4) if md[p, 5] > 1)
    bad[p, 3] -= 1
    bad[p, 5] -= 1
    _expect_fail(L, bad, ns)
    # overlapping ranges cover a block twice
    bad = md.copy()
    bad[p + 1, 1] = max(0, bad[p + 1, 1] - 1) if bad[p + 1, 0] == bad[p, 2] else bad[p + 1, 1]
    if (bad != md).any():
        bad[p + 1, 5] += 1
        _expect_fail(L, bad, ns)
    # wrong prefix sum
    bad_ns = ns.copy()
    bad_ns[2] += 1
    _expect_fail(L, md, bad_ns)
    # wrong first slot
    bad = md.copy()
    bad[1, 4] += 1
    _expect_fail(L, bad, ns)
    # a segment past the end of a sequence
    bad = md.copy()
    bad[-1, 2], bad[-1, 3] = len(L) - 1, M.n_blocks(L)[-1] + 1
    _expect_fail(L, bad, ns)


def test_brute_force_small_partitions():
    """On tiny inputs, enumerate the walk by hand-simple means: every block is
    handed out in order, and the splits of b count the parts that touch b."""
    rng = np.random.default_rng(7)
    for _ in range(200):
        B = int(rng.integers(1, 6))
        L = _rand_seqlens(rng, B, 0, 400, 0.2)
        parts = int(rng.integers(1, 9))
        md, ns = M.schedule(L, parts)
        M.check_metadata(L, md, ns)
        owners = {}
        for p in range(parts):
            for (b, lo, hi) in M.part_segments(md[p], L):
                for k in range(lo, hi):
                    owners[(b, k)] = p
        nb = M.n_blocks(L)
        prev = 0
        for b in range(B):
            for k in range(nb[b]):
                assert owners[(b, k)] >= prev      # parts are visited in order
                prev = owners[(b, k)]
            touch = {owners[(b, k)] for k in range(nb[b])}
            assert ns[b + 1] - ns[b] == len(touch)
