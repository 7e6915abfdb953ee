"""Pins of the oracle's n-gram (prompt-lookup) drafter (no GPU needed).

An independent vectorised search (numpy sliding windows) gives the expected
match on random contexts of a small vocabulary; hand cases pin the overlap,
the n fallback, the clipped continuation and the too-short contexts.
"""
import numpy as np
from numpy.lib.stride_tricks import sliding_window_view


def _np_draft(c, n_max, n_min, gamma):
    L = c.shape[0]
    for n in range(n_max, max(n_min, 1) - 1, -1):
        if L < n + 1:
            continue
        suffix = c[L - n:]
        win = sliding_window_view(c[:L - 1], n)  # starts 0 .. L - 1 - n
        hits = np.nonzero((win == suffix).all(axis=1))[0]
        if hits.size:
            j = int(hits.max())
            cont = c[j + n: j + n + gamma]
            return j, n, np.concatenate([cont, np.full(gamma - cont.size, -1, np.int32)])
    return -1, 0, np.full(gamma, -1, np.int32)


def test_random_contexts_match_sliding_windows(orc):
    rng = np.random.default_rng(3)
    for trial in range(60):
        B = int(rng.integers(1, 20))
        lens = rng.integers(0, 400, size=B)
        lens[0] = 0
        vocab = int(rng.choice([3, 8, 50, 5000]))
        ctx = rng.integers(0, vocab, size=int(lens.sum())).astype(np.int32)
        off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        n_max = int(rng.integers(1, 6))
        n_min = int(rng.integers(1, n_max + 1))
        gamma = int(rng.integers(0, 10))
        got = orc.ngram_draft(ctx, off, n_max, n_min, gamma)
        for b in range(B):
            j, n, d = _np_draft(ctx[off[b]:off[b + 1]], n_max, n_min, gamma)
            assert got["match_pos"][b] == j and got["match_n"][b] == n, (trial, b)
            assert np.array_equal(got["draft"][b], d), (trial, b)
            assert got["n_draft"][b] == int((d >= 0).sum())


def test_hand_cases(orc):
    def one(seq, n_max, n_min, gamma):
        r = orc.ngram_draft(np.array(seq, np.int32), [0, len(seq)], n_max, n_min, gamma)
        return int(r["match_pos"][0]), int(r["match_n"][0]), r["draft"][0].tolist(), int(r["n_draft"][0])

    # the latest earlier occurrence of the suffix "5 6", and what followed it
    assert one([5, 6, 7, 8, 5, 6, 9, 1, 5, 6], 2, 1, 4) == (4, 2, [9, 1, 5, 6], 4)
    # an occurrence may overlap the suffix: "a a" at 1 overlaps "a a" at 2
    assert one([1, 1, 1, 1], 2, 2, 3) == (1, 2, [1, -1, -1], 1)
    # no 3-gram repeats; the 2-gram "2 3" does
    assert one([2, 3, 4, 9, 2, 3], 3, 2, 2) == (0, 2, [4, 9], 2)
    # n_min above every match length: nothing
    assert one([2, 3, 4, 9, 2, 3], 3, 3, 2) == (-1, 0, [-1, -1], 0)
    # the continuation stops at the end of the context
    assert one([7, 8, 7], 1, 1, 5) == (0, 1, [8, 7, -1, -1, -1], 2)
    # too short for any n-gram plus a following token
    assert one([4], 1, 1, 3) == (-1, 0, [-1, -1, -1], 0)
    assert one([], 2, 1, 3) == (-1, 0, [-1, -1, -1], 0)
    assert one([4, 5], 2, 2, 1) == (-1, 0, [-1], 0)
    # gamma = 0 drafts nothing but still reports the match
    assert one([5, 6, 5], 1, 1, 0) == (0, 1, [], 0)
