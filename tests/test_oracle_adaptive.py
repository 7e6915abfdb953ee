"""Pins of the oracle's adaptive-gamma functions (no GPU needed).

The speedup E / (1 + gamma c) is pinned to every worked value the pages print
(tests/golden/speedup_cases.txt, tests/golden/expected_tokens.txt at c = 0).
The choice of gamma is pinned by closed-form limits (alpha = 0, alpha = 1,
c = 0), by the pages' statements (a loss below break-even, the peak between
3 and 8 at alpha = 0.8), and by exact rational arithmetic on sampled cases.
The float32 acceptance average is pinned by numpy float32 arithmetic and by
its fixed point.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                yield line.split()


def test_speedup_printed_cases(orc):
    n = 0
    for parts in _rows("speedup_cases.txt"):
        a, g, c, printed, dec = float(parts[0]), int(parts[1]), float(parts[2]), float(parts[3]), int(parts[4])
        sp = orc.speedups(a, g, c)
        assert round(sp[g], dec) == printed, parts
        n += 1
    assert n == 6


def test_speedup_at_zero_cost_is_expected_tokens(orc):
    for parts in _rows("expected_tokens.txt"):
        a, g, printed, dec = float(parts[0]), int(parts[1]), float(parts[2]), int(parts[3])
        assert round(orc.speedups(a, g, 0.0)[g], dec) == printed, parts
    sp = orc.speedups(0.0, 8, 0.1)  # alpha = 0: one token per pass, cost 1 + g c
    np.testing.assert_allclose(sp, 1.0 / (1.0 + 0.1 * np.arange(9)), rtol=2e-7)
    sp = orc.speedups(1.0, 8, 0.0)  # alpha = 1: the limit g + 1
    assert np.array_equal(sp, np.arange(1, 10, dtype=np.float32))
    # the closed form at alpha near 1 (where it cancels) against exact rationals
    for a in (0.999, 0.9999, 0.5):
        a32 = float(np.float32(a))
        sp = orc.speedups(a32, 64, 0.0)
        fa = Fraction(a32)
        for g in (1, 8, 64):
            exact = float((1 - fa ** (g + 1)) / (1 - fa))
            assert abs(float(sp[g]) - exact) <= 1e-5 * exact, (a, g)


def _exact_best(alpha: Fraction, gmax: int, c: Fraction):
    """Best gamma in exact rational arithmetic, and the relative gap to the runner-up."""
    sp = []
    for g in range(gmax + 1):
        E = Fraction(g + 1) if alpha == 1 else (1 - alpha ** (g + 1)) / (1 - alpha)
        sp.append(E / (1 + g * c))
    best = max(range(gmax + 1), key=lambda g: (sp[g], -g))
    others = [sp[g] for g in range(gmax + 1) if g != best]
    gap = (sp[best] - max(others)) / sp[best] if others else Fraction(1)
    return best, gap


def test_best_gamma_matches_exact_rationals(orc):
    rng = np.random.default_rng(5)
    checked = 0
    for _ in range(400):
        a32 = np.float32(rng.uniform(0.0, 1.0))
        c32 = np.float32(rng.choice([0.0, 0.01, 0.02, 0.05, 0.1, 0.2, 0.3, 0.5]))
        gmax = int(rng.integers(0, 17))
        best, gap = _exact_best(Fraction(float(a32)), gmax, Fraction(float(c32)))
        if gap < Fraction(1, 10**5):
            continue  # a near tie: float32 may order it either way
        assert orc.best_gamma(float(a32), gmax, float(c32)) == best, (a32, c32, gmax)
        checked += 1
    assert checked > 350


def test_best_gamma_limits_and_page_statements(orc):
    assert orc.best_gamma(0.0, 8, 0.05) == 0      # nothing is ever accepted
    assert orc.best_gamma(0.3, 8, 0.0) == 8       # free drafts: the longest chain
    assert orc.best_gamma(1.0, 8, 0.5) == 8       # (g + 1) / (1 + g/2) rises with g
    assert orc.best_gamma(1.0, 8, 1.5) == 0       # (g + 1) / (1 + 1.5 g) falls with g
    assert orc.best_gamma(0.1, 8, 0.5) == 0       # below break-even at every g
    g = orc.best_gamma(0.8, 16, 0.05)             # "pick gamma about 3-8 where that ratio peaks"
    assert 3 <= g <= 8
    # the loss case printed at gamma = 4 (0.75x) still gains at gamma = 1
    sp = orc.speedups(0.4, 4, 0.3)
    assert sp[4] < 1.0 < sp[1] and orc.best_gamma(0.4, 4, 0.3) == 1
    assert orc.best_gamma(float("nan"), 8, 0.05) == 0  # NaN read as 0
    assert orc.best_gamma(1.7, 8, 0.05) == orc.best_gamma(1.0, 8, 0.05)  # clamped


def test_adapt_gamma_batch_switch(orc):
    ema = np.array([0.9, 0.8, 0.2, 0.0], np.float32)
    g, total = orc.adapt_gamma(ema, 8, 0.05)
    assert total == int((g + 1).sum())
    assert g[3] == 0 and g[0] >= g[1] >= g[2]
    g2, t2 = orc.adapt_gamma(ema, 8, 0.05, max_positions=total)  # exactly at the budget: kept
    assert np.array_equal(g2, g) and t2 == total
    g3, t3 = orc.adapt_gamma(ema, 8, 0.05, max_positions=total - 1)  # over it: speculation off
    assert np.all(g3 == 0) and t3 == total  # the positions reported are the ones compared


def test_acceptance_ema_float32_steps(orc):
    rng = np.random.default_rng(6)
    B, gmax = 300, 8
    gam = rng.integers(0, gmax + 1, size=B).astype(np.int32)
    acc = np.array([rng.integers(0, g + 1) for g in gam], np.int32)
    st = np.where(rng.random(B) < 0.1, 3, 0).astype(np.int32)
    ema = rng.random(B).astype(np.float32)
    lam = np.float32(0.125)
    got = orc.acceptance_ema(acc, gam, gmax, ema, lam, status=st)
    t = np.where(acc < gam, acc + 1, gam)
    want = ema.copy()
    upd = (st == 0) & (gam > 0)
    x = (acc[upd].astype(np.float32) / t[upd].astype(np.float32)).astype(np.float32)
    want[upd] = (ema[upd] + lam * (x - ema[upd])).astype(np.float32)
    assert np.array_equal(got, want)
    assert np.array_equal(got[~upd], ema[~upd])  # untouched
    # all accepted -> x = 1; first rejected -> x = 0
    one = orc.acceptance_ema([4], [4], 8, [0.5], 0.25)
    zero = orc.acceptance_ema([0], [4], 8, [0.5], 0.25)
    assert one[0] == np.float32(0.625) and zero[0] == np.float32(0.375)


def test_acceptance_ema_converges_to_test_success_rate(orc):
    """Rounds whose accept tests pass at a fixed fraction drive the average
    to that fraction: gamma = 4 and 2 accepted is 3 tests, 2 passed."""
    e = np.zeros(1, np.float32)
    for _ in range(400):
        e = orc.acceptance_ema([2], [4], 8, e, 0.1)
    assert abs(float(e[0]) - 2.0 / 3.0) < 1e-6
    # gamma = 0 rounds never move it; nor does a negative accepted count
    assert orc.acceptance_ema([0], [0], 8, e, 0.1)[0] == e[0]
    assert orc.acceptance_ema([-1], [4], 8, e, 0.1)[0] == e[0]
