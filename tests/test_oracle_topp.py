"""Pins of the oracle's top-p (nucleus) truncation, after top-k or alone (no GPU).

The threshold tau is fixed by two inequalities on the top-k-kept
distribution: the columns at or above tau carry at least top_p of the mass,
the columns strictly above tau carry less. The tests check those (with
scipy's softmax for the masses), the limits, ties, top-p with top-k off
(the whole row's nucleus), and the acceptance-rate closed form on numpy-truncated
pairs.
"""
import numpy as np
import pytest
import scipy.special

from speculative_decoding_verification_38_gb300 import workloads as wl


def _masses(vals, T, tau_k, probs):
    kept = vals >= tau_k
    if probs:
        w = np.where(kept, vals, 0.0)
    else:
        w = scipy.special.softmax(np.where(kept, vals / T, -np.inf))
    return w / w.sum()


@pytest.mark.parametrize("probs", [False, True])
def test_threshold_is_the_nucleus_boundary(orc, probs):
    rng = np.random.default_rng(2 + probs)
    for trial in range(60):
        V = int(rng.integers(2, 600))
        if probs:
            x = rng.dirichlet(np.ones(V) * 0.3).astype(np.float32)
        else:
            x = (2.0 * rng.standard_normal(V)).astype(np.float32)
        if trial % 3 == 0:
            x = np.round(x * (4 if not probs else 400)) / (4 if not probs else 400)  # ties
            x = x.astype(np.float32)
        T = float(np.float32(rng.uniform(0.5, 1.5)))
        k = int(rng.integers(1, V + 1))
        tau_k = orc.topk_threshold(x, k)
        for top_p in (1e-6, 0.1, 0.5, 0.9, 0.99, float(np.float32(rng.uniform(0.01, 0.99)))):
            tau = orc.topp_threshold(x, T, tau_k, top_p, probs=probs)
            v = x.astype(np.float64)
            w = _masses(v, T, tau_k, probs)
            assert tau >= tau_k
            assert w[v >= tau].sum() >= top_p - 1e-12
            assert w[v > tau].sum() < top_p + 1e-12
            assert np.any(v == tau)  # a value of the row


def test_limits(orc):
    x = np.array([3.0, 1.0, 2.0, 2.0, -1.0], np.float32)
    assert orc.topp_threshold(x, 1.0, -np.inf, 1.0) == -np.inf  # off: top-k's threshold comes back
    assert orc.topp_threshold(x, 1.0, 1.0, 1.5) == 1.0
    assert orc.topp_threshold(x, 1.0, -np.inf, float("nan")) == -np.inf
    assert orc.topp_threshold(x, 1.0, -np.inf, 0.0) == -np.inf  # zero means off
    assert orc.topp_threshold(x, 1.0, -np.inf, -2.0) == -np.inf
    assert orc.topp_threshold(x, 1.0, -np.inf, 1e-9) == 3.0  # a tiny p keeps the largest group
    # the tie group at 2.0 enters whole: 3 alone is below 0.9, 3 + both 2s reach it
    w = scipy.special.softmax(x.astype(np.float64))
    p = float(w[0] + w[2] + w[3] - 1e-9)
    assert orc.topp_threshold(x, 1.0, -np.inf, p) == 2.0
    st, q = orc.softmax_row_topk(x, 1.0, 2.0)
    assert np.count_nonzero(q) == 3


def _wl(tgt, dft, gammas, toks, **kw):
    gammas = np.asarray(gammas, np.int32)
    return wl.Workload(name="tiny-topp", batch=len(gammas), vocab=tgt.shape[1], gamma_max=int(gammas.max()),
                       gammas=gammas, target=np.ascontiguousarray(tgt, np.float32),
                       draft=np.ascontiguousarray(dft, np.float32), draft_tokens=np.asarray(toks, np.int32), **kw)


def test_top_p_without_top_k_is_the_whole_row_nucleus(orc):
    """With top-k off (k <= 0 or k >= V) an active top-p takes the nucleus of
    the whole row: the position rows are the softmax over the columns at or
    above topp_threshold(row, T, -inf, p), every status OK; p outside (0, 1)
    (or NaN) leaves the row whole."""
    rng = np.random.default_rng(4)
    V, g, B = 30, 3, 6
    tgt = rng.standard_normal((B * (g + 1), V)).astype(np.float32)
    dft = rng.standard_normal((B * g, V)).astype(np.float32)
    toks = rng.integers(0, V, size=B * g)
    ks = np.array([0, 5, V, 5, 0, 5], np.int32)
    ps = np.array([0.9, 0.9, 0.5, 1.0, 0.0, np.nan], np.float32)
    w = _wl(tgt, dft, np.full(B, g), toks, top_ks=ks, top_ps=ps)
    res = orc.verify_sample(w, seed=1)
    assert res["status"].tolist() == [0] * B
    for b in (0, 2, 4):
        for i in range(g + 1):
            st, p, q, wt, Z = orc.position_rows(w, b, i)
            vals = tgt[b * (g + 1) + i].astype(np.float64)
            tau = orc.topp_threshold(tgt[b * (g + 1) + i], 1.0, -np.inf, float(ps[b]))
            ref = scipy.special.softmax(np.where(vals >= tau, vals, -np.inf))
            assert st == 0 and np.max(np.abs(p - ref)) < 1e-14
            if b == 4:
                assert tau == -np.inf  # p = 0: off
            else:
                kept = ref[vals >= tau]
                assert kept.sum() > 0 and np.count_nonzero(vals >= tau) < V
                # the nucleus of the whole row, from its definition: tau is one of
                # the row's values, the columns at or above it carry at least p of
                # the softmax mass, the columns strictly above it less
                full = scipy.special.softmax(vals)
                assert tau in vals
                assert full[vals >= tau].sum() >= ps[b] - 1e-12 and full[vals > tau].sum() < ps[b]
    # the greedy verify ignores top-p
    assert orc.verify_greedy(_wl(tgt, dft, np.full(B, g), toks, top_ks=ks, top_ps=ps, greedy=True))[
        "status"].tolist() == [0] * B


def test_position_rows_follow_the_nucleus(orc):
    rng = np.random.default_rng(5)
    V, g, B = 50, 2, 4
    tgt = (2 * rng.standard_normal((B * (g + 1), V))).astype(np.float32)
    dft = (2 * rng.standard_normal((B * g, V))).astype(np.float32)
    toks = rng.integers(0, V, size=B * g)
    ks = np.array([20, 49, 3, 10], np.int32)
    ps = np.array([0.8, 0.5, 0.95, 0.3], np.float32)
    w = _wl(tgt, dft, np.full(B, g), toks, top_ks=ks, top_ps=ps, temperature=0.7)
    T = float(np.float32(0.7))
    for b in range(B):
        for i in range(g + 1):
            st, p, q, wt, Z = orc.position_rows(w, b, i)
            vals = tgt[b * (g + 1) + i].astype(np.float64)
            tau_k = orc.topk_threshold(tgt[b * (g + 1) + i], int(ks[b]))
            tau = orc.topp_threshold(tgt[b * (g + 1) + i], T, tau_k, float(ps[b]))
            ref = scipy.special.softmax(np.where(vals >= tau, vals / T, -np.inf))
            assert st == 0 and np.max(np.abs(p - ref)) < 1e-14
            assert (ref[vals >= tau_k][ref[vals >= tau_k] > 0]).size <= int(ks[b]) + 5


def test_acceptance_rate_of_nucleus_pair(orc):
    """i.i.d. positions with top-k 8 and top-p 0.7 on both rows: the mean
    emitted tokens follow the closed form at alpha' = sum min(p', q') of the
    truncated pair (built here from the boundary inequalities)."""
    rng = np.random.default_rng(6)
    V, k, top_p, gamma, B = 12, 8, 0.7, 4, 100_000
    p = rng.dirichlet(np.ones(V) * 0.6)
    q = rng.dirichlet(np.ones(V) * 0.6)
    lp = np.log(p).astype(np.float32)
    q32 = q.astype(np.float32)

    def nucleus(vals, probs):
        tau_k = orc.topk_threshold(vals, k)
        tau = orc.topp_threshold(vals, 1.0, tau_k, top_p, probs=probs)
        v = vals.astype(np.float64)
        w = _masses(v, 1.0, tau_k, probs)
        keep = v >= tau
        assert w[keep].sum() >= top_p and w[v > tau].sum() < top_p
        out = np.where(keep, w, 0.0)
        return out / out.sum()

    pt, qt = nucleus(lp, False), nucleus(q32, True)
    alpha = float(np.minimum(pt, qt).sum())
    E = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    cq = np.cumsum(qt)
    toks = np.minimum(np.searchsorted(cq, rng.random(B * gamma) * cq[-1], side="right"), V - 1)
    w = _wl(np.broadcast_to(lp, (B * (gamma + 1), V)), np.broadcast_to(q32, (B * gamma, V)), np.full(B, gamma), toks,
            draft_is_probs=True, top_k=k, top_p=top_p)
    res = orc.verify_sample(w, seed=9, rnd=1, nthreads=8)
    emitted = res["accepted"] + 1
    assert abs(emitted.mean() - E) / E < 0.01, (emitted.mean(), E)
    first = res["tokens"].reshape(B, gamma + 1)[:, 0]
    assert np.all(np.bincount(first, minlength=V)[pt == 0] == 0)


def test_whole_row_threshold_brute_force(orc):
    """topp_threshold over a whole row (tau_k = -inf) against brute force on
    small rows with ties: walk the groups of equal values from the largest
    down and stop at the first whose cumulative softmax mass reaches p."""
    rng = np.random.default_rng(21)
    for _ in range(300):
        V = int(rng.integers(1, 9))
        row = rng.choice(np.array([-3.0, -1.5, -1.0, 0.0, 0.5, 2.0], np.float32), size=V)
        T = float(rng.choice([0.5, 1.0, 1.7]))
        p = float(np.float32(rng.uniform(0.01, 0.99)))
        mass = scipy.special.softmax(row.astype(np.float64) / T)
        want = None
        for v in np.unique(row)[::-1]:
            if mass[row >= v].sum() >= p:
                want = v
                break
        got = orc.topp_threshold(row, T, -np.inf, p)
        assert got == want, (row, T, p, got, want)
