"""Pins of the oracle's top-k truncation (no GPU needed).

The reading: the threshold of a row is its k-th largest value (NaN ranks as
-inf), every column at least that large is kept (ties at the threshold all
stay), the kept columns are renormalised, and target and draft rows of a
sequence are truncated alike. k <= 0 or k >= V keeps the row whole.

The expected values come from numpy sorts and scipy's softmax on masked rows,
from the greedy verify (which top-k = 1 must reproduce), and from the
acceptance-rate closed form evaluated on distributions truncated in numpy.
"""
import numpy as np
import pytest
import scipy.special
import scipy.stats

from speculative_decoding_verification_38_gb300 import workloads as wl


def _np_threshold(vals, k):
    v = np.where(np.isnan(vals), -np.inf, vals.astype(np.float64))
    V = v.shape[0]
    if k < 1 or k >= V:
        return -np.inf
    return float(np.sort(v)[::-1][k - 1])


def _np_trunc_softmax(logits, T, k):
    l64 = logits.astype(np.float64)
    tau = _np_threshold(l64, k)
    z = np.where(l64 >= tau, l64 / T, -np.inf)
    return scipy.special.softmax(z)


def _np_trunc_probs(q, k):
    q64 = q.astype(np.float64)
    tau = _np_threshold(q64, k)
    kept = np.where(q64 >= tau, q64, 0.0)
    return kept / kept.sum()


def _rows_with_ties(rng, V):
    """Integer-valued logits (many exact ties), a few -inf and one NaN."""
    x = rng.integers(-6, 7, size=V).astype(np.float32)
    x[rng.choice(V, size=3, replace=False)] = -np.inf
    return x


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_threshold_matches_sort(orc, dtype):
    rng = np.random.default_rng(3)
    for trial in range(40):
        V = int(rng.integers(2, 300))
        x = (2.0 * rng.standard_normal(V)).astype(np.float32) if trial % 2 else _rows_with_ties(rng, V)
        if trial % 5 == 0:
            x[int(rng.integers(0, V))] = np.nan
        row = wl.bf16_bits(x) if dtype == "bf16" else x
        stored = wl.stored_f32(row)
        for k in {-3, 0, 1, 2, V // 2, V - 1, V, V + 4, int(rng.integers(1, V + 1))}:
            got = orc.topk_threshold(row, k)
            ref = _np_threshold(stored, k)
            assert got == ref, (trial, V, k, got, ref)


@pytest.mark.parametrize("T", [1.0, 0.7, 1.9])
def test_softmax_topk_matches_masked_scipy(orc, T):
    rng = np.random.default_rng(5)
    T32 = float(np.float32(T))
    for trial in range(30):
        V = int(rng.integers(3, 500))
        x = (2.5 * rng.standard_normal(V)).astype(np.float32)
        if trial % 3 == 0:
            x = np.round(x)  # exact ties, some of them at the threshold
        for k in (1, 2, 5, V // 3 + 1, V - 1):
            tau = orc.topk_threshold(x, k)
            st, p = orc.softmax_row_topk(x, T32, tau)
            assert st == orc.SEQ_OK
            ref = _np_trunc_softmax(x, T32, k)
            assert np.max(np.abs(p - ref)) < 1e-14
            kept = x.astype(np.float64) >= _np_threshold(x, k)
            assert kept.sum() >= k  # ties can only widen the kept set
            assert np.all(p[~kept] == 0.0) and np.all(p[kept] > 0.0)


def test_topk_off_and_full_width_equal_plain_softmax(orc):
    rng = np.random.default_rng(6)
    x = (3 * rng.standard_normal(257)).astype(np.float32)
    _, plain = orc.softmax_row(x, 0.8)
    for k in (-1, 0, 257, 258, 10**6):
        tau = orc.topk_threshold(x, k)
        assert tau == -np.inf
        _, p = orc.softmax_row_topk(x, 0.8, tau)
        assert np.max(np.abs(p - plain)) < 1e-16
    # k = V - 1 drops exactly the smallest column (values are distinct)
    tau = orc.topk_threshold(x, 256)
    _, p = orc.softmax_row_topk(x, 0.8, tau)
    assert p[np.argmin(x)] == 0.0 and np.count_nonzero(p) == 256


def test_k_one_keeps_every_tie_of_the_maximum(orc):
    x = np.array([1.0, 3.0, -2.0, 3.0, 0.5, 3.0, -np.inf], np.float32)
    tau = orc.topk_threshold(x, 1)
    assert tau == 3.0
    _, p = orc.softmax_row_topk(x, 1.3, tau)
    np.testing.assert_allclose(p, [0, 1 / 3, 0, 1 / 3, 0, 1 / 3, 0], rtol=0, atol=1e-16)
    # a tie at the k-th place keeps both: k = 2 here keeps the same three columns
    assert orc.topk_threshold(x, 2) == 3.0 and orc.topk_threshold(x, 4) == 1.0


def test_normalize_topk_matches_numpy(orc):
    rng = np.random.default_rng(8)
    for trial in range(20):
        V = int(rng.integers(2, 200))
        q = rng.dirichlet(np.ones(V)).astype(np.float32)
        if trial % 4 == 0:
            q[: V // 2] = q[0]  # ties
        for k in (1, 3, V - 1, V):
            _, got = orc.normalize_row_topk(q, orc.topk_threshold(q, k))
            assert np.max(np.abs(got - _np_trunc_probs(q, k))) < 1e-15


def _workload(tgt, dft, gammas, toks, **kw):
    gammas = np.asarray(gammas, np.int32)
    return wl.Workload(
        name="tiny-topk", batch=len(gammas), vocab=tgt.shape[1], gamma_max=int(gammas.max()),
        gammas=gammas, target=np.ascontiguousarray(tgt, np.float32),
        draft=np.ascontiguousarray(dft, np.float32), draft_tokens=np.asarray(toks, np.int32), **kw)


def test_accept_terms_and_residual_per_sequence_k(orc):
    """p_i(x), q_i(x) and the residual weights under a per-sequence k, against
    numpy truncations of the stored rows."""
    rng = np.random.default_rng(9)
    V, g = 40, 3
    ks = np.array([0, 1, 4, 17, V - 1, V], np.int32)
    B = ks.shape[0]
    tgt = np.round(2 * rng.standard_normal((B * (g + 1), V))).astype(np.float32)  # ties
    dft = (2 * rng.standard_normal((B * g, V))).astype(np.float32)
    toks = rng.integers(0, V, size=B * g)
    w = _workload(tgt, dft, np.full(B, g), toks, temperature=0.9, top_ks=ks)
    T = float(np.float32(0.9))
    for b in range(B):
        for i in range(g + 1):
            pref = _np_trunc_softmax(tgt[b * (g + 1) + i], T, ks[b])
            st, p, q, wt, z = orc.position_rows(w, b, i)
            assert st == 0 and np.max(np.abs(p - pref)) < 1e-14
            if i == g:
                continue
            qref = _np_trunc_softmax(dft[b * g + i], T, ks[b])
            assert np.max(np.abs(q - qref)) < 1e-14
            r = np.maximum(0.0, pref - qref)
            assert abs(z - r.sum()) < 1e-13 and np.max(np.abs(wt - r)) < 1e-13
            st, px, qx = orc.accept_terms(w, b, i)
            x = toks[b * g + i]
            assert abs(px - pref[x]) < 1e-14 and abs(qx - qref[x]) < 1e-14
    # the scalar top_k applies to every sequence when top_ks is absent
    w1 = _workload(tgt, dft, np.full(B, g), toks, temperature=0.9, top_k=4)
    for b in range(B):
        _, p, q, _, _ = orc.position_rows(w1, b, 0)
        assert np.max(np.abs(p - _np_trunc_softmax(tgt[b * (g + 1)], T, 4))) < 1e-14


def test_sampling_with_k_one_is_greedy(orc):
    """k = 1 with distinct maxima turns both models into point masses at their
    argmax: a draft that proposes its argmax is accepted exactly while it
    matches the target's argmax, the rejection and the bonus emit the target's
    argmax. The sampled verify must then give the greedy verify's output."""
    rng = np.random.default_rng(10)
    gam = rng.integers(0, 7, size=400)
    tro, dro = wl.offsets_for(gam)
    V = 33
    tgt = rng.standard_normal((tro[-1], V)).astype(np.float32)
    dft = rng.standard_normal((dro[-1], V)).astype(np.float32)
    # make the draft agree with the target on a prefix of random length
    for b in range(400):
        agree = int(rng.integers(0, gam[b] + 1))
        for i in range(agree):
            dft[dro[b] + i] = tgt[tro[b] + i] + 0.01 * rng.standard_normal(V).astype(np.float32)
    toks = np.argmax(dft, axis=1)
    kw = dict(target_row_off=tro, draft_row_off=dro)
    ws = _workload(tgt, dft, gam, toks, top_k=1, **kw)
    wg = _workload(tgt, dft, gam, toks, greedy=True, **kw)
    rs = orc.verify_sample(ws, seed=17, rnd=2, nthreads=4)
    rg = orc.verify_greedy(wg)
    assert np.array_equal(rs["accepted"], rg["accepted"])
    assert np.array_equal(rs["tokens"], rg["tokens"])
    assert rs["accepted"].max() > 0 and (rs["accepted"] < gam).any()


def _expected_tokens(alpha, gamma):
    return (1 - alpha ** (gamma + 1)) / (1 - alpha)


def test_acceptance_rate_of_truncated_pair(orc):
    """i.i.d. positions, target logits log p and draft probabilities q, both
    truncated to k = 4 of V = 10: the mean emitted tokens per round follows
    the closed form at alpha' = sum min(p', q') of the numpy truncations, and
    the first emitted token follows p'. Truncating only one side would move
    the mean by far more than the 1% tolerance (checked below)."""
    rng = np.random.default_rng(11)
    V, k, gamma, B = 10, 4, 4, 100_000
    p = rng.dirichlet(np.ones(V) * 0.7)
    q = rng.dirichlet(np.ones(V) * 0.7)
    lp = np.log(p).astype(np.float32)
    pt = _np_trunc_softmax(lp, 1.0, k)
    qt = _np_trunc_probs(q.astype(np.float32), k)
    alpha = float(np.minimum(pt, qt).sum())
    E = _expected_tokens(alpha, gamma)
    q32 = q.astype(np.float64) / q.astype(np.float32).astype(np.float64).sum()
    alpha_one_side = float(np.minimum(pt, q32).sum())
    assert abs(_expected_tokens(alpha_one_side, gamma) - E) / E > 0.05
    cq = np.cumsum(qt)
    toks = np.minimum(np.searchsorted(cq, rng.random(B * gamma) * cq[-1], side="right"), V - 1)
    tgt = np.broadcast_to(lp, (B * (gamma + 1), V))
    dft = np.broadcast_to(q.astype(np.float32), (B * gamma, V))
    w = _workload(tgt, dft, np.full(B, gamma), toks, draft_is_probs=True, top_k=k)
    res = orc.verify_sample(w, seed=23, rnd=1, nthreads=8)
    emitted = res["accepted"] + 1
    assert abs(emitted.mean() - E) / E < 0.01, (emitted.mean(), E)
    first = res["tokens"].reshape(B, gamma + 1)[:, 0]
    c = np.bincount(first, minlength=V)
    assert np.all(c[pt == 0] == 0)
    keep = pt > 0
    assert scipy.stats.chisquare(c[keep], B * pt[keep]).pvalue > 1e-3
