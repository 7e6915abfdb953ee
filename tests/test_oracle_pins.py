"""Pins of the float64 oracle to things other than itself (no GPU needed).

Each test states what fixes the expected value: a number printed on the
pages (tests/golden/), a closed form, an identity from the pages' proof,
brute force on tiny inputs, or an independent library routine.
"""
import itertools
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import scipy.special
import scipy.stats

from speculative_decoding_verification_38_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            out[k] = [float(x) for x in v]
    return out


def _tiny_workload(target_rows, draft_rows, gammas, tokens, *, T=1.0, probs=False, kv=None,
                   block_size=0, temps=None, dtype=np.float32):
    gammas = np.asarray(gammas, dtype=np.int32)
    tro, dro = wl.offsets_for(gammas)
    uniform = bool(np.all(gammas == gammas.max()))
    return wl.Workload(
        name="tiny", batch=len(gammas), vocab=target_rows.shape[1], gamma_max=int(gammas.max()),
        gammas=gammas, target=np.ascontiguousarray(target_rows, dtype=dtype),
        draft=np.ascontiguousarray(draft_rows, dtype=dtype), draft_tokens=np.asarray(tokens, np.int32),
        draft_is_probs=probs, temperature=T, temperatures=temps, kv_in=kv, block_size=block_size,
        target_row_off=None if uniform else tro, draft_row_off=None if uniform else dro,
    )


# --------------------------------------------------------------------- Philox
TRITON_SCRIPT = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl
@triton.jit
def k(out_ptr, c0_ptr, c1_ptr, c2_ptr, c3_ptr, seed, N: tl.constexpr):
    o = tl.arange(0, N)
    c0 = tl.load(c0_ptr + o); c1 = tl.load(c1_ptr + o); c2 = tl.load(c2_ptr + o); c3 = tl.load(c3_ptr + o)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out_ptr + o * 4 + 0, a); tl.store(out_ptr + o * 4 + 1, b)
    tl.store(out_ptr + o * 4 + 2, c); tl.store(out_ptr + o * 4 + 3, d)
cases = json.loads(sys.argv[1])
res = []
for seed, ctrs in cases:
    n = len(ctrs)
    cols = [torch.tensor([c[j] for c in ctrs], dtype=torch.int64).to(torch.int32) for j in range(4)]
    out = torch.zeros(n * 4, dtype=torch.int32)
    k[(1,)](out, *cols, seed, N=n)
    res.append([x & 0xffffffff for x in out.tolist()])
print(json.dumps(res))
"""


def test_philox_matches_triton_reference():
    """The oracle's Philox4x32-10 equals Triton's independent implementation
    (run on the CPU through Triton's interpreter) for assorted keys/counters."""
    pytest.importorskip("triton")
    rng = np.random.default_rng(7)
    cases = []
    for seed in [0, 1, 0xDEADBEEF12345678, 2**64 - 1, int(rng.integers(0, 2**63))]:
        ctrs = [[int(x) for x in rng.integers(0, 2**32, size=4, dtype=np.uint64)] for _ in range(8)]
        ctrs[0] = [0, 0, 0, 0]
        ctrs[1] = [2**32 - 1] * 4
        cases.append([seed, ctrs])
    env = dict(os.environ, TRITON_INTERPRET="1")
    out = subprocess.run([sys.executable, "-c", TRITON_SCRIPT, json.dumps(cases)], env=env,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    ref = json.loads(out.stdout.strip().splitlines()[-1])
    import oracle
    for (seed, ctrs), words in zip(cases, ref):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for j, c in enumerate(ctrs):
            got = [int(x) for x in oracle.philox4x32_10(c, key)]
            assert got == words[4 * j:4 * j + 4], (seed, c)


def test_philox_known_answer_vectors(orc):
    """The oracle's Philox4x32-10 reproduces the published known-answer
    vectors of the SC'11 generator (zero, all-ones and pi-digit inputs;
    tests/golden/philox4x32_10_kat.txt)."""
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x, 16) for x in line.split()[1:]])
    assert len(rows) == 3
    for r in rows:
        ctr, key, want = r[0:4], r[4:6], r[6:10]
        assert [int(x) for x in orc.philox4x32_10(ctr, key)] == want


def test_uniform_pair_layout_and_uniformity(orc):
    """u = (w >> 8) * 2^-24 from words 0/1 of the block keyed (seed) with counter
    (pos, seq, round lo, round hi); 2^20 draws pass a 256-bin chi-square."""
    seed, rnd = 0x0123456789ABCDEF, (5 << 32) | 17
    w = orc.philox4x32_10([3, 9, 17, 5], [seed & 0xFFFFFFFF, seed >> 32])
    ua, us = orc.uniform_pair(seed, rnd, 9, 3)
    assert ua == (int(w[0]) >> 8) / 2**24 and us == (int(w[1]) >> 8) / 2**24
    # uniformity over many counters, checked as a histogram (word stream from the oracle)
    n = 1 << 14
    vals = []
    for s in range(n // 64):
        for p_ in range(64):
            a, b = orc.uniform_pair(11, 0, s, p_)
            vals.append(a)
            vals.append(b)
    vals = np.array(vals)
    assert vals.min() >= 0.0 and vals.max() < 1.0
    counts = np.histogram(vals, bins=256, range=(0, 1))[0]
    assert scipy.stats.chisquare(counts).pvalue > 1e-3


# --------------------------------------------------------------- distributions
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1.0, 0.8, 0.5, 1.7])
def test_softmax_matches_scipy(orc, dtype, T):
    rng = np.random.default_rng(1)
    x = (3.0 * rng.standard_normal(777)).astype(np.float32)
    row = wl.bf16_bits(x) if dtype == "bf16" else x
    T32 = float(np.float32(T))  # the library takes temperatures as float32
    st, p = orc.softmax_row(row, T32)
    assert st == orc.SEQ_OK
    ref = scipy.special.softmax(wl.stored_f32(row).astype(np.float64) / T32)
    assert np.max(np.abs(p - ref)) < 1e-14  # a few ulps of float64
    assert abs(p.sum() - 1.0) < 1e-13


def test_softmax_closed_forms(orc):
    # two logits: p_1 = logistic((l1 - l0) / T)
    for l0, l1, T in [(0.0, 1.0, 1.0), (2.5, -1.0, 0.8), (-3.0, -3.0, 1.3)]:
        T32 = float(np.float32(T))
        st, p = orc.softmax_row(np.array([l0, l1], dtype=np.float32), T32)
        assert abs(p[1] - 1.0 / (1.0 + math.exp((l0 - l1) / T32))) < 1e-15
    # equal logits give the uniform distribution; -inf entries get zero mass
    st, p = orc.softmax_row(np.zeros(10, np.float32), 0.9)
    assert np.allclose(p, 0.1, atol=1e-16, rtol=0)
    st, p = orc.softmax_row(np.array([0, -np.inf, 1, -np.inf], np.float32), 1.0)
    assert p[1] == 0.0 and p[3] == 0.0 and abs(p[2] - math.e / (1 + math.e)) < 1e-15


def test_softmax_invalid_rows(orc):
    assert orc.softmax_row(np.array([1, np.nan, 2], np.float32), 1.0)[0] == orc.SEQ_BAD_ROW
    assert orc.softmax_row(np.full(4, -np.inf, np.float32), 1.0)[0] == orc.SEQ_BAD_ROW
    assert orc.softmax_row(np.array([1, np.inf], np.float32), 1.0)[0] == orc.SEQ_BAD_ROW
    assert orc.softmax_row(np.array([1, 2], np.float32), 0.0)[0] == orc.SEQ_BAD_TEMP
    assert orc.softmax_row(np.array([1, 2], np.float32), -1.0)[0] == orc.SEQ_BAD_TEMP


def test_normalize_closed_form(orc):
    st, q = orc.normalize_row(np.array([1, 1, 2, 0], np.float32))
    assert st == 0 and np.array_equal(q, [0.25, 0.25, 0.5, 0.0])
    assert orc.normalize_row(np.zeros(3, np.float32))[0] == orc.SEQ_BAD_ROW


def test_bf16_read_matches_torch(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(4096) * 10.0 ** rng.integers(-30, 30, 4096)).astype(np.float32)
    bits = wl.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(bits, ref.view(torch.int16).numpy().view(np.uint16))
    ref64 = ref.to(torch.float64).numpy()
    for j in range(0, 4096, 97):
        assert orc.value(bits, j) == ref64[j]


# ------------------------------------------------------------------- residual
def test_residual_page_worked_example(orc):
    """p = [.5,.3,.15,.05] and uniform q from the page's statistical check:
    Z = 0.3 = 1 - 0.700 and norm(max(0, p - q)) = [5/6, 1/6, 0, 0]."""
    g = _golden_kv("p1_worked_example.txt")
    p, q = np.array(g["p"]), np.array(g["q"])
    r, Z = orc.residual(p, q)
    assert abs(Z - g["Z"][0]) < 1e-15
    assert abs((1.0 - np.minimum(p, q).sum()) - g["Z"][0]) < 1e-15
    assert abs(np.minimum(p, q).sum() - g["alpha"][0]) < 1e-15
    assert np.allclose(r / Z, g["residual_normalised"], atol=1e-15, rtol=0)


def test_residual_identity_random(orc):
    """Z = sum max(0, p - q) = 1 - sum min(p, q) and min(p, q) + r = p (the
    proof's two cases), to 1e-12 on random Dirichlet pairs."""
    rng = np.random.default_rng(5)
    for V in [2, 3, 8, 1000]:
        for _ in range(20):
            p, q = rng.dirichlet(np.ones(V) * 0.5), rng.dirichlet(np.ones(V) * 0.5)
            r, Z = orc.residual(p, q)
            assert abs(Z - (1.0 - np.minimum(p, q).sum())) < 1e-12
            assert np.max(np.abs(np.minimum(p, q) + r - p)) < 1e-15
            assert np.all(r >= 0)


# ------------------------------------------------------------------ inverse CDF
def test_inverse_cdf_measure_on_dyadic_grid(orc):
    """With dyadic weights every grid point u = k / 2^12 is exact, so the number
    of grid points mapped to j must equal w_j * 2^12 exactly, and zero-mass
    entries are never returned."""
    w = np.array([0, 3, 0, 5, 8, 0, 1, 15], dtype=np.float64) / 32.0
    M = 1 << 12
    counts = np.zeros(w.shape[0], dtype=np.int64)
    for k in range(M):
        counts[orc.inverse_cdf(w, k / M)] += 1
    assert np.array_equal(counts, (w * M).astype(np.int64))
    # unnormalised input is tolerated: the same measure at 7x the scale
    counts2 = np.zeros_like(counts)
    for k in range(M):
        counts2[orc.inverse_cdf(7.0 * w, k / M)] += 1
    assert np.array_equal(counts2, counts)


def test_inverse_cdf_edges(orc):
    w = np.array([0.0, 0.25, 0.0, 0.75, 0.0])
    assert orc.inverse_cdf(w, 0.0) == 1
    assert orc.inverse_cdf(w, 0.25) == 3
    assert orc.inverse_cdf(w, 1.0 - 2**-24) == 3
    assert orc.cdf_edges(w, 3) == (0.25, 1.0)
    # u = 1 is outside the uniform's range; the fallback is the last index with mass
    assert orc.inverse_cdf(w, 1.0) == 3


# ----------------------------------------------------------------------- argmax
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_argmax_matches_numpy_with_ties_and_nan(orc, dtype):
    rng = np.random.default_rng(9)
    for trial in range(200):
        V = int(rng.integers(1, 300))
        x = rng.integers(-5, 5, size=V).astype(np.float32)  # many exact ties
        if trial % 3 == 0:
            x[rng.integers(0, V, size=max(1, V // 7))] = np.nan
        if trial % 11 == 0:
            x[:] = -np.inf
        row = wl.bf16_bits(x) if dtype == "bf16" else x
        vals = wl.stored_f32(row).astype(np.float64)
        ref = int(np.argmax(np.where(np.isnan(vals), -np.inf, vals)))
        assert orc.argmax_row(row) == ref


# ------------------------------------------------------------ exact enumeration
def _enumerate_string_dist(P, Q, gamma, L, orc):
    """Exact distribution of the first L emitted tokens when every round starting
    at stream position t drafts x_i ~ Q[t+i], accepts with min(1, P/Q) and draws
    the residual at the first rejection (bonus from P[t+gamma])."""
    V = P.shape[1]
    dist = {}
    resid = {}
    for t in range(P.shape[0]):
        if t < Q.shape[0]:
            r, Z = orc.residual(P[t], Q[t])
            resid[t] = r / Z if Z > 0 else P[t]

    def add(prefix, prob):
        key = tuple(prefix[:L])
        dist[key] = dist.get(key, 0.0) + prob

    def round_from(t, prefix, prob):
        if t >= L:
            add(prefix, prob)
            return
        step(t, 0, prefix, prob)

    def step(t, i, prefix, prob):
        pos = t + i
        if pos >= L:
            add(prefix, prob)
            return
        if i == gamma:
            for z in range(V):
                if P[pos, z] > 0:
                    round_from(pos + 1, prefix + [z], prob * P[pos, z])
            return
        for x in range(V):
            qx = Q[pos, x]
            if qx == 0:
                continue
            acc = min(1.0, P[pos, x] / qx)
            if acc > 0:
                step(t, i + 1, prefix + [x], prob * qx * acc)
            if acc < 1:
                for z in range(V):
                    if resid[pos][z] > 0:
                        round_from(pos + 1, prefix + [z], prob * qx * (1 - acc) * resid[pos][z])

    round_from(0, [], 1.0)
    return dist


@pytest.mark.parametrize("V,gamma,L", [(2, 1, 4), (3, 2, 4), (4, 3, 4), (8, 2, 3), (5, 3, 4)])
def test_exact_enumeration_equals_target(orc, V, gamma, L):
    """P(y_1..y_L) = prod_t p^(t)(y_t) to 1e-12, position-dependent p and q."""
    rng = np.random.default_rng(100 + V * 10 + gamma)
    npos = L + gamma + 1
    P = np.array([orc.softmax_row((2 * rng.standard_normal(V)).astype(np.float32), 0.9)[1]
                  for _ in range(npos)])
    Q = np.array([orc.softmax_row((2 * rng.standard_normal(V)).astype(np.float32), 0.9)[1]
                  for _ in range(npos)])
    dist = _enumerate_string_dist(P, Q, gamma, L, orc)
    total = 0.0
    for ys in itertools.product(range(V), repeat=L):
        ref = float(np.prod([P[t, y] for t, y in enumerate(ys)]))
        got = dist.get(ys, 0.0)
        assert abs(got - ref) < 1e-12, (ys, got, ref)
        total += got
    assert abs(total - 1.0) < 1e-12


def test_enumeration_detects_planted_residual_bug(orc):
    """The enumeration is sensitive: dropping max(0, .) from the residual (the
    pages' named pitfall) breaks the identity."""
    rng = np.random.default_rng(4)
    V, gamma, L = 4, 2, 3
    P = np.array([orc.softmax_row(rng.standard_normal(V).astype(np.float32), 1.0)[1] for _ in range(6)])
    Q = np.array([orc.softmax_row(rng.standard_normal(V).astype(np.float32), 1.0)[1] for _ in range(6)])

    class Planted:
        @staticmethod
        def residual(p, q):
            r = np.abs(p - q)  # wrong: |p - q| instead of max(0, p - q)
            return r, r.sum()

    dist = _enumerate_string_dist(P, Q, gamma, L, Planted)
    errs = [abs(dist.get(ys, 0.0) - float(np.prod([P[t, y] for t, y in enumerate(ys)])))
            for ys in itertools.product(range(V), repeat=L)]
    assert max(errs) > 1e-3


# ------------------------------------------------------- batch verify statistics
def _iid_workload(p, q, gamma, B, rng, kv=None):
    """B sequences whose every position has target p (as logits log p) and draft
    probabilities q; draft tokens drawn x ~ q by the harness."""
    V = p.shape[0]
    with np.errstate(divide="ignore"):
        lp = np.log(p).astype(np.float32)
    tgt = np.broadcast_to(lp, (B * (gamma + 1), V))
    dft = np.broadcast_to(q.astype(np.float32), (B * gamma, V))
    cq = np.cumsum(q)
    toks = np.minimum(np.searchsorted(cq, rng.random(B * gamma) * cq[-1], side="right"), V - 1)
    return _tiny_workload(tgt, dft, np.full(B, gamma), toks, probs=True, kv=kv)


def test_page_statistical_check(orc):
    """The page's own check: gamma = 1, p = [.5,.3,.15,.05], uniform q, 400k
    draws: the first emitted token follows p within 0.005 and the acceptance
    rate is 0.700."""
    g = _golden_kv("p1_worked_example.txt")
    p, q = np.array(g["p"]), np.array(g["q"])
    n = int(g["draws"][0])
    w = _iid_workload(p, q, 1, n, np.random.default_rng(2024))
    res = orc.verify_sample(w, seed=99, rnd=0, nthreads=8)
    first = res["tokens"][0::2]
    freq = np.bincount(first, minlength=4) / n
    assert np.all(np.abs(freq - p) < g["tolerance"][0]), freq
    acc = res["accepted"].mean()
    assert abs(acc - g["alpha"][0]) < g["tolerance"][0]


def _expected_tokens(alpha, gamma):
    return (1 - alpha ** (gamma + 1)) / (1 - alpha)


def test_expected_tokens_printed_values():
    """The closed form reproduces every worked value the pages print."""
    with open(os.path.join(GOLDEN, "expected_tokens.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            a, g, printed, dec = float(parts[0]), int(parts[1]), float(parts[2]), int(parts[3])
            assert round(_expected_tokens(a, g), dec) == printed, line


@pytest.mark.parametrize("alpha,gamma", [(0.8, 4), (0.8, 8), (0.7, 4)])
def test_mean_tokens_per_pass_known_alpha(orc, alpha, gamma):
    """Pairs with sum min(p, q) = alpha exactly: p = alpha s + (1-alpha) a and
    q = alpha s + (1-alpha) b with a, b on disjoint supports (alpha = 0.7 uses the
    page's own p and uniform q). Mean emitted tokens over 1e5 rounds is within
    1% of (1 - alpha^(gamma+1)) / (1 - alpha)."""
    rng = np.random.default_rng(int(alpha * 100) + gamma)
    if alpha == 0.7:
        p, q = np.array([0.5, 0.3, 0.15, 0.05]), np.full(4, 0.25)
    else:
        V = 8
        s = rng.dirichlet(np.ones(V))
        a = np.zeros(V)
        a[:3] = rng.dirichlet(np.ones(3))
        b = np.zeros(V)
        b[4:] = rng.dirichlet(np.ones(4))
        p, q = alpha * s + (1 - alpha) * a, alpha * s + (1 - alpha) * b
    assert abs(np.minimum(p, q).sum() - alpha) < 1e-12
    B = 100_000
    w = _iid_workload(p, q, gamma, B, rng)
    res = orc.verify_sample(w, seed=5, rnd=1, nthreads=8)
    emitted = res["accepted"] + 1
    E = _expected_tokens(alpha, gamma)
    assert abs(emitted.mean() - E) / E < 0.01, (emitted.mean(), E)
    assert emitted.min() >= 1 and emitted.max() <= gamma + 1


def test_chi_square_stream_1e6(orc):
    """1e6 rounds through the oracle's real uniform -> token code. The stream
    of emitted tokens of i.i.d. positions follows p (first token and
    consecutive non-overlapping pairs), chi-square p-value > 1e-3."""
    rng = np.random.default_rng(77)
    V, gamma = 6, 3
    p = orc.softmax_row(rng.standard_normal(V).astype(np.float32) * 1.5, 1.0)[1]
    q = orc.softmax_row(rng.standard_normal(V).astype(np.float32) * 1.5, 1.0)[1]
    B = 1_000_000
    w = _iid_workload(p, q, gamma, B, rng)
    res = orc.verify_sample(w, seed=1234, rnd=3, nthreads=8)
    toks = res["tokens"].reshape(B, gamma + 1)
    n_emit = res["accepted"] + 1
    first = toks[:, 0]
    c1 = np.bincount(first, minlength=V)
    assert scipy.stats.chisquare(c1, B * p).pvalue > 1e-3
    stream = toks[np.arange(gamma + 1)[None, :] < n_emit[:, None]]
    n2 = (stream.shape[0] // 2) * 2
    pairs = stream[:n2:2] * V + stream[1:n2:2]
    c2 = np.bincount(pairs, minlength=V * V)
    assert scipy.stats.chisquare(c2, (n2 // 2) * np.outer(p, p).reshape(-1)).pvalue > 1e-3
    # the full stream's marginal too
    assert scipy.stats.chisquare(np.bincount(stream, minlength=V), stream.shape[0] * p).pvalue > 1e-3


def test_chi_square_position_dependent_strings(orc):
    """Position-dependent p^(t), q^(t): run rounds until L tokens are emitted
    per sequence; the joint law of (y_1..y_L) is prod_t p^(t) (chi-square)."""
    rng = np.random.default_rng(31)
    V, gamma, L, B = 3, 2, 3, 200_000
    npos = L + gamma + 1
    P = np.array([orc.softmax_row(rng.standard_normal(V).astype(np.float32) * 1.2, 1.0)[1] for _ in range(npos)])
    Q = np.array([orc.softmax_row(rng.standard_normal(V).astype(np.float32) * 1.2, 1.0)[1] for _ in range(npos)])
    with np.errstate(divide="ignore"):
        LP = np.log(P).astype(np.float32)
    pos = np.zeros(B, dtype=np.int64)
    out = np.full((B, L + gamma + 1), -1, dtype=np.int64)
    rnd = 0
    while (pos < L).any():
        live = np.nonzero(pos < L)[0]
        t = pos[live]
        tgt = LP[(t[:, None] + np.arange(gamma + 1)[None, :]).reshape(-1)]
        didx = (t[:, None] + np.arange(gamma)[None, :]).reshape(-1)
        dft = Q[didx].astype(np.float32)
        cq = np.cumsum(Q[didx], axis=1)
        u = rng.random(didx.shape[0])
        toks = np.minimum((cq < u[:, None] * cq[:, -1:]).sum(axis=1), V - 1)
        w = _tiny_workload(tgt, dft, np.full(live.shape[0], gamma), toks, probs=True)
        res = orc.verify_sample(w, seed=8, rnd=rnd, seq_offset=0, nthreads=8)
        tk = res["tokens"].reshape(-1, gamma + 1)
        ne = res["accepted"] + 1
        for k in range(gamma + 1):
            m = ne > k
            out[live[m], t[m] + k] = tk[m, k]
        pos[live] = t + ne
        rnd += 1
    ys = out[:, :L]
    idx = np.zeros(B, dtype=np.int64)
    for k in range(L):
        idx = idx * V + ys[:, k]
    counts = np.bincount(idx, minlength=V ** L)
    probs = np.ones(1)
    for k in range(L):
        probs = np.outer(probs, P[k]).reshape(-1)
    assert scipy.stats.chisquare(counts, B * probs).pvalue > 1e-3


# ------------------------------------------------------------ special cases
def test_q_equals_p_accepts_everything(orc):
    rng = np.random.default_rng(12)
    B, g, V = 64, 5, 50
    tgt = rng.standard_normal((B * (g + 1), V)).astype(np.float32)
    dft = np.ascontiguousarray(tgt.reshape(B, g + 1, V)[:, :g].reshape(-1, V))
    toks = rng.integers(0, V, size=B * g)
    res = orc.verify_sample(_tiny_workload(tgt, dft, np.full(B, g), toks, T=0.7), seed=3, nthreads=4)
    assert np.all(res["accepted"] == g)


def test_disjoint_one_hot_rejects_to_argmax(orc):
    V, g, B = 6, 3, 10
    tgt = np.full((B * (g + 1), V), -np.inf, np.float32)
    tgt[:, 2] = 0.0
    dft = np.full((B * g, V), -np.inf, np.float32)
    dft[:, 4] = 0.0
    toks = np.full(B * g, 4)
    res = orc.verify_sample(_tiny_workload(tgt, dft, np.full(B, g), toks), seed=1)
    assert np.all(res["accepted"] == 0)
    assert np.all(res["tokens"].reshape(B, g + 1)[:, 0] == 2)
    assert np.all(res["tokens"].reshape(B, g + 1)[:, 1:] == -1)


def test_gamma_zero_is_plain_sampling(orc):
    """gamma = 0 emits one token from p_1 (chi-square over 2e5 sequences)."""
    rng = np.random.default_rng(13)
    V, B = 7, 200_000
    p = orc.softmax_row(rng.standard_normal(V).astype(np.float32), 1.0)[1]
    tgt = np.broadcast_to(np.log(p).astype(np.float32), (B, V))
    dft = np.zeros((0, V), np.float32)
    w = _tiny_workload(tgt, dft, np.zeros(B), np.zeros(0))
    res = orc.verify_sample(w, seed=21, nthreads=8)
    assert np.all(res["accepted"] == 0)
    assert scipy.stats.chisquare(np.bincount(res["tokens"], minlength=V), B * p).pvalue > 1e-3


def test_invariants_and_kv(orc):
    rng = np.random.default_rng(14)
    gam = rng.integers(0, 6, size=300)
    tro, dro = wl.offsets_for(gam)
    V = 40
    tgt = rng.standard_normal((tro[-1], V)).astype(np.float32)
    dft = rng.standard_normal((dro[-1], V)).astype(np.float32)
    toks = rng.integers(0, V, size=dro[-1])
    kv = rng.integers(6, 100, size=300).astype(np.int32)
    w = _tiny_workload(tgt, dft, gam, toks, kv=kv, block_size=16)
    res = orc.verify_sample(w, seed=2, rnd=7, nthreads=4)
    for b in range(300):
        a = res["accepted"][b]
        assert 0 <= a <= gam[b]
        seg = res["tokens"][tro[b]:tro[b + 1]]
        assert np.all(seg[:a + 1] >= 0) and np.all(seg[a + 1:] == -1)
        assert np.array_equal(seg[:a], toks[dro[b]:dro[b] + a])
        assert res["kv"][b] == kv[b] - (gam[b] - a)
        assert res["blocks"][b] == -(-res["kv"][b] // 16)
        assert res["status"][b] == 0


def test_error_statuses(orc):
    V, g = 10, 2
    rng = np.random.default_rng(15)
    tgt = rng.standard_normal((5 * (g + 1), V)).astype(np.float32)
    dft = rng.standard_normal((5 * g, V)).astype(np.float32)
    toks = rng.integers(0, V, size=5 * g)
    toks[2 * g] = V  # seq 2: token out of range
    kv = np.full(5, 50, np.int32)
    kv[3] = 1  # seq 3: kv shorter than gamma
    tgt[4 * (g + 1)] = np.nan  # seq 4: NaN in the first target row
    temps = np.array([1.0, -1.0, 1.0, 1.0, 1.0], np.float32)  # seq 1: bad temperature
    w = _tiny_workload(tgt, dft, np.full(5, g), toks, kv=kv, temps=temps)
    res = orc.verify_sample(w, seed=0)
    assert list(res["status"]) == [0, orc.SEQ_BAD_TEMP, orc.SEQ_BAD_TOKEN, orc.SEQ_BAD_KV, orc.SEQ_BAD_ROW]
    for b in range(1, 5):
        assert res["accepted"][b] == 0 and res["kv"][b] == kv[b]
        assert np.all(res["tokens"][b * (g + 1):(b + 1) * (g + 1)] == -1)


# ------------------------------------------------------------------- greedy
def test_greedy_bruteforce(orc):
    """Accept while x_i == first-index argmax (NaN as -inf), then the target's
    pick; against numpy's argmax."""
    rng = np.random.default_rng(16)
    B, g, V = 400, 4, 37
    tgt = rng.integers(-3, 3, size=(B * (g + 1), V)).astype(np.float32)
    tgt[rng.random(tgt.shape) < 0.05] = np.nan
    vals = np.where(np.isnan(tgt), -np.inf, tgt)
    picks = np.argmax(vals, axis=1).reshape(B, g + 1)
    toks = picks[:, :g].copy()
    lead = rng.integers(0, g + 1, size=B)
    for b in range(B):
        if lead[b] < g:
            toks[b, lead[b]] = (toks[b, lead[b]] + 1 + rng.integers(0, V - 1)) % V
    kv = rng.integers(g, 1000, size=B).astype(np.int32)
    w = _tiny_workload(tgt, np.zeros((B * g, V), np.float32), np.full(B, g), toks.reshape(-1), kv=kv)
    w.greedy = True
    res = orc.verify_greedy(w)
    for b in range(B):
        a = int(np.argmin(np.append(toks[b] == picks[b, :g], False)))
        assert res["accepted"][b] == a
        seg = res["tokens"][b * (g + 1):(b + 1) * (g + 1)]
        assert np.array_equal(seg[:a], toks[b, :a]) and seg[a] == picks[b, a]
        assert np.all(seg[a + 1:] == -1)
        assert res["kv"][b] == kv[b] - (g - a)


def test_greedy_draft_equals_target_accepts_all(orc):
    rng = np.random.default_rng(17)
    B, g, V = 20, 5, 100
    tgt = rng.standard_normal((B * (g + 1), V)).astype(np.float32)
    picks = np.argmax(tgt, axis=1).reshape(B, g + 1)
    w = _tiny_workload(tgt, np.zeros((B * g, V), np.float32), np.full(B, g), picks[:, :g].reshape(-1))
    res = orc.verify_greedy(w)
    assert np.all(res["accepted"] == g)
    assert np.array_equal(res["tokens"].reshape(B, g + 1), picks)


def test_kv_rollback_closed_form(orc):
    kv = np.array([100, 5, 17, 3, 40], np.int32)
    acc = np.array([2, 5, 0, 1, 9], np.int32)
    gam = np.array([4, 5, 3, 4, 8], np.int32)
    out = orc.kv_rollback(kv, acc, gam, 8, block_size=16)
    # 100-(4-2)=98; 5-0=5; 17-3=14; kv 3 < gamma 4 -> error; 40-(8-9) invalid (acc > gamma)
    assert list(out["kv"]) == [98, 5, 14, 3, 40]
    assert list(out["blocks"]) == [7, 1, 1, 1, 3]
    assert list(out["status"]) == [0, 0, 0, orc.SEQ_BAD_KV, orc.SEQ_BAD_LAYOUT]


def test_c2_sigma_matches_golden():
    with open(os.path.join(GOLDEN, "c2_sigma.json")) as f:
        g = json.load(f)
    assert wl.C2_SIGMA == g["sigma"]
    assert abs(g["alpha_at_sigma"] - 0.8) < 1e-3
