"""Pins of the oracle's tree verification (no GPU).

A chain-shaped tree must give exactly what the (separately pinned) chain
verify gives, for sampling and for greedy. With candidates drawn i.i.d. from
the draft, the emitted tokens must follow the target (chi-square on the
first token and on the first two). Greedy trees are checked against a brute
force walk, and every status.
"""
import numpy as np
import pytest
import scipy.stats

from speculative_decoding_verification_38_gb300 import workloads as wl


def _chain_as_tree(w):
    """The chain workload w (uniform gamma) as one chain-shaped tree per sequence."""
    B, g, V = w.batch, w.gamma_max, w.vocab
    n = g + 1
    parent = np.tile(np.arange(-1, g, dtype=np.int32), B)
    toks = np.full(B * n, -1, np.int32)
    toks.reshape(B, n)[:, 1:] = np.asarray(w.draft_tokens, np.int32).reshape(B, g)
    if w.draft is None:  # greedy: draft rows are not read
        dft = np.zeros((B * n, V), np.float32)
    else:
        dft = np.zeros((B * n,) + w.draft.shape[1:], w.draft.dtype)
        dft.reshape(B, n, V)[:, :g] = w.draft.reshape(B, g, V)  # the leaf's draft row is not used
    return wl.TreeWorkload(name="chain tree", batch=B, vocab=V, node_off=np.arange(B + 1, dtype=np.int64) * n,
                           parent=parent, tokens=toks, target=w.target, draft=dft, draft_is_probs=w.draft_is_probs,
                           temperatures=w.temperatures, temperature=w.temperature, greedy=w.greedy)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chain_tree_equals_chain_verify(orc, dtype):
    w = wl.sampling_workload("chain", config=80, batch=64, vocab=300, gammas=np.full(64, 5), profile="zipf",
                             dtype=dtype, sigma=1.0, temps=0.9, pool=1)
    t = _chain_as_tree(w)
    for rnd in range(3):
        c = orc.verify_sample(w, seed=7, rnd=rnd, seq_offset=3)
        r = orc.tree_verify(t, seed=7, rnd=rnd, seq_offset=3)
        assert np.array_equal(r["accepted"], c["accepted"])
        assert np.array_equal(r["tokens"], c["tokens"])
        acc = c["accepted"]
        path = r["path"].reshape(64, 6)
        for b in range(64):
            assert path[b, :acc[b]].tolist() == list(range(1, acc[b] + 1))
    assert 0 < c["accepted"].mean() < 5


def test_chain_tree_equals_greedy(orc):
    w = wl.config4(batch=40, vocab=2000)
    t = _chain_as_tree(w)
    c = orc.verify_greedy(w)
    r = orc.tree_verify(t, greedy=True)
    assert np.array_equal(r["accepted"], c["accepted"]) and np.array_equal(r["tokens"], c["tokens"])


def _star_workload(rng, p0, q0, P1, m, B):
    """B trees: a root with m leaf candidates drawn i.i.d. from q0; the target
    row of a leaf with token y is log P1[y]."""
    V = p0.shape[0]
    n = m + 1
    parent = np.tile(np.array([-1] + [0] * m, np.int32), B)
    cq = np.cumsum(q0)
    toks = np.full(B * n, -1, np.int32)
    cand = np.minimum(np.searchsorted(cq, rng.random((B, m)) * cq[-1], side="right"), V - 1)
    toks.reshape(B, n)[:, 1:] = cand
    tgt = np.empty((B * n, V), np.float32)
    with np.errstate(divide="ignore"):
        tgt.reshape(B, n, V)[:, 0] = np.log(p0)
        tgt.reshape(B, n, V)[:, 1:] = np.log(P1)[cand]
    dft = np.broadcast_to(q0.astype(np.float32), (B * n, V))
    return wl.TreeWorkload(name="star", batch=B, vocab=V, node_off=np.arange(B + 1, dtype=np.int64) * n,
                           parent=parent, tokens=toks, target=tgt, draft=np.ascontiguousarray(dft), draft_is_probs=True)


@pytest.mark.parametrize("m", [1, 2, 3])
def test_candidates_iid_from_q_give_target(orc, m):
    """Recursive rejection over m i.i.d. candidates keeps the target: the first
    token follows p0, and (first, second) follows p0(y1) P1[y1](y2)."""
    rng = np.random.default_rng(40 + m)
    V, B = 5, 200_000
    p0 = rng.dirichlet(np.ones(V))
    q0 = rng.dirichlet(np.ones(V))
    P1 = rng.dirichlet(np.ones(V), size=V)
    t = _star_workload(rng, p0, q0, P1, m, B)
    r = orc.tree_verify(t, seed=11, rnd=2)
    toks = r["tokens"].reshape(B, m + 1)
    y1 = toks[:, 0]
    assert scipy.stats.chisquare(np.bincount(y1, minlength=V), B * p0).pvalue > 1e-3
    two = r["accepted"] == 1
    joint = np.bincount(toks[two, 0] * V + toks[two, 1], minlength=V * V)
    # given an accepted first token, the second is the bonus from P1[y1]
    for y in range(V):
        sel = joint[y * V:(y + 1) * V]
        if sel.sum() > 500:
            assert scipy.stats.chisquare(sel, sel.sum() * P1[y]).pvalue > 1e-4
    # more candidates accept more often
    if m > 1:
        assert (r["accepted"] == 1).mean() > 0.0


def _greedy_walk(t, b):
    o = t.node_off[b]
    n = t.node_off[b + 1] - o
    vals = wl.stored_f32(t.target[o:o + n]).astype(np.float64)
    vals = np.where(np.isnan(vals), -np.inf, vals)
    u, toks, path = 0, [], []
    while True:
        g = int(np.argmax(vals[u]))
        kids = [v for v in range(u + 1, n) if t.parent[o + v] == u and t.tokens[o + v] == g]
        toks.append(g)
        if not kids:
            return toks, path
        path.append(kids[0])
        u = kids[0]


def test_greedy_bruteforce(orc):
    w = wl.tree_workload("greedy tree", config=5, batch=50, vocab=40, branching=[3, 2, 2], dtype="bf16",
                         greedy_agree=0.5)
    w.greedy = True
    r = orc.tree_verify(w)
    n = w.node_off[1]
    for b in range(50):
        toks, path = _greedy_walk(w, b)
        o = b * n
        assert r["accepted"][b] == len(path)
        assert r["tokens"][o:o + len(toks)].tolist() == toks and np.all(r["tokens"][o + len(toks):o + n] == -1)
        assert r["path"][o:o + len(path)].tolist() == path
    assert r["accepted"].max() >= 2


def test_statuses(orc):
    w = wl.tree_workload("status tree", config=6, batch=6, vocab=30, branching=[2, 2], dtype="f32")
    n = int(w.node_off[1])
    par = w.parent.copy()
    tok = w.tokens.copy()
    tgt = w.target.copy()
    par[1 * n + 3] = 3          # sequence 1: a node is its own parent
    tok[2 * n + 2] = 30         # sequence 2: a token outside the vocabulary
    tgt[3 * n + 0, 4] = np.nan  # sequence 3: a NaN in the root's row
    par[4 * n + 0] = 0          # sequence 4: the root has a parent
    w.target = tgt
    temps = np.ones(6, np.float32)
    temps[5] = 0.0              # sequence 5: temperature 0
    w.temperatures = temps
    r = orc.tree_verify(w, parent=par, tokens=tok, seed=3)
    assert r["status"].tolist() == [0, orc.SEQ_BAD_LAYOUT, orc.SEQ_BAD_TOKEN, orc.SEQ_BAD_ROW, orc.SEQ_BAD_LAYOUT,
                                    orc.SEQ_BAD_TEMP]
    assert np.all(r["tokens"][2 * n:3 * n] == -1) and r["accepted"][2] == 0


def test_offsets_past_the_rows_are_a_layout_error(orc):
    w = wl.tree_workload("short rows", config=7, batch=3, vocab=20, branching=[2], dtype="f32")
    off = w.node_off.copy()
    off[3] = off[3] + 1  # the last sequence claims a node past the 9 rows given
    w.node_off = off
    r = orc.tree_verify(w, seed=1)
    assert r["status"].tolist() == [0, 0, orc.SEQ_BAD_LAYOUT]
    assert np.all(r["tokens"][6:9] == -7)  # a layout error writes none of the sequence's slots


def _fan(B, m, V, rng):
    """B trees, each a root with m leaf children (tokens drawn at random)."""
    n = m + 1
    parent = np.tile(np.array([-1] + [0] * m, np.int32), B)
    toks = np.full(B * n, -1, np.int32)
    toks.reshape(B, n)[:, 1:] = rng.integers(0, V, size=(B, m))
    tgt = rng.standard_normal((B * n, V)).astype(np.float32)
    dft = rng.standard_normal((B * n, V)).astype(np.float32)
    return wl.TreeWorkload(name="fan", batch=B, vocab=V, node_off=np.arange(B + 1, dtype=np.int64) * n,
                           parent=parent, tokens=toks, target=tgt, draft=dft)


def test_candidate_limit(orc):
    rng = np.random.default_rng(12)
    ok = orc.tree_verify(_fan(3, 64, 50, rng), seed=2)
    assert ok["status"].tolist() == [0, 0, 0]
    over = orc.tree_verify(_fan(3, 65, 50, rng), seed=2)
    assert over["status"].tolist() == [orc.SEQ_UNSUPPORTED] * 3
    assert np.all(over["tokens"] == -1) and np.all(over["accepted"] == 0)
    # greedy keeps no residual: no limit
    assert orc.tree_verify(_fan(3, 65, 50, rng), greedy=True)["status"].tolist() == [0, 0, 0]


def test_candidate_limit_applies_to_visited_nodes_only(orc):
    """Node 1 has 70 children but the walk never reaches it: the root's
    target is sure of node 2's token and its draft of node 1's, so node 1
    fails (q > 0 = p there) and node 2 passes."""
    V = 30
    parent = np.array([-1, 0, 0] + [1] * 70, np.int32)
    toks = np.concatenate([[-1, 4, 9], np.arange(70) % V]).astype(np.int32)
    tgt = np.zeros((73, V), np.float32)
    tgt[0] = -60.0
    tgt[0, 9] = 60.0
    dft = np.zeros((73, V), np.float32)
    dft[0] = -60.0
    dft[0, 4] = 60.0
    t = wl.TreeWorkload(name="deep fan", batch=1, vocab=V, node_off=np.array([0, 73], np.int64), parent=parent,
                        tokens=toks, target=tgt, draft=dft)
    r = orc.tree_verify(t, seed=5)
    assert r["status"].tolist() == [0] and r["path"][0] == 2 and r["accepted"][0] == 1
    assert r["tokens"][0] == 9
    t.parent = parent.copy()
    t.parent[3:] = 2  # now the visited node 2 has the 70 children
    assert orc.tree_verify(t, seed=5)["status"].tolist() == [orc.SEQ_UNSUPPORTED]
