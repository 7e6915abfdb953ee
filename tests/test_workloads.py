"""The synthetic inputs follow the stated recipe (no GPU): shapes, dtypes
and parameters of each configuration at reduced sizes, the Zipf profile's
mean, the draft noise, and draft tokens drawn from the draft distribution."""
import numpy as np
import scipy.special
import scipy.stats

from speculative_decoding_verification_38_gb300 import workloads as wl


def test_config1_gaussian_rows_and_noise():
    w = wl.config1(pool=2)
    assert w.target.shape == (5, 1000) and w.target.dtype == np.float32
    assert w.draft.shape == (4, 1000) and w.temperature == 1.0 and w.temperatures is None
    assert abs(w.target.std() - 2.0) < 0.1
    noise = w.draft - w.target[:4]
    assert abs(noise.std() - 0.5) < 0.03 and abs(noise.mean()) < 0.03


def test_config3_recipe_at_reduced_size():
    B, V = 8, 4000
    w = wl.config3(batch=B, vocab=V, pool=1)
    assert w.target.dtype == np.uint16 and w.target.shape == (B * 9, V) and w.draft.shape == (B * 8, V)
    assert w.temperature == np.float32(0.8) and w.block_size == 16
    assert np.all((w.kv_in >= 512) & (w.kv_in <= 4096))
    sig = w.info["sigma"]
    assert sig.shape == (B,) and np.all((sig >= 0.2) & (sig <= 1.5))
    # Zipf rows: -1.1 ln(rank) + N(0, 1), so each row's mean is -1.1 ln(V!)/V
    vals = wl.stored_f32(w.target).astype(np.float64)
    want = -1.1 * scipy.special.gammaln(V + 1) / V
    assert np.all(np.abs(vals.mean(axis=1) - want) < 0.1)
    # and its variance is 1.1^2 Var(ln rank) + 1 (the unit noise)
    want_var = 1.21 * np.var(np.log(np.arange(1, V + 1))) + 1.0
    assert np.all(np.abs(vals.var(axis=1) / want_var - 1) < 0.05)


def test_config5_ragged_recipe():
    w = wl.config5(batch=24, vocab=1000, pool=1)
    g = np.asarray(w.gammas)
    assert np.all((g >= 1) & (g <= 8)) and w.gamma_max == g.max()
    assert w.target_row_off is not None and w.target_row_off[-1] == (g + 1).sum()
    assert w.draft_row_off[-1] == g.sum() == w.draft.shape[0]
    assert np.all((w.temperatures >= 0.5) & (w.temperatures <= 1.5))
    assert np.all((w.kv_in >= 128) & (w.kv_in <= 32768))


def test_config4_greedy_recipe():
    w = wl.config4(batch=64, vocab=3000)
    assert w.greedy and w.draft is None and w.target.dtype == np.uint16
    vals = wl.stored_f32(w.target).reshape(64, 6, 3000)
    am = vals[:, :5].argmax(axis=2)
    same = (np.asarray(w.draft_tokens).reshape(64, 5) == am).mean()
    assert 0.65 < same < 0.85  # the draft token is the target's argmax w.p. 0.75


def test_draft_tokens_follow_q():
    rng = np.random.default_rng(3)
    logits = np.tile(rng.standard_normal(6).astype(np.float32), (20000, 1))
    T = 0.7
    x = wl.gumbel_argmax(np.random.default_rng(9), logits, np.full(20000, T, np.float32))
    q = scipy.special.softmax(logits[0].astype(np.float64) / T)
    assert scipy.stats.chisquare(np.bincount(x, minlength=6), 20000 * q).pvalue > 1e-3
    # a drafter with its own top-k draws only among its k largest
    xk = wl.gumbel_argmax(np.random.default_rng(9), logits, np.full(20000, T, np.float32),
                          k_per_row=np.full(20000, 2, np.int32))
    assert set(np.unique(xk)) <= set(np.argsort(logits[0])[::-1][:2].tolist())


def test_tree_workload_structure():
    w = wl.tree_workload("recipe tree", config=12, batch=5, vocab=500, branching=[3, 2], dtype="bf16")
    n = int(w.node_off[1])
    assert n == 1 + 3 + 6 and np.array_equal(w.node_off, np.arange(6) * n)
    for b in range(5):
        par = w.parent[b * n:(b + 1) * n]
        assert par[0] == -1 and np.all((par[1:] >= 0) & (par[1:] < np.arange(1, n)))
        assert np.bincount(par[1:], minlength=n)[0] == 3  # the root's three candidates
        tok = w.tokens[b * n:(b + 1) * n]
        assert tok[0] == -1 and np.all((tok[1:] >= 0) & (tok[1:] < 500))
    r = wl.ragged_tree_workload("recipe ragged", config=13, batch=6, vocab=300, max_nodes=12)
    sizes = np.diff(w.node_off)
    sizes_r = np.diff(r.node_off)
    assert sizes.min() == n and sizes_r[0] == 1 and sizes_r[-1] == 12 and sizes_r.max() <= 12


def test_tree_candidates_drawn_from_q_at_the_parent():
    """Trees of one root with 4 candidates over a 6-token vocabulary: the sum
    over draws of q(x), under each tree's own root q = softmax(draft / T),
    matches its expectation sum_t 4 sum_j q_j^2 (z-score), and the same
    statistic rejects draws from the target's p, so the test has power."""
    M = 4000
    w = wl.tree_workload("recipe root draws", config=14, batch=M, vocab=6, branching=[4], dtype="f32",
                         temps=0.8)
    roots = np.arange(M) * 5
    q = scipy.special.softmax(wl.stored_f32(w.draft)[roots].astype(np.float64) / 0.8, axis=1)
    p = scipy.special.softmax(wl.stored_f32(w.target)[roots].astype(np.float64) / 0.8, axis=1)
    toks = w.tokens.reshape(M, 5)[:, 1:]
    stat = np.take_along_axis(q, toks, axis=1).sum()
    s2, s3 = (q ** 2).sum(axis=1), (q ** 3).sum(axis=1)
    mean, var = 4 * s2.sum(), 4 * (s3 - s2 ** 2).sum()
    assert abs(stat - mean) / np.sqrt(var) < 4
    mean_p = 4 * (p * q).sum()  # the statistic's mean if the candidates came from p
    assert abs(mean_p - mean) / np.sqrt(var) > 6


def test_ngram_contexts_copy_the_document():
    ctx, off = wl.ngram_contexts(batch=3, doc_len=400, gen_len=100, vocab=5000)
    assert off[0] == 0 and np.all(np.diff(off) >= 500) and ctx.dtype == np.int32
    for b in range(3):
        c = ctx[off[b]:off[b + 1]]
        doc, gen = c[:400], c[400:]
        assert np.all((c >= 0) & (c < 5000))
        # with 5 % edits, most generated 4-grams occur in the document
        grams = {tuple(doc[i:i + 4]) for i in range(len(doc) - 3)}
        hit = np.mean([tuple(gen[i:i + 4]) in grams for i in range(len(gen) - 3)])
        assert hit > 0.6
