"""GPU parity of tree verification against the float64 oracle: chain-shaped
trees (which the oracle pins to the chain verify), fixed and ragged random
trees in both dtypes with per-sequence temperatures, probability drafts,
wide nodes (64 candidates, more nodes than threads), p == q rows (every
residual empty), the candidates-i.i.d.-from-q distribution check, greedy
walks bit-exact, every status, and the benchmarked workload at full size
(see tests/parity.py, compare_tree, for the rule)."""
import numpy as np
import pytest
import scipy.stats

import oracle
from speculative_decoding_verification_38_gb300 import workloads as wl
from tests.parity import Tally, compare_tree
from tests.test_gpu_parity import sv  # noqa: F401  (fixture)
from tests.test_oracle_tree import _chain_as_tree, _fan, _star_workload

pytestmark = pytest.mark.gpu

# The tree of the benchmark: B = 64 trees of branching (4, 2, 2), 29 nodes each.
BENCH_TREE = dict(batch=64, vocab=128256, branching=[4, 2, 2], dtype="bf16", sigma=0.6, temps=0.8)


def _dev(w, **kw):
    from speculative_decoding_verification_38_gb300.harness import DeviceTree

    return DeviceTree(w, **kw)


def run_tree_rounds(w, rounds, *, seed=0, seq_offset=0, label=""):
    dt = _dev(w, seed=seed, seq_offset=seq_offset)
    tally = Tally()
    for r in rounds:
        dt.run(rnd=r)
        g = dt.results()
        o = oracle.tree_verify(w, seed=seed, rnd=r, seq_offset=seq_offset, diagnostics=True)
        tally.merge(compare_tree(w, g, o))
    print(label, tally)
    tally.check(label)
    return tally


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chain_trees_match_the_chain_verify(sv, dtype):
    """One chain per sequence: the GPU tree walk against the oracle, and its
    tokens against the GPU chain verify of the same chain (they may differ
    only where the oracle's draw lies within the band)."""
    from speculative_decoding_verification_38_gb300.harness import DeviceBatch

    w = wl.sampling_workload("chain", config=80, batch=48, vocab=5003, gammas=np.full(48, 6), profile="zipf",
                             dtype=dtype, sigma=0.8, temps=0.9, pool=1)
    t = _chain_as_tree(w)
    run_tree_rounds(t, range(4), seed=7, seq_offset=3, label=f"chain tree {dtype}")
    dt = _dev(t, seed=7, seq_offset=3)
    db = DeviceBatch(w, seed=7, seq_offset=3)
    differ = 0
    for r in range(4):
        dt.run(rnd=r)
        db.run(rnd=r)
        a, c = dt.results(), db.results()
        differ += int(np.sum(a["accepted"] != c["accepted"]))
        o = oracle.tree_verify(t, seed=7, rnd=r, seq_offset=3, diagnostics=True)
        for b in range(48):
            seg = slice(b * 7, b * 7 + 7)
            if not np.array_equal(a["tokens"][seg], c["tokens"][seg]):
                d = o["diag"]
                assert min(d["acc_margin"][b], abs(d["u_smp"][b] - d["cdf_lo"][b]),
                           abs(d["u_smp"][b] - d["cdf_hi"][b])) < 1e-5, (r, b)
    assert differ <= 1


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V,branching", [(33, [3, 2, 2]), (3001, [4, 4]), (32000, [2, 2, 2, 2]),
                                         (16411, [1, 1, 1, 1, 1, 1])])
def test_random_trees(sv, dtype, V, branching):
    rng = np.random.default_rng(V)
    B = 24
    w = wl.tree_workload(f"tree V{V}", config=V % 97, batch=B, vocab=V, branching=branching, dtype=dtype,
                         sigma=float(rng.uniform(0.3, 1.2)), temps=rng.uniform(0.5, 1.5, B).astype(np.float32))
    t = run_tree_rounds(w, range(6), seed=11, seq_offset=5, label=f"tree V={V} {branching} {dtype}")
    assert t.draws > B * 6


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_trees(sv, dtype):
    w = wl.ragged_tree_workload("ragged", config=3, batch=40, vocab=7001, max_nodes=45, dtype=dtype, sigma=0.5,
                                temps=0.8)
    run_tree_rounds(w, range(6), seed=21, label=f"ragged trees {dtype}")


def test_wide_nodes(sv):
    """Branching (64, 8): 577 nodes per tree, more than the CTA's threads,
    and 64 candidates at the root (the most the walk keeps)."""
    w = wl.tree_workload("wide", config=9, batch=4, vocab=61, branching=[64, 8], dtype="f32", sigma=2.0, temps=1.3)
    run_tree_rounds(w, range(8), seed=4, label="wide")


def test_probability_drafts(sv):
    rng = np.random.default_rng(5)
    w = wl.tree_workload("probs", config=10, batch=16, vocab=4099, branching=[3, 3], dtype="f32", sigma=0.7)
    d = wl.stored_f32(w.draft).astype(np.float64)
    p = np.exp(d - d.max(axis=1, keepdims=True))
    p *= rng.uniform(0.5, 2.0, size=(p.shape[0], 1))  # unnormalised: the walk divides by the sum
    w.draft = np.ascontiguousarray(p, np.float32)
    w.draft_is_probs = True
    run_tree_rounds(w, range(6), seed=8, label="probs drafts")


def test_equal_rows_leave_every_residual_empty(sv):
    """Target row == draft row at every node, candidates on tokens of zero
    probability: every test fails, every residual is empty (Z = 0) and the
    token is drawn from p itself."""
    rng = np.random.default_rng(6)
    V, B, m = 257, 12, 3
    n = m + 1
    rows = (2.0 * rng.standard_normal((B * n, V))).astype(np.float32)
    dead = rng.choice(V, size=20, replace=False)
    rows[:, dead] = -np.inf
    parent = np.tile(np.array([-1] + [0] * m, np.int32), B)
    toks = np.full(B * n, -1, np.int32)
    toks.reshape(B, n)[:, 1:] = rng.choice(dead, size=(B, m))
    w = wl.TreeWorkload(name="p == q", batch=B, vocab=V, node_off=np.arange(B + 1, dtype=np.int64) * n,
                        parent=parent, tokens=toks, target=rows, draft=rows.copy())
    run_tree_rounds(w, range(4), seed=2, label="p == q")
    g = _dev(w, seed=2)
    g.run(rnd=0)
    assert np.all(g.results()["accepted"] == 0)


def test_candidates_iid_from_q_give_the_target(sv):
    """The GPU walk over m = 3 candidates drawn i.i.d. from q keeps the
    target: the first token follows p0 (chi-square, 4 rounds of 60k trees)."""
    rng = np.random.default_rng(43)
    V, B, m = 5, 60_000, 3
    p0 = rng.dirichlet(np.ones(V))
    q0 = rng.dirichlet(np.ones(V))
    P1 = rng.dirichlet(np.ones(V), size=V)
    t = _star_workload(rng, p0, q0, P1, m, B)
    g = _dev(t, seed=11)
    counts = np.zeros(V, np.int64)
    for rnd in range(4):
        g.run(rnd=rnd)
        r = g.results()
        counts += np.bincount(r["tokens"].reshape(B, m + 1)[:, 0], minlength=V)
        o = oracle.tree_verify(t, seed=11, rnd=rnd, diagnostics=True)
        compare_tree(t, r, o).check("star")
    assert scipy.stats.chisquare(counts, counts.sum() * p0).pvalue > 1e-3


@pytest.mark.parametrize("dtype,V", [("bf16", 32000), ("f32", 1000)])
def test_greedy_bit_exact(sv, dtype, V):
    w = wl.tree_workload("greedy", config=12, batch=64, vocab=V, branching=[3, 2, 2, 1], dtype=dtype,
                         greedy_agree=0.6)
    w.greedy = True
    if dtype == "f32":
        tg = w.target.copy()
        tg[5, :10] = np.nan  # NaN reads as -inf
        tg[9] = -np.inf      # no finite logit: index 0
        w.target = tg
    g = _dev(w)
    g.run()
    r = g.results()
    o = oracle.tree_verify(w)
    for k in ("tokens", "accepted", "path", "status"):
        assert np.array_equal(r[k], o[k]), k
    assert r["accepted"].max() >= 2
    rg = wl.ragged_tree_workload("greedy ragged", config=4, batch=30, vocab=999, max_nodes=70, dtype="bf16",
                                 greedy_agree=0.7)
    rg.greedy = True
    g = _dev(rg)
    g.run()
    r, o = g.results(), oracle.tree_verify(rg)
    for k in ("tokens", "accepted", "path", "status"):
        assert np.array_equal(r[k], o[k]), k


def test_statuses(sv):
    w = wl.tree_workload("status tree", config=6, batch=10, vocab=30, branching=[2, 2], dtype="f32")
    n = int(w.node_off[1])
    par = w.parent.copy()
    tok = w.tokens.copy()
    tgt = w.target.copy()
    dft = w.draft.copy()
    par[1 * n + 3] = 3          # 1: a node is its own parent
    tok[2 * n + 2] = 30         # 2: a token outside the vocabulary
    tgt[3 * n + 0, 4] = np.nan  # 3: a NaN in the root's target row
    par[4 * n + 0] = 0          # 4: the root has a parent
    tgt[6 * n + 0, 7] = np.inf  # 6: +inf in the root's target row
    dft[7 * n + 0, 2] = np.nan  # 7: a NaN in the root's draft row
    tgt[8 * n + 0] = -np.inf    # 8: no finite logit at the root
    w.parent, w.tokens, w.target, w.draft = par, tok, tgt, dft
    temps = np.ones(10, np.float32)
    temps[5] = 0.0              # 5: temperature 0
    temps[9] = np.inf           # 9: infinite temperature
    w.temperatures = temps
    g = _dev(w, seed=3)
    g.run()
    r = g.results()
    o = oracle.tree_verify(w, seed=3, diagnostics=True)
    S = oracle
    assert o["status"].tolist() == [0, S.SEQ_BAD_LAYOUT, S.SEQ_BAD_TOKEN, S.SEQ_BAD_ROW, S.SEQ_BAD_LAYOUT,
                                    S.SEQ_BAD_TEMP, S.SEQ_BAD_ROW, S.SEQ_BAD_ROW, S.SEQ_BAD_ROW, S.SEQ_BAD_TEMP]
    compare_tree(w, r, o).check("statuses")
    # layout errors write none of the sequence's slots
    assert np.all(r["tokens"][n:2 * n] == -7) and np.all(r["tokens"][4 * n:5 * n] == -7)


def test_candidate_limit_and_offsets(sv):
    rng = np.random.default_rng(12)
    for m, want in [(64, 0), (65, oracle.SEQ_UNSUPPORTED)]:
        t = _fan(3, m, 50, rng)
        g = _dev(t, seed=2)
        g.run()
        r = g.results()
        o = oracle.tree_verify(t, seed=2, diagnostics=True)
        assert o["status"].tolist() == [want] * 3
        compare_tree(t, r, o).check(f"fan {m}")
        t.greedy = True  # greedy keeps no residual: no limit
        g = _dev(t)
        g.run()
        assert g.results()["status"].tolist() == [0] * 3
    w = wl.tree_workload("short rows", config=7, batch=3, vocab=20, branching=[2], dtype="f32")
    off = w.node_off.copy()
    off[3] += 1  # the last sequence claims a node past the rows
    w.node_off = off
    g = _dev(w, seed=1)
    g.run()
    r = g.results()
    assert r["status"].tolist() == [0, 0, oracle.SEQ_BAD_LAYOUT]
    o = oracle.tree_verify(w, seed=1, diagnostics=True)
    assert np.array_equal(r["status"], o["status"])


def test_bench_workload_full_size(sv):
    """The benchmarked trees (64 x 29 nodes, V = 128256, bf16) in the launch
    configuration the benchmark times, against the oracle on every sequence."""
    w = wl.tree_workload("bench tree", config=20, **BENCH_TREE)
    t = run_tree_rounds(w, range(2), seed=0, label="bench tree")
    assert t.draws >= 128
