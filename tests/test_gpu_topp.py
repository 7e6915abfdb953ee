"""GPU parity of top-p (nucleus) against the float64 oracle, after top-k
and alone: per-sequence p with off values, both dtypes and odd
vocabularies, the row path (large k, ties), probability drafts, top-p
without top-k (the whole row's nucleus: short, flat and full-size rows), the truncated
distributions within 1e-5 with the same kept columns, and the benchmarked
workload at k = 50, p = 0.9."""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_38_gb300 import workloads as wl
from tests.test_gpu_parity import _harness, run_rounds, sv  # noqa: F401  (fixture)
from tests.test_gpu_topk import _tied_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [33, 3001, 16411])
def test_topp_ragged_small(sv, dtype, V):
    rng = np.random.default_rng(700 + V)
    B = 21
    gam = rng.integers(0, 9, size=B)
    gam[0], gam[-1] = 0, 8
    ks = rng.integers(1, max(2, min(V, 300)), size=B).astype(np.int32)
    ps = rng.uniform(0.05, 0.99, size=B).astype(np.float32)
    ps[:5] = [0.0, 1.0, np.nan, 1e-6, 0.999]
    w = wl.sampling_workload(f"topp V{V}", config=390, batch=B, vocab=V, gammas=gam, profile="zipf",
                             dtype=dtype, sigma=rng.uniform(0.2, 2.0, B), temps=rng.uniform(0.5, 1.5, B),
                             kv_range=(8, 5000), block_size=16, ragged=True, pool=3, dataset=V, top_k=ks, top_p=ps)
    run_rounds(w, range(8), seed=13, seq_offset=2, label=f"top-p ragged V={V} {dtype}")


@pytest.mark.parametrize("k,p", [(50, 0.9), (1000, 0.5), (200, 0.99)])
def test_topp_scalar(sv, k, p):
    w = wl.sampling_workload(f"topp k{k} p{p}", config=391, batch=12, vocab=32000, gammas=np.full(12, 4),
                             profile="zipf", dtype="bf16", sigma=0.6, temps=0.9, pool=4, top_k=k, top_p=p)
    run_rounds(w, range(8), seed=5, label=f"top-k={k} top-p={p}")


@pytest.mark.parametrize("dtype,k", [("bf16", 1500), ("f32", 700)])
def test_topp_row_path(sv, dtype, k):
    w = wl.sampling_workload(f"topp big k{k}", config=392, batch=6, vocab=40_009, gammas=[3, 1, 4, 0, 2, 5],
                             profile="gaussian", dtype=dtype, sigma=0.5, temps=1.0, ragged=True, pool=3,
                             top_k=k, top_p=0.8)
    run_rounds(w, range(6), seed=6, label=f"top-p row path k={k} {dtype}")


def test_topp_heavy_ties(sv):
    w = _tied_workload("bf16", 300)
    w.top_p = 0.6
    run_rounds(w, range(4), seed=8, label="top-p ties")


def test_topp_probs_draft(sv):
    rng = np.random.default_rng(33)
    B, g, V = 8, 4, 6007
    base = wl.sampling_workload("probs", config=394, batch=B, vocab=V, gammas=np.full(B, g), profile="zipf",
                                dtype="f32", sigma=0.7, temps=1.0, pool=2, top_k=40)
    dvals = wl.stored_f32(base.draft)
    probs = np.exp(dvals - dvals.max(axis=1, keepdims=True)).astype(np.float32)
    probs *= rng.uniform(0.5, 3.0, size=(probs.shape[0], 1)).astype(np.float32)
    w = wl.Workload(name="probs top-p", batch=B, vocab=V, gamma_max=g, gammas=base.gammas,
                    target=wl.bf16_bits(wl.stored_f32(base.target)), draft=probs, draft_tokens=base.token_pool[0],
                    token_pool=base.token_pool, draft_is_probs=True, temperature=1.0,
                    top_ks=np.array([40, 1, 7, 40, 200, 3, 100, 60], np.int32),
                    top_ps=np.array([0.9, 0.5, 0.0, 0.3, 0.95, 0.99, 0.7, 1e-4], np.float32))
    run_rounds(w, range(10), seed=4, label="probs draft top-p")


def test_topp_without_top_k(sv):
    """Top-p with top-k off (k <= 0 or k >= V): the nucleus of the whole
    row. Per-sequence p with off values, and top-k rows, mixed in."""
    B = 8
    w = wl.sampling_workload("topp alone", config=395, batch=B, vocab=3001, gammas=np.full(B, 3), profile="zipf",
                             dtype="bf16", sigma=0.5, temps=1.0, pool=2,
                             top_k=np.array([0, 5, 3001, 5, 0, 5, -1, 10], np.int32),
                             top_p=np.array([0.9, 0.9, 0.5, 1.0, 0.0, np.nan, 0.2, 0.5], np.float32))
    run_rounds(w, range(4), seed=3, label="top-p alone")
    DeviceBatch = _harness()
    db = DeviceBatch(w, seed=3)
    db.run()
    assert db.results()["status"].tolist() == [0] * B


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [33, 1031, 32000])
def test_topp_alone_sizes(sv, dtype, V):
    rng = np.random.default_rng(900 + V)
    B = 12
    ps = rng.uniform(0.05, 0.99, size=B).astype(np.float32)
    ps[:3] = [0.999, 0.5, 1e-6]
    w = wl.sampling_workload(f"topp alone V{V}", config=397, batch=B, vocab=V, gammas=rng.integers(0, 6, size=B),
                             profile="zipf", dtype=dtype, sigma=rng.uniform(0.2, 1.5, B),
                             temps=rng.uniform(0.5, 1.5, B), ragged=True, pool=2, dataset=V, top_p=ps)
    run_rounds(w, range(4), seed=9, label=f"top-p alone V={V} {dtype}")


def test_topp_alone_flat_rows(sv):
    """High temperature on Gaussian logits: the nucleus at p = 0.95 holds
    tens of thousands of columns, with many equal bf16 values at its edge."""
    w = wl.sampling_workload("topp alone flat", config=398, batch=6, vocab=40_009, gammas=np.full(6, 2),
                             profile="gaussian", dtype="bf16", sigma=0.4, temps=1.5, pool=2, top_p=0.95,
                             gauss_std=1.0)
    run_rounds(w, range(3), seed=2, label="top-p alone, flat rows")


def test_topp_alone_probs_draft(sv):
    rng = np.random.default_rng(34)
    B, g, V = 6, 3, 5003
    base = wl.sampling_workload("probs alone", config=399, batch=B, vocab=V, gammas=np.full(B, g), profile="zipf",
                                dtype="f32", sigma=0.7, temps=1.0, pool=2)
    dvals = wl.stored_f32(base.draft)
    probs = np.exp(dvals - dvals.max(axis=1, keepdims=True)).astype(np.float32)
    probs *= rng.uniform(0.5, 3.0, size=(probs.shape[0], 1)).astype(np.float32)
    w = wl.Workload(name="probs top-p alone", batch=B, vocab=V, gamma_max=g, gammas=base.gammas,
                    target=wl.bf16_bits(wl.stored_f32(base.target)), draft=probs, draft_tokens=base.token_pool[0],
                    token_pool=base.token_pool, draft_is_probs=True, temperature=1.0,
                    top_ps=np.array([0.9, 0.5, 0.0, 0.3, 0.95, 0.99], np.float32))
    run_rounds(w, range(6), seed=4, label="probs draft top-p alone")


def test_topp_alone_target_at_a_group_edge(sv):
    """Rows of two groups, n columns at logit 0 and the rest at -1 (T = 1),
    with p the float nearest to the top group's share: the target sits
    within a float rounding of the top group's mass, where a float sum can
    take the other side from the double-float one (which decides)."""
    B, g, V = 16, 2, 2003
    base = wl.sampling_workload("group edge", config=400, batch=B, vocab=V, gammas=np.full(B, g), profile="zipf",
                                dtype="f32", sigma=0.5, temps=1.0, pool=2)
    ns = 3 + 7 * np.arange(B)
    tgt = np.full((B, g + 1, V), -1.0, np.float32)
    dft = np.full((B, g, V), -1.0, np.float32)
    ps = np.empty(B, np.float32)
    for b, n in enumerate(ns):
        cols = np.random.default_rng(b).permutation(V)[:n]
        tgt[b][:, cols] = 0.0
        dft[b][:, cols] = 0.0
        ps[b] = np.float32(n / (n + (V - n) * np.exp(-1.0)))
    w = wl.Workload(name="top-p at a group edge", batch=B, vocab=V, gamma_max=g, gammas=base.gammas,
                    target=wl.bf16_bits(tgt.reshape(B * (g + 1), V)), draft=dft.reshape(B * g, V),
                    draft_tokens=base.token_pool[0], token_pool=base.token_pool, draft_is_probs=False,
                    temperature=1.0, top_ps=ps)
    run_rounds(w, range(4), seed=5, label="top-p alone at a group edge")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [5003, 4096, 128256])
def test_topp_debug_probs_within_1e5(sv, V, dtype):
    """The nucleus-truncated p_i, q_i, sampling weights, p(x), q(x) and Z
    within 1e-5 of the oracle's, with the same nucleus, for top-p inside a
    top-k set and over the whole row."""
    from tests.parity import check_debug_probs

    DeviceBatch = _harness()
    rng = np.random.default_rng(23)
    B = 5
    gam = np.array([3, 0, 5, 1, 2])
    w = wl.sampling_workload("dbg top-p", config=396, batch=B, vocab=V, gammas=gam, profile="zipf", dtype=dtype,
                             sigma=rng.uniform(0.2, 2.0, B), temps=rng.uniform(0.5, 1.5, B), ragged=True, pool=1,
                             top_k=np.array([50, 1, 0, 20, V], np.int32),
                             top_p=np.array([0.9, 0.5, 0.3, 0.0, 0.99], np.float32))
    db = DeviceBatch(w, seed=3)
    db.run(rnd=1)
    pos = [(b, i) for b in range(B) for i in range(gam[b] + 1)]
    print(f"top-p V={V} {dtype} worst abs error", check_debug_probs(sv, w, db, pos, same_support=True))


def test_topp_config3_full_size(sv):
    w = wl.config3(top_k=50, top_p=0.9)
    run_rounds(w, range(8), seed=0, label="C3 top-k 50 top-p 0.9")


def test_topp_alone_config3_full_size(sv):
    """Top-p 0.9 without top-k on the benchmarked workload (B=64, gamma=8,
    V=128256 bf16): every row's whole-row nucleus, in the bench's launch."""
    w = wl.config3(top_k=0, top_p=0.9)
    run_rounds(w, range(3), seed=0, label="C3 top-p 0.9 alone")


def test_topp_alone_bf16_pattern_counts(sv):
    """Whole-row nucleus of bf16 logits rows from pattern counts: a row where
    one value fills 70,000 of 131,072 columns (its 16-bit counter wraps, so
    the row takes the narrowing search), rows of +0 and -0 (joined to one
    pattern; 40,000 of each, and 70,000 of -0), a row with NaN (invalid), a
    row with -inf columns, and plain rows, all at top-p 0.9 with top-k off."""
    rng = np.random.default_rng(41)
    B, g, V = 8, 1, 131072
    base = wl.sampling_workload("counts", config=401, batch=B, vocab=V, gammas=np.full(B, g), profile="zipf",
                                dtype="bf16", sigma=0.6, temps=1.0, pool=2)
    tgt = wl.stored_f32(base.target).reshape(B, g + 1, V).copy()
    dft = wl.stored_f32(base.draft).reshape(B, g, V).copy()

    def fill(b, cols, val):
        tgt[b][:, cols] = val
        dft[b][:, cols] = val

    fill(0, rng.permutation(V)[:70_000], np.float32(-1.5))
    perm = rng.permutation(V)
    fill(1, perm[:40_000], np.float32(0.0))
    fill(1, perm[40_000:80_000], np.float32(-0.0))
    fill(2, rng.permutation(V)[:70_000], np.float32(-0.0))
    tgt[3][0, 777] = np.nan  # position 0's target row: always read
    fill(4, rng.permutation(V)[:5_000], np.float32(-np.inf))
    w = wl.Workload(name="bf16 pattern counts", batch=B, vocab=V, gamma_max=g, gammas=base.gammas,
                    target=wl.bf16_bits(tgt.reshape(B * (g + 1), V)), draft=wl.bf16_bits(dft.reshape(B * g, V)),
                    draft_tokens=base.token_pool[0], token_pool=base.token_pool, draft_is_probs=False,
                    temperature=1.0, top_p=0.9)
    run_rounds(w, range(3), seed=7, label="top-p alone, bf16 pattern counts")
    DeviceBatch = _harness()
    db = DeviceBatch(w, seed=7)
    db.run()
    st = db.results()["status"].tolist()
    assert st[3] != 0 and [s for i, s in enumerate(st) if i != 3] == [0] * (B - 1)


def test_topp_alone_config3_high_p(sv):
    """Top-p 0.99 without top-k on the benchmarked workload: most rows' edges
    lie among columns too light to be counted on the first pass, so they are
    counted again with every column (the exact path), at full size."""
    w = wl.config3(top_k=0, top_p=0.99)
    run_rounds(w, range(2), seed=1, label="C3 top-p 0.99 alone")


@pytest.mark.parametrize("V", [1, 5, 7, 600_011])
def test_topp_alone_bf16_edge_sizes(sv, V):
    """The whole-row nucleus kernel at its edges: rows shorter than one
    16-byte vector (head and tail columns only), and rows of 600,011 columns
    (19 ring stages, unaligned starts)."""
    rng = np.random.default_rng(950 + V)
    B = 6 if V < 1000 else 2
    ps = rng.uniform(0.3, 0.99, size=B).astype(np.float32)
    w = wl.sampling_workload(f"topp alone edge V{V}", config=403, batch=B, vocab=V,
                             gammas=rng.integers(0, 4, size=B), profile="zipf", dtype="bf16",
                             sigma=rng.uniform(0.2, 1.5, B), temps=rng.uniform(0.6, 1.4, B), ragged=True,
                             pool=2, dataset=V, top_p=ps)
    run_rounds(w, range(3), seed=11, label=f"top-p alone bf16 V={V}")
