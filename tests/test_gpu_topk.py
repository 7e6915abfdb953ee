"""GPU parity of the top-k truncated sampling verify against the float64 oracle.

Covers the filtering path (small k, both dtypes, misaligned rows), the paths
that select over the whole row (k past half a warp buffer, more equal values
at the threshold than a buffer holds, k off for some sequences), probability
drafts, per-sequence k, the distributions the sampler uses (within 1e-5),
k = 1 against the greedy verify, and the benchmarked workload at full size.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_38_gb300 import workloads as wl
from tests.test_gpu_parity import _harness, run_rounds, sv  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [7, 33, 3001, 16411])
def test_topk_ragged_small(sv, dtype, V):
    """Per-sequence k from off through 1 to V, ragged gamma, per-sequence T,
    odd vocabularies (rows off 16-byte boundaries, ragged tails)."""
    rng = np.random.default_rng(500 + V)
    B = 21
    gam = rng.integers(0, 9, size=B)
    gam[0], gam[-1] = 0, 8
    ks = rng.integers(1, max(2, min(V, 400)), size=B).astype(np.int32)
    ks[:6] = [0, 1, 2, V - 1, V, -3]
    w = wl.sampling_workload(f"topk V{V}", config=190, batch=B, vocab=V, gammas=gam, profile="zipf",
                             dtype=dtype, sigma=rng.uniform(0.2, 2.0, B), temps=rng.uniform(0.5, 1.5, B),
                             kv_range=(8, 5000), block_size=16, ragged=True, pool=3, dataset=V, top_k=ks)
    run_rounds(w, range(10), seed=12, seq_offset=3, label=f"top-k ragged V={V} {dtype}")


@pytest.mark.parametrize("k", [1, 20, 50, 1000])
def test_topk_scalar_k_bf16(sv, k):
    """One k for every sequence at a mid-size vocabulary."""
    w = wl.sampling_workload(f"topk k{k}", config=191, batch=12, vocab=32000, gammas=np.full(12, 4),
                             profile="zipf", dtype="bf16", sigma=0.6, temps=0.9, pool=4, top_k=k)
    run_rounds(w, range(8), seed=5, label=f"top-k={k}")


@pytest.mark.parametrize("dtype,k", [("bf16", 1500), ("f32", 700), ("f32", 9000)])
def test_topk_large_k_selects_over_row(sv, dtype, k):
    """k beyond half a warp's buffer: the select runs over the row itself."""
    w = wl.sampling_workload(f"topk big k{k}", config=192, batch=6, vocab=40_009, gammas=[3, 1, 4, 0, 2, 5],
                             profile="gaussian", dtype=dtype, sigma=0.5, temps=1.0, ragged=True, pool=3,
                             top_k=k)
    run_rounds(w, range(6), seed=6, label=f"top-k={k} {dtype}")


def _tied_workload(dtype, k, V=120_000, B=4, g=3, levels=3):
    """Logits on three levels: each warp's share of a row holds more equal
    values at the threshold than its buffer does."""
    rng = np.random.default_rng(77)
    tv = -rng.integers(0, levels, size=(B * (g + 1), V)).astype(np.float32)
    dv = -rng.integers(0, levels, size=(B * g, V)).astype(np.float32)
    store = wl.bf16_bits if dtype == "bf16" else (lambda x: np.ascontiguousarray(x, np.float32))
    toks = [np.argmax(dv + rng.gumbel(size=dv.shape).astype(np.float32), axis=1).astype(np.int32)
            for _ in range(3)]
    return wl.Workload(name="ties", batch=B, vocab=V, gamma_max=g, gammas=np.full(B, g, np.int32),
                       target=store(tv), draft=store(dv), draft_tokens=toks[0], token_pool=toks, temperature=1.0,
                       top_k=k)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("k", [5, 300])
def test_topk_heavy_ties(sv, dtype, k):
    """Ties at the threshold all stay; buffers overflow and the row path runs."""
    w = _tied_workload(dtype, k)
    vals = wl.stored_f32(w.target[0])
    kth = np.sort(vals)[::-1][k - 1]
    assert (vals == kth).sum() > 16 * 2048  # more ties per warp share than one warp's buffer
    run_rounds(w, range(6), seed=8, label=f"ties k={k} {dtype}")


def test_topk_probs_draft(sv):
    """Probability drafts (unnormalised fp32) truncated by their own values."""
    rng = np.random.default_rng(31)
    B, g, V = 8, 4, 6007
    base = wl.sampling_workload("probs", config=194, batch=B, vocab=V, gammas=np.full(B, g), profile="zipf",
                                dtype="f32", sigma=0.7, temps=1.0, pool=2, top_k=40)
    dvals = wl.stored_f32(base.draft)
    probs = np.exp(dvals - dvals.max(axis=1, keepdims=True)).astype(np.float32)
    probs *= rng.uniform(0.5, 3.0, size=(probs.shape[0], 1)).astype(np.float32)
    ks = np.array([40, 1, 0, 7, 40, 200, 3, V], np.int32)
    w = wl.Workload(name="probs top-k", batch=B, vocab=V, gamma_max=g, gammas=base.gammas,
                    target=wl.bf16_bits(wl.stored_f32(base.target)), draft=probs, draft_tokens=base.token_pool[0],
                    token_pool=base.token_pool, draft_is_probs=True, temperature=1.0, top_ks=ks)
    run_rounds(w, range(12), seed=4, label="probs draft top-k")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [5003, 4096, 128256])
def test_topk_debug_probs_within_1e5(sv, V, dtype):
    """The truncated p_i, q_i, sampling weights, p(x), q(x) and Z the GPU path
    uses, within 1e-5 of the oracle's, with the same kept columns."""
    from tests.parity import check_debug_probs

    DeviceBatch = _harness()
    rng = np.random.default_rng(22)
    B = 5
    gam = np.array([3, 0, 5, 1, 2])
    ks = np.array([10, 1, 300, 0, 2], np.int32)
    w = wl.sampling_workload("dbg top-k", config=195, batch=B, vocab=V, gammas=gam, profile="zipf",
                             dtype=dtype, sigma=rng.uniform(0.2, 2.0, B), temps=rng.uniform(0.5, 1.5, B),
                             ragged=True, pool=1, top_k=ks)
    db = DeviceBatch(w, seed=3)
    db.run(rnd=1)
    pos = [(b, i) for b in range(B) for i in range(gam[b] + 1)]
    print(f"top-k V={V} {dtype} worst abs error", check_debug_probs(sv, w, db, pos, same_support=True))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [77_777, 4096])
def test_topk_row_stats(sv, V, dtype):
    """(m, s) of every row: the raw maximum exactly, s over the kept columns
    within 1e-5 relative of numpy's float64 sum."""
    from tests.parity import check_row_stats

    DeviceBatch = _harness()
    ks = np.array([5, 64, 0, 1], np.int32)
    w = wl.sampling_workload("rs top-k", config=196, batch=4, vocab=V, gammas=[2, 3, 1, 4], profile="zipf",
                             dtype=dtype, sigma=0.8, temps=[0.6, 1.0, 1.4, 0.9], ragged=True, pool=1, top_k=ks)
    db = DeviceBatch(w)
    db.run()
    print(f"top-k V={V} {dtype} worst relative error of s", check_row_stats(sv, w, db, top_ks=ks))


def test_topk_one_matches_greedy(sv):
    """k = 1 with distinct maxima reduces the sampling verify to the greedy
    one: same accepted counts and tokens as the GPU's greedy verify."""
    DeviceBatch = _harness()
    w = wl.sampling_workload("k1", config=197, batch=40, vocab=50_000, gammas=np.full(40, 6), profile="zipf",
                             dtype="f32", sigma=0.05, temps=1.0, pool=1, top_k=1)
    ds = DeviceBatch(w, seed=1)
    ds.run(rnd=0)
    rs = ds.results()
    wg = wl.Workload(name="k1 greedy", batch=w.batch, vocab=w.vocab, gamma_max=w.gamma_max, gammas=w.gammas,
                     target=w.target, draft=None, draft_tokens=w.draft_tokens, token_pool=[w.draft_tokens],
                     greedy=True)
    dg = DeviceBatch(wg)
    dg.run()
    rg = dg.results()
    assert np.array_equal(rs["accepted"], rg["accepted"])
    assert np.array_equal(rs["tokens"], rg["tokens"])
    assert (rs["accepted"] > 0).any() and (rs["accepted"] < 6).any()


def test_topk_config3_full_size(sv):
    """The benchmarked workload (B=64, gamma=8, V=128256 bf16) with top-k 50."""
    w = wl.config3(top_k=50)
    run_rounds(w, range(12), seed=0, label="C3 top-k 50")
