"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs and uniforms (see tests/parity.py for the rule)."""
import os

import numpy as np
import pytest
import scipy.stats

import oracle
from speculative_decoding_verification_38_gb300 import workloads as wl
from tests.parity import Tally, compare_exact, compare_sample, offsets

pytestmark = pytest.mark.gpu
NTHREADS = os.cpu_count() or 4


@pytest.fixture(scope="module")
def sv():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_38_gb300 as sv

    sv.build()
    oracle.build()
    return sv


def _harness():
    from speculative_decoding_verification_38_gb300.harness import DeviceBatch

    return DeviceBatch


def run_rounds(w, rounds, *, seed=0, seq_offset=0, uniforms_fn=None, label=""):
    DeviceBatch = _harness()
    tally = Tally()
    db = DeviceBatch(w, seed=seed, seq_offset=seq_offset,
                     uniforms=None if uniforms_fn is None else uniforms_fn(0))
    for r in rounds:
        toks = w.tokens_for_round(r)
        unif = None
        if uniforms_fn is not None:
            unif = uniforms_fn(r)
            db.uniforms.copy_(__import__("torch").from_numpy(unif))
        db.run(rnd=r, pool_index=r)
        g = db.results()
        o = oracle.verify_sample(w, seed=seed, rnd=r, seq_offset=seq_offset, uniforms=unif, draft_tokens=toks,
                                 nthreads=NTHREADS, diagnostics=True)
        tally.merge(compare_sample(w, g, o, seed=seed, rnd=r, tokens=toks, seq_offset=seq_offset,
                                   uniforms=unif))
    print(label, tally)
    tally.check(label)
    return tally


# ------------------------------------------------------------------------ RNG
def test_philox_bit_exact(sv):
    import torch

    for seed, rnd, off in [(0, 0, 0), (0xDEADBEEFCAFEF00D, (7 << 32) | 3, 1000), (2**64 - 1, 2**64 - 1, 2**31)]:
        B, npos = 37, 9
        out = torch.zeros(B * npos * 2, dtype=torch.float32, device="cuda")
        sv.check(sv.spec_debug_philox(seed, rnd, off, B, npos, out), "philox")
        got = out.cpu().numpy().reshape(B, npos, 2)
        for b in range(B):
            for i in range(npos):
                ua, us = oracle.uniform_pair(seed, rnd, off + b, i)
                assert got[b, i, 0] == ua and got[b, i, 1] == us


# --------------------------------------------------------------- small configs
def test_config1_all_rounds(sv):
    """B=1, gamma=4, V=1000 fp32 Gaussian logits, all 10,000 rounds."""
    w = wl.config1()
    run_rounds(w, range(10_000), seed=0, label="C1")


def test_config2_all_rounds(sv):
    """B=1, gamma=4, V=50257 fp32 Zipf (rows not 16-byte aligned), 2,000 rounds."""
    w = wl.config2()
    run_rounds(w, range(2_000), seed=0, label="C2")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [1, 7, 33, 3001, 16411])
def test_ragged_small(sv, dtype, V):
    """Ragged gamma in 0..8, odd vocabularies (misaligned rows, ragged tails),
    per-sequence temperatures, KV lengths with paging."""
    rng = np.random.default_rng(V)
    B = 23
    gam = rng.integers(0, 9, size=B)
    gam[0], gam[-1] = 0, 8
    w = wl.sampling_workload(f"ragged V{V}", config=90, batch=B, vocab=V, gammas=gam, profile="zipf",
                             dtype=dtype, sigma=rng.uniform(0.2, 2.0, B), temps=rng.uniform(0.5, 1.5, B),
                             kv_range=(8, 5000), block_size=16, ragged=True, pool=3, dataset=V)
    run_rounds(w, range(12), seed=11, seq_offset=5, label=f"ragged V={V} {dtype}")


def test_probs_draft_and_mixed_dtypes(sv):
    """Draft given as (unnormalised) probabilities in fp32 with a bf16 target."""
    rng = np.random.default_rng(3)
    B, g, V = 9, 5, 4099
    base = wl.sampling_workload("probs", config=91, batch=B, vocab=V, gammas=np.full(B, g), profile="zipf",
                                dtype="f32", sigma=0.7, temps=1.0, pool=2)
    tvals = wl.stored_f32(base.target)
    dvals = wl.stored_f32(base.draft)
    probs = np.exp(dvals - dvals.max(axis=1, keepdims=True)).astype(np.float32)
    probs *= rng.uniform(0.5, 3.0, size=(probs.shape[0], 1)).astype(np.float32)  # unnormalised rows
    w = wl.Workload(name="probs", batch=B, vocab=V, gamma_max=g, gammas=base.gammas,
                    target=wl.bf16_bits(tvals), draft=probs, draft_tokens=base.token_pool[0],
                    token_pool=base.token_pool, draft_is_probs=True, temperature=1.0)
    run_rounds(w, range(20), seed=4, label="probs draft")


def test_caller_uniforms(sv):
    """Uniforms from a caller buffer instead of Philox."""
    w = wl.sampling_workload("unif", config=92, batch=17, vocab=2048, gammas=np.full(17, 3), profile="zipf",
                             dtype="bf16", sigma=0.5, temps=0.9, pool=4)

    def unif(r):
        rng = np.random.default_rng(1000 + r)
        u = (rng.integers(0, 1 << 24, size=(w.rows_target, 2)) / float(1 << 24)).astype(np.float32)
        return u

    run_rounds(w, range(10), uniforms_fn=unif, label="caller uniforms")


def test_large_vocab_multi_slot(sv):
    """V larger than one streaming slice and than one sampler CTA's chunk."""
    w = wl.sampling_workload("bigV", config=93, batch=3, vocab=600_011, gammas=[2, 0, 4], profile="zipf",
                             dtype="bf16", sigma=[0.3, 1.0, 2.0], temps=1.1, ragged=True, pool=2)
    run_rounds(w, range(6), seed=9, label="V=600011")


# ----------------------------------------------------------- full-size configs
def test_config3_full_size(sv):
    """B=64, gamma=8, V=128256 bf16, the benchmarked workload and launch."""
    w = wl.config3()
    run_rounds(w, range(200), seed=0, label="C3")


def test_config5_full_size(sv):
    """B=512 ragged gamma 1..8, V=128256 bf16, per-sequence T, paged KV."""
    w = wl.config5()
    run_rounds(w, range(50), seed=0, label="C5")


def test_config4_greedy_full_size(sv):
    """Greedy, B=256, gamma=5, V=152064 bf16 with injected ties: bit-exact."""
    DeviceBatch = _harness()
    w = wl.config4()
    db = DeviceBatch(w)
    db.run()
    g = db.results()
    o = oracle.verify_greedy(w, nthreads=NTHREADS)
    compare_exact(w, g, o)
    acc = g["accepted"]
    print("C4 mean tokens/pass", (acc + 1).mean(), "ties injected", len(w.info["tie_rows"]))


@pytest.mark.parametrize("dataset", range(8))
def test_config4_greedy_datasets(sv, dataset):
    """Eight independent greedy datasets (reduced batch), bit-exact."""
    DeviceBatch = _harness()
    w = wl.config4(batch=24, dataset=dataset + 1, tie_every=3)
    db = DeviceBatch(w)
    db.run()
    compare_exact(w, db.results(), oracle.verify_greedy(w, nthreads=NTHREADS))


def test_greedy_small_odd_shapes(sv):
    rng = np.random.default_rng(8)
    for V, dtype in [(1, "f32"), (5, "bf16"), (1001, "f32"), (70001, "bf16")]:
        B, g = 13, 4
        vals = rng.integers(-4, 4, size=(B * (g + 1), V)).astype(np.float32)
        vals[rng.random(vals.shape) < 0.03] = np.nan
        vals[::7] = -np.inf
        tgt = wl.bf16_bits(vals) if dtype == "bf16" else vals
        picks = np.array([oracle.argmax_row(r) for r in tgt]).reshape(B, g + 1)
        toks = picks[:, :g].copy()
        toks[rng.random((B, g)) < 0.3] = 0
        w = wl.Workload(name="g", batch=B, vocab=V, gamma_max=g, gammas=np.full(B, g, np.int32), target=tgt,
                        draft=None, draft_tokens=toks.reshape(-1).astype(np.int32),
                        kv_in=rng.integers(g, 99, B).astype(np.int32), block_size=8, greedy=True)
        DeviceBatch = _harness()
        db = DeviceBatch(w)
        db.run()
        compare_exact(w, db.results(), oracle.verify_greedy(w))


# -------------------------------------------------------------- probabilities
# Vocabularies whose rows are 16-byte aligned in both dtypes (4096, 128256)
# take the bulk-copy streaming kernel and its separate finalize kernel, the
# launches the benchmark times; 5003 and 77,777 take the plain-load kernel.
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [5003, 4096, 128256])
def test_debug_probs_within_1e5(sv, V, dtype):
    """p_i, q_i, the normalised residual / bonus weights, p(x), q(x) and Z of
    the GPU path within 1e-5 absolute of the oracle's float64 values."""
    from tests.parity import bulk_copy_path, check_debug_probs

    DeviceBatch = _harness()
    rng = np.random.default_rng(21)
    B = 6
    gam = np.array([3, 0, 5, 1, 8, 2])
    w = wl.sampling_workload("dbg", config=94, batch=B, vocab=V, gammas=gam, profile="zipf", dtype=dtype,
                             sigma=rng.uniform(0.2, 2.0, B), temps=rng.uniform(0.5, 1.5, B), ragged=True, pool=1)
    db = DeviceBatch(w, seed=3)
    assert bulk_copy_path(w, db) == (V != 5003)
    db.run(rnd=2)
    pos = [(b, i) for b in range(B) for i in range(gam[b] + 1)]
    print(f"V={V} {dtype} worst abs error", check_debug_probs(sv, w, db, pos))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [77_777, 4096, 128256])
def test_row_stats_match_oracle(sv, V, dtype):
    from tests.parity import bulk_copy_path, check_row_stats

    DeviceBatch = _harness()
    w = wl.sampling_workload("rs", config=95, batch=4, vocab=V, gammas=[2, 3, 1, 4], profile="zipf",
                             dtype=dtype, sigma=0.8, temps=[0.6, 1.0, 1.4, 0.9], ragged=True, pool=1)
    db = DeviceBatch(w)
    assert bulk_copy_path(w, db) == (V != 77_777)
    db.run()
    print(f"V={V} {dtype} worst relative error of s", check_row_stats(sv, w, db))


def test_config3_reduced_batch_stats_and_probs(sv):
    """The benchmarked shape (gamma=8, V=128256 bf16, T=0.8) at B=8: (m, s)
    of all 136 rows, and p, q, r/Z, p(x), q(x), Z at every accept position of
    two sequences and at the position each sequence stopped."""
    from tests.parity import bulk_copy_path, check_debug_probs, check_row_stats

    DeviceBatch = _harness()
    w = wl.config3(batch=8, pool=1)
    db = DeviceBatch(w, seed=0)
    assert bulk_copy_path(w, db)
    db.run(rnd=0)
    acc = db.results()["accepted"]
    print("C3/8 worst relative error of s", check_row_stats(sv, w, db))
    pos = [(b, i) for b in (0, 5) for i in range(9)] + [(b, int(acc[b])) for b in range(8)]
    print("C3/8 worst abs error", check_debug_probs(sv, w, db, pos))


# ------------------------------------------------------------ errors and reuse
def test_error_statuses_match_oracle(sv):
    rng = np.random.default_rng(5)
    B, g, V = 8, 3, 301
    w = wl.sampling_workload("err", config=96, batch=B, vocab=V, gammas=np.full(B, g), profile="zipf",
                             dtype="f32", sigma=0.5, temps=np.ones(B, np.float32), kv_range=(10, 20),
                             block_size=4, ragged=True, pool=1)
    w.temperatures[1] = -1.0                      # bad temperature
    w.draft_tokens[2 * g + 1] = V                 # token out of range
    w.kv_in[3] = 2                                # kv shorter than gamma
    w.target[4 * (g + 1)] = np.nan                # NaN in a needed target row
    w.draft[5 * g][:] = -np.inf                   # all -inf draft row
    w.target[6 * (g + 1) + g][7] = np.inf         # +inf in the bonus row (error only if reached)
    w.token_pool = [w.draft_tokens]
    DeviceBatch = _harness()
    db = DeviceBatch(w, seed=1)
    db.run(rnd=0)
    gpu = db.results()
    o = oracle.verify_sample(w, seed=1, rnd=0, nthreads=2, diagnostics=True)
    assert list(gpu["status"][:6]) == list(o["status"][:6])
    assert list(o["status"][:6]) == [0, 5, 1, 2, 3, 3]
    compare_sample(w, gpu, o, seed=1, rnd=0, tokens=w.draft_tokens).check("errors")


def test_bad_layout_is_reported(sv):
    """Offsets that stay monotone but break gamma_b + 1 == target rows."""
    gam = np.array([2, 3, 1])
    w = wl.sampling_workload("lay", config=97, batch=3, vocab=64, gammas=gam, profile="zipf", dtype="f32",
                             sigma=0.5, temps=1.0, ragged=True, pool=1)
    tro, dro = offsets(w)
    tro = tro.copy()
    tro[1] += 1  # seq 0 gets 4 target rows for gamma 2; seq 1 one fewer
    w.target_row_off = tro
    DeviceBatch = _harness()
    db = DeviceBatch(w)
    db.run()
    gpu = db.results()
    o = oracle.verify_sample(w, seed=0, diagnostics=True)
    assert list(gpu["status"]) == list(o["status"]) == [4, 4, 0]
    assert gpu["tokens"][tro[2]:tro[3]].tolist() == o["tokens"][tro[2]:tro[3]].tolist()


def test_repeat_calls_identical_and_workspace_reuse(sv):
    """The arrival counters reset themselves: identical calls give identical
    bytes; the same workspace then serves a different shape."""
    DeviceBatch = _harness()
    w = wl.sampling_workload("rep", config=98, batch=11, vocab=9000, gammas=np.full(11, 4), profile="zipf",
                             dtype="bf16", sigma=0.6, temps=1.0, pool=1)
    db = DeviceBatch(w, seed=2)
    outs = []
    for _ in range(3):
        db.run(rnd=5)
        outs.append(db.results())
    for o in outs[1:]:
        for k in outs[0]:
            assert np.array_equal(outs[0][k], o[k])
    # different batch on the same workspace buffer
    w2 = wl.sampling_workload("rep2", config=99, batch=5, vocab=9000, gammas=np.full(5, 2), profile="zipf",
                              dtype="bf16", sigma=0.6, temps=1.0, pool=1)
    db2 = DeviceBatch(w2, seed=2)
    db2.args.set_workspace(db.ws)
    db2.run(rnd=1)
    o2 = oracle.verify_sample(w2, seed=2, rnd=1, diagnostics=True)
    compare_sample(w2, db2.results(), o2, seed=2, rnd=1, tokens=w2.draft_tokens).check("reuse")
    db.run(rnd=5)
    r = db.results()
    for k in outs[0]:
        assert np.array_equal(outs[0][k], r[k])


def test_kv_rollback_matches_oracle(sv):
    import torch

    rng = np.random.default_rng(6)
    B = 1000
    gam = rng.integers(0, 9, size=B).astype(np.int32)
    acc = rng.integers(-1, 10, size=B).astype(np.int32)
    kv = rng.integers(0, 40000, size=B).astype(np.int32)
    t = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    kv_out = torch.zeros(B, dtype=torch.int32, device="cuda")
    blocks = torch.zeros_like(kv_out)
    st = torch.zeros_like(kv_out)
    sv.check(sv.spec_kv_rollback(t(kv), kv_out, t(acc), t(gam), 8, 16, blocks, st), "kv_rollback")
    o = oracle.kv_rollback(kv, acc, gam, 8, block_size=16)
    assert np.array_equal(kv_out.cpu().numpy(), o["kv"])
    assert np.array_equal(blocks.cpu().numpy(), o["blocks"])
    assert np.array_equal(st.cpu().numpy(), o["status"])


# --------------------------------------------------------------- statistics
def _iid_gpu_workload(p, q, gamma, B, rng, pool=8):
    V = p.shape[0]
    with np.errstate(divide="ignore"):
        lp = np.log(p).astype(np.float32)
    tgt = np.ascontiguousarray(np.broadcast_to(lp, (B * (gamma + 1), V)))
    dft = np.ascontiguousarray(np.broadcast_to(q.astype(np.float32), (B * gamma, V)))
    cq = np.cumsum(q)
    pool = [np.minimum(np.searchsorted(cq, rng.random(B * gamma) * cq[-1], side="right"), V - 1).astype(np.int32)
            for _ in range(pool)]
    return wl.Workload(name="iid", batch=B, vocab=V, gamma_max=gamma, gammas=np.full(B, gamma, np.int32),
                       target=tgt, draft=dft, draft_tokens=pool[0], token_pool=pool, draft_is_probs=True)


def test_gpu_chi_square_1e6(sv):
    """1e6 GPU rounds: the emitted stream follows p (chi-square p > 1e-3)."""
    DeviceBatch = _harness()
    rng = np.random.default_rng(77)
    V, gamma, B = 6, 3, 65536
    p = oracle.softmax_row(rng.standard_normal(V).astype(np.float32) * 1.5, 1.0)[1]
    q = oracle.softmax_row(rng.standard_normal(V).astype(np.float32) * 1.5, 1.0)[1]
    w = _iid_gpu_workload(p, q, gamma, B, rng, pool=16)
    db = DeviceBatch(w, seed=1234)
    firsts, streams = [], []
    for r in range(16):
        db.run(rnd=r, pool_index=r)
        g = db.results()
        toks = g["tokens"].reshape(B, gamma + 1)
        ne = g["accepted"] + 1
        firsts.append(toks[:, 0])
        streams.append(toks[np.arange(gamma + 1)[None, :] < ne[:, None]])
    first = np.concatenate(firsts)
    stream = np.concatenate(streams)
    assert scipy.stats.chisquare(np.bincount(first, minlength=V), first.shape[0] * p).pvalue > 1e-3
    assert scipy.stats.chisquare(np.bincount(stream, minlength=V), stream.shape[0] * p).pvalue > 1e-3


@pytest.mark.parametrize("alpha,gamma", [(0.8, 4), (0.8, 8)])
def test_gpu_mean_tokens_known_alpha(sv, alpha, gamma):
    DeviceBatch = _harness()
    rng = np.random.default_rng(int(alpha * 100) + gamma)
    V = 8
    s = rng.dirichlet(np.ones(V))
    a = np.zeros(V)
    a[:3] = rng.dirichlet(np.ones(3))
    bb = np.zeros(V)
    bb[4:] = rng.dirichlet(np.ones(4))
    p, q = alpha * s + (1 - alpha) * a, alpha * s + (1 - alpha) * bb
    w = _iid_gpu_workload(p, q, gamma, 50_000, rng, pool=2)
    db = DeviceBatch(w, seed=5)
    em = []
    for r in range(2):  # 1e5 rounds: two calls of 50,000 sequences
        db.run(rnd=r, pool_index=r)
        em.append(db.results()["accepted"] + 1)
    emitted = np.concatenate(em)
    E = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(emitted.mean() - E) / E < 0.01
    assert emitted.min() >= 1 and emitted.max() <= gamma + 1


def test_light_exp2_is_unbiased(sv):
    """The sampler's light 2^x (exponents in [-45, -13]) as its sums see it
    (SFU value plus the sum-level correction) against exact 2^x: mean relative
    error below 3e-9; each SFU value within 3e-7."""
    import torch

    rng = np.random.default_rng(12)
    x = rng.uniform(-45.0, -13.0, 1 << 22).astype(np.float32)
    xt = torch.from_numpy(x).cuda()
    yt = torch.empty(2 * x.shape[0], dtype=torch.float32, device="cuda")
    sv.check(sv.spec_debug_light_exp2(xt, yt), "light_exp2")
    y = yt.cpu().numpy().astype(np.float64).reshape(-1, 2)
    ex = np.exp2(x.astype(np.float64))
    assert np.abs((y[:, 0] - ex) / ex).max() < 3e-7
    rel = (y[:, 0] + y[:, 1] - ex) / ex
    assert abs(rel.mean()) < 3e-9, rel.mean()
