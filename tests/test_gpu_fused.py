"""GPU parity of the fused verify kernel (one cooperative launch: the
streaming pass in waves of sequences, each sequence's decision, tile pass and
draw while later rows stream) against the float64 oracle, under the same
rule as the separate kernels (tests/parity.py). The library's default path
is the separate kernels; these tests select the fused kernel with the
spec_debug_set_path hook, on shapes it takes: sampling without truncation,
rows on 16-byte boundaries."""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_38_gb300 import workloads as wl
from tests.parity import bulk_copy_path, check_debug_probs, check_row_stats, compare_sample
from tests.test_gpu_parity import _harness, run_rounds

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_38_gb300 as sv

    sv.build()
    oracle.build()
    sv.check(sv.spec_debug_set_path(sv.PATH_FUSED), "set_path")
    yield sv
    sv.spec_debug_set_path(sv.PATH_DEFAULT)


def test_path_hook_rejects_bad_values(sv):
    assert sv.spec_debug_set_path(3) == sv.SPEC_ERR_INVALID_ARG
    assert sv.spec_debug_set_path(-1) == sv.SPEC_ERR_INVALID_ARG
    sv.check(sv.spec_debug_set_path(sv.PATH_FUSED), "set_path")


def test_fused_config3(sv):
    """The benchmarked workload (B=64, gamma=8, V=128256 bf16), 50 rounds."""
    w = wl.config3()
    run_rounds(w, range(50), seed=0, label="fused C3")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [1024, 4096, 32000])
def test_fused_ragged(sv, dtype, V):
    """Ragged gamma 0..8 (a sequence of gamma 0 draws its bonus at once), per
    sequence temperatures and KV lengths, several waves and ragged tiles."""
    rng = np.random.default_rng(V + 7)
    B = 29
    gam = rng.integers(0, 9, size=B)
    gam[0], gam[-1] = 0, 8
    w = wl.sampling_workload(f"fused ragged V{V}", config=90, batch=B, vocab=V, gammas=gam, profile="zipf",
                             dtype=dtype, sigma=rng.uniform(0.2, 2.0, B), temps=rng.uniform(0.5, 1.5, B),
                             kv_range=(8, 5000), block_size=16, ragged=True, pool=3, dataset=V)
    run_rounds(w, range(8), seed=11, seq_offset=5, label=f"fused ragged V={V} {dtype}")


def test_fused_probs_draft_mixed_dtypes(sv):
    """Unnormalised fp32 probability drafts beside a bf16 target."""
    rng = np.random.default_rng(3)
    B, g, V = 9, 5, 4096
    base = wl.sampling_workload("probs", config=91, batch=B, vocab=V, gammas=np.full(B, g), profile="zipf",
                                dtype="f32", sigma=0.7, temps=1.0, pool=2)
    dvals = wl.stored_f32(base.draft)
    probs = np.exp(dvals - dvals.max(axis=1, keepdims=True)).astype(np.float32)
    probs *= rng.uniform(0.5, 3.0, size=(probs.shape[0], 1)).astype(np.float32)
    w = wl.Workload(name="probs", batch=B, vocab=V, gamma_max=g, gammas=base.gammas,
                    target=wl.bf16_bits(wl.stored_f32(base.target)), draft=probs, draft_tokens=base.token_pool[0],
                    token_pool=base.token_pool, draft_is_probs=True, temperature=1.0)
    run_rounds(w, range(12), seed=4, label="fused probs draft")


def test_fused_caller_uniforms(sv):
    w = wl.sampling_workload("unif", config=92, batch=17, vocab=2048, gammas=np.full(17, 3), profile="zipf",
                             dtype="bf16", sigma=0.5, temps=0.9, pool=4)

    def unif(r):
        rng = np.random.default_rng(1000 + r)
        return (rng.integers(0, 1 << 24, size=(w.rows_target, 2)) / float(1 << 24)).astype(np.float32)

    run_rounds(w, range(8), uniforms_fn=unif, label="fused caller uniforms")


def test_fused_ragged_c5_shape(sv):
    """The ragged C5 generator at B=64 (gamma_b in 1..8, T_b in [0.5, 1.5])."""
    w = wl.config5(batch=64)
    run_rounds(w, range(5), seed=0, label="fused C5 B=64")


def test_fused_probabilities_and_row_stats(sv):
    """p, q, r/Z, p(x), q(x), Z within 1e-5 and every row's (m, s), as the
    fused kernel leaves them."""
    DeviceBatch = _harness()
    rng = np.random.default_rng(21)
    B = 6
    gam = np.array([3, 0, 5, 1, 8, 2])
    w = wl.sampling_workload("dbg", config=94, batch=B, vocab=4096, gammas=gam, profile="zipf", dtype="bf16",
                             sigma=rng.uniform(0.2, 2.0, B), temps=rng.uniform(0.5, 1.5, B), ragged=True, pool=1)
    db = DeviceBatch(w, seed=3)
    assert bulk_copy_path(w, db)
    db.run(rnd=2)
    check_row_stats(sv, w, db)
    check_debug_probs(sv, w, db, [(b, i) for b in range(B) for i in range(gam[b] + 1)])


def test_fused_errors_layout_and_reuse(sv):
    """Error statuses, a broken layout, repeated calls (every header word back
    at zero) and the same workspace serving another shape."""
    DeviceBatch = _harness()
    B, g, V = 8, 3, 304
    w = wl.sampling_workload("err", config=96, batch=B, vocab=V, gammas=np.full(B, g), profile="zipf",
                             dtype="f32", sigma=0.5, temps=np.ones(B, np.float32), kv_range=(10, 20),
                             block_size=4, ragged=True, pool=1)
    w.temperatures[1] = -1.0
    w.draft_tokens[2 * g + 1] = V
    w.kv_in[3] = 2
    w.target[4 * (g + 1)] = np.nan
    w.draft[5 * g][:] = -np.inf
    w.token_pool = [w.draft_tokens]
    db = DeviceBatch(w, seed=1)
    outs = []
    for _ in range(3):
        db.run(rnd=0)
        outs.append(db.results())
    o = oracle.verify_sample(w, seed=1, rnd=0, nthreads=2, diagnostics=True)
    assert list(outs[0]["status"][:6]) == list(o["status"][:6]) == [0, 5, 1, 2, 3, 3]
    compare_sample(w, outs[0], o, seed=1, rnd=0, tokens=w.draft_tokens).check("fused errors")
    for r in outs[1:]:
        for k in outs[0]:
            assert np.array_equal(outs[0][k], r[k])
    gam = np.array([2, 3, 1])
    w2 = wl.sampling_workload("lay", config=97, batch=3, vocab=64, gammas=gam, profile="zipf", dtype="f32",
                              sigma=0.5, temps=1.0, ragged=True, pool=1)
    tro = np.asarray(w2.target_row_off).copy()
    tro[1] += 1
    w2.target_row_off = tro
    db2 = DeviceBatch(w2)
    db2.args.set_workspace(db.ws)
    db2.run()
    g2 = db2.results()
    o2 = oracle.verify_sample(w2, seed=0, diagnostics=True)
    assert list(g2["status"]) == list(o2["status"]) == [4, 4, 0]
    db.run(rnd=0)
    r = db.results()
    for k in outs[0]:
        assert np.array_equal(outs[0][k], r[k])
