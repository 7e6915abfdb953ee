"""GPU parity of adaptive gamma: the running acceptance that the verify calls
update in place, and spec_adapt_gamma's choice of the next gamma, both
bit-exact against the oracle (the same float32 / float64 operations in the
same order)."""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_38_gb300 import workloads as wl
from tests.test_gpu_parity import _harness, sv  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def _run_with_ema(w, rounds, lam, seed=0):
    import torch

    DeviceBatch = _harness()
    db = DeviceBatch(w, seed=seed)
    rng = np.random.default_rng(seed + 7)
    ema0 = rng.random(w.batch).astype(np.float32)
    ema = torch.from_numpy(ema0.copy()).cuda()
    db.args.set_accept_ema(ema, lam)
    want = ema0.copy()
    for r in rounds:
        db.run(rnd=r, pool_index=r)
        res = db.results()
        gam = None if w.target_row_off is None else np.diff(np.asarray(w.draft_row_off)).astype(np.int32)
        want = oracle.acceptance_ema(res["accepted"], gam, w.gamma_max, want, lam, status=res["status"])
        got = ema.cpu().numpy()
        assert np.array_equal(got, want), (r, np.nonzero(got != want)[0][:10])
    return want, ema0


def test_ema_sampling_c3_shape(sv):
    w = wl.config3(batch=32, vocab=32000, pool=4)
    final, start = _run_with_ema(w, range(6), 0.125)
    assert not np.array_equal(final, start)


def test_ema_ragged_with_errors(sv):
    """Ragged gamma (some 0), per-sequence temperatures, and sequences with a
    bad token: only status-OK sequences with gamma > 0 move."""
    rng = np.random.default_rng(11)
    B = 40
    gam = rng.integers(0, 9, size=B)
    gam[:3] = 0
    w = wl.sampling_workload("ema ragged", config=290, batch=B, vocab=5003, gammas=gam, profile="zipf",
                             dtype="bf16", sigma=rng.uniform(0.2, 2.0, B), temps=rng.uniform(0.5, 1.5, B),
                             ragged=True, pool=3)
    dro = np.asarray(w.draft_row_off)
    for t in w.token_pool:  # sequence 5 drafts an out-of-range token in every round
        if gam[5] > 0:
            t[dro[5]] = w.vocab + 3
    final, start = _run_with_ema(w, range(4), 0.3)
    assert final[5] == start[5] and np.array_equal(final[:3], start[:3])


def test_ema_greedy(sv):
    import torch

    DeviceBatch = _harness()
    w = wl.config4(batch=64, vocab=32000)
    db = DeviceBatch(w)
    ema0 = np.linspace(0, 1, 64, dtype=np.float32)
    ema = torch.from_numpy(ema0.copy()).cuda()
    db.args.set_accept_ema(ema, 0.25)
    db.run()
    res = db.results()
    want = oracle.acceptance_ema(res["accepted"], None, w.gamma_max, ema0, 0.25, status=res["status"])
    assert np.array_equal(ema.cpu().numpy(), want)


@pytest.mark.parametrize("B", [1, 64, 5000, 65536])
def test_adapt_gamma_matches_oracle(sv, B):
    import torch

    rng = np.random.default_rng(B)
    ema = rng.random(B).astype(np.float32)
    ema[: min(B, 6)] = np.array([0.0, 1.0, np.nan, 1.7, -0.2, 0.8], np.float32)[: min(B, 6)]
    d_ema = torch.from_numpy(ema).cuda()
    out = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    tot = torch.zeros(1, dtype=torch.int64, device="cuda")
    for gmax in (0, 1, 8, 64):
        for c in (0.0, 0.02, 0.05, 0.3, 1.5):
            want, wt = oracle.adapt_gamma(ema, gmax, c)
            sv.check(sv.spec_adapt_gamma(d_ema, gmax, c, out, total_positions_out=tot), "adapt_gamma")
            assert np.array_equal(out.cpu().numpy(), want), (gmax, c)
            assert int(tot.item()) == wt
    # the batch switch: one position under the unswitched total turns speculation off
    want, wt = oracle.adapt_gamma(ema, 8, 0.05)
    for budget in (wt, wt - 1, 0):
        w2, t2 = oracle.adapt_gamma(ema, 8, 0.05, max_positions=budget)
        sv.check(sv.spec_adapt_gamma(d_ema, 8, 0.05, out, max_positions=budget, total_positions_out=tot), "switch")
        assert np.array_equal(out.cpu().numpy(), w2) and int(tot.item()) == t2
