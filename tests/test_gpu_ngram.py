"""GPU parity of the n-gram (prompt lookup) drafter: bit-exact against the
oracle on random and edit-style contexts, long contexts that force a full
scan, and its drafts fed to the greedy verify."""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_38_gb300 import workloads as wl
from tests.test_gpu_parity import sv  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def _gpu_draft(sv, ctx, off, n_max, n_min, gamma):
    import torch

    B = off.shape[0] - 1
    d_ctx = torch.from_numpy(np.ascontiguousarray(ctx, np.int32)).cuda() if ctx.size else None
    d_off = torch.from_numpy(np.ascontiguousarray(off, np.int64)).cuda()
    draft = torch.full((max(B * gamma, 1),), -7, dtype=torch.int32, device="cuda")
    nd = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    pos = torch.full((B,), -7, dtype=torch.int64, device="cuda")
    mn = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    sv.check(sv.spec_ngram_draft(d_ctx, d_off, n_max, n_min, gamma, draft, nd, pos, mn), "spec_ngram_draft")
    torch.cuda.synchronize()
    return {"draft": draft.cpu().numpy()[:B * gamma].reshape(B, gamma), "n_draft": nd.cpu().numpy(),
            "match_pos": pos.cpu().numpy(), "match_n": mn.cpu().numpy()}


def _same(g, o):
    for k in ("draft", "n_draft", "match_pos", "match_n"):
        assert np.array_equal(g[k], o[k]), (k, np.nonzero(np.asarray(g[k]) != np.asarray(o[k]))[0][:10])


def test_random_contexts(sv):
    rng = np.random.default_rng(1)
    for trial in range(25):
        B = int(rng.integers(1, 300))
        lens = rng.integers(0, 3000, size=B)
        lens[0] = 0
        vocab = int(rng.choice([2, 3, 8, 50, 5000, 128256]))
        ctx = rng.integers(0, vocab, size=int(lens.sum())).astype(np.int32)
        off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        n_max = int(rng.integers(1, 17))
        n_min = int(rng.integers(1, n_max + 1))
        gamma = int(rng.integers(0, 65))
        _same(_gpu_draft(sv, ctx, off, n_max, n_min, gamma), oracle.ngram_draft(ctx, off, n_max, n_min, gamma))


def test_edit_style_contexts(sv):
    ctx, off = wl.ngram_contexts(batch=64)
    for n_max, n_min, gamma in ((3, 1, 8), (5, 2, 16), (1, 1, 4)):
        g = _gpu_draft(sv, ctx, off, n_max, n_min, gamma)
        _same(g, oracle.ngram_draft(ctx, off, n_max, n_min, gamma))
        # copied text repeats (an edited token in a longer suffix can hide the copy)
        assert (g["n_draft"] > 0).mean() > (0.9 if n_min == 1 else 0.75)


def test_long_contexts_full_scan(sv):
    """No repeat anywhere (a full scan for every n), a repeat only at the very
    start, and a repeat right before the suffix."""
    L = 200_000
    base = np.arange(L, dtype=np.int32)  # all distinct
    start = base.copy()
    start[-2:] = start[:2]  # the suffix "0 1" also opens the context
    near = base.copy()
    near[-3:] = [7, 7, 7]  # "7 7" at L-3 overlaps the suffix
    ctx = np.concatenate([base, start, near])
    off = np.array([0, L, 2 * L, 3 * L], np.int64)
    g = _gpu_draft(sv, ctx, off, 4, 1, 8)
    _same(g, oracle.ngram_draft(ctx, off, 4, 1, 8))
    assert g["match_pos"].tolist() == [-1, 0, L - 3]


def test_drafts_feed_greedy_verify(sv):
    """Drafts (ragged: each sequence drafts what it found) verified greedily
    against target rows whose argmax follows the document: the GPU verify
    agrees with the oracle's on the same tokens, and copies are accepted."""
    from speculative_decoding_verification_38_gb300.harness import DeviceBatch

    ctx, off = wl.ngram_contexts(batch=32, doc_len=2048, gen_len=256, vocab=32000, edit_prob=0.02)
    g = _gpu_draft(sv, ctx, off, 3, 1, 8)
    gam = g["n_draft"].astype(np.int32)
    tro, dro = wl.offsets_for(gam)
    toks = np.concatenate([g["draft"][b, :gam[b]] for b in range(32)]).astype(np.int32)
    V = 32000
    rng = np.random.default_rng(4)
    tgt = rng.standard_normal((int(tro[-1]), V)).astype(np.float32)
    for b in range(32):  # the target agrees with the first half of each draft, then disagrees
        for i in range(gam[b] + 1):
            r = tro[b] + i
            if i < gam[b] and i < (gam[b] + 1) // 2:
                tgt[r, toks[dro[b] + i]] = 10.0
    w = wl.Workload(name="ngram greedy", batch=32, vocab=V, gamma_max=int(gam.max()), gammas=gam,
                    target=wl.bf16_bits(tgt), draft=None, draft_tokens=toks, token_pool=[toks], greedy=True,
                    target_row_off=tro, draft_row_off=dro)
    db = DeviceBatch(w)
    db.run()
    res = db.results()
    ref = oracle.verify_greedy(w)
    assert np.array_equal(res["tokens"], ref["tokens"]) and np.array_equal(res["accepted"], ref["accepted"])
    assert (res["accepted"] == (gam + 1) // 2).sum() >= 28
