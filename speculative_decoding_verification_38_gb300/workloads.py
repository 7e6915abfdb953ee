"""Seeded synthetic inputs for the verify step: the only module that both the
CUDA path's tests/bench and the float64 oracle consume.

It holds none of the verify arithmetic: no softmax normalisation, no accept
test, no residual, no inverse CDF, no argmax of the verify. It only draws
logits with numpy's PCG64, rounds them once to their storage dtype, and
simulates the drafter (step 1 of the decode round, outside the verify):

* sampling configs draw each draft token x_i ~ softmax(draft_logits_i / T) by
  the Gumbel-max trick (argmax of logits / T plus Gumbel noise), which never
  forms a probability vector;
* the greedy config's drafter picks the argmax of its own logits, which equal
  the target's logits with probability 0.75 per position.

Logit profiles (the five verify workloads):
  gaussian: l ~ N(0, 2^2) iid; draft = target + N(0, 0.5^2)             (C1)
  zipf:     l = -1.1 ln(rank) + N(0, 1), ranks 1..V randomly permuted per
            row; draft = target + N(0, sigma^2)                          (C2-C5)
Seeds: numpy PCG64(SeedSequence([dataset, config])).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# Draft-noise sigma of the 50257-vocab Zipf workload, chosen by bisection so that
# the mean acceptance rate sum_x min(p, q) over its rows is 0.80 at T = 1. The
# value is written by tests/golden/make_c2_sigma.py (which calls only the
# oracle) into tests/golden/c2_sigma.json; a test checks the two agree.
C2_SIGMA = 0.4853515625


def bf16_bits(x) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (NaN kept quiet)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    # uint32 arithmetic: u + 0x8000 overflows only for NaN patterns, set below
    u = x.view(np.uint32)
    t = (u >> 16) & 1
    t += 0x7FFF
    t += u
    t >>= 16
    r = t.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def stored_f32(a: np.ndarray) -> np.ndarray:
    """Values of a stored row block as float32 (exact for both storage dtypes)."""
    return bf16_to_f32(a) if a.dtype == np.uint16 else np.asarray(a, dtype=np.float32)


@dataclass
class Workload:
    """One batch of verify inputs, host-side (numpy), packed row-major.

    target [rows_target, V] and draft [rows_draft, V] are float32 or uint16 bf16
    bits. Sequence b owns target rows target_row_off[b] .. +gamma_b (gamma_b + 1
    rows, the last is the bonus position) and draft rows draft_row_off[b] ..
    +gamma_b - 1. Offsets are None when every gamma_b equals gamma_max.
    """

    name: str
    batch: int
    vocab: int
    gamma_max: int
    gammas: np.ndarray
    target: np.ndarray
    draft: np.ndarray | None
    draft_tokens: np.ndarray
    token_pool: list = field(default_factory=list)
    draft_is_probs: bool = False
    temperatures: np.ndarray | None = None
    temperature: float = 1.0
    kv_in: np.ndarray | None = None
    block_size: int = 0
    target_row_off: np.ndarray | None = None
    draft_row_off: np.ndarray | None = None
    greedy: bool = False
    info: dict = field(default_factory=dict)
    top_k: int = 0                    # top-k truncation of every row (0: off)
    top_ks: np.ndarray | None = None  # per-sequence k (int32 [B]) instead of top_k
    top_p: float = 0.0                # top-p, after top-k when that is on (active for 0 < p < 1)
    top_ps: np.ndarray | None = None  # per-sequence p (float32 [B]) instead of top_p

    @property
    def rows_target(self) -> int:
        return int(self.target.shape[0])

    @property
    def rows_draft(self) -> int:
        """Draft positions sum_b gamma_b (greedy keeps no draft logits, only tokens)."""
        return int(np.asarray(self.gammas, dtype=np.int64).sum())

    @property
    def dtype_name(self) -> str:
        return "bf16" if self.target.dtype == np.uint16 else "f32"

    def input_bytes(self) -> int:
        """Bytes of logits one verify call must read once (greedy: target only)."""
        n = self.target.nbytes
        if not self.greedy and self.draft is not None:
            n += self.draft.nbytes
        return int(n)

    def vocab_rows(self) -> int:
        return self.rows_target + (0 if self.greedy else self.rows_draft)

    def tokens_for_round(self, r: int) -> np.ndarray:
        if not self.token_pool:
            return self.draft_tokens
        return self.token_pool[r % len(self.token_pool)]


def _rng(config: int, dataset: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([dataset, config])))


def offsets_for(gammas: np.ndarray):
    g = np.asarray(gammas, dtype=np.int64)
    tro = np.zeros(g.shape[0] + 1, dtype=np.int64)
    dro = np.zeros(g.shape[0] + 1, dtype=np.int64)
    tro[1:] = np.cumsum(g + 1)
    dro[1:] = np.cumsum(g)
    return tro, dro


def zipf_rows(rng: np.random.Generator, rows: int, V: int, block: int = 256) -> np.ndarray:
    """-1.1 ln(rank) + N(0,1) with ranks 1..V permuted independently per row."""
    base = (-1.1 * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    out = np.empty((rows, V), dtype=np.float32)
    for r0 in range(0, rows, block):
        n = min(block, rows - r0)
        prof = rng.permuted(np.broadcast_to(base, (n, V)).copy(), axis=1)
        out[r0:r0 + n] = prof + rng.standard_normal((n, V), dtype=np.float32)
    return out


def gumbel_argmax(rng: np.random.Generator, logits_f32: np.ndarray, temps_per_row: np.ndarray,
                  block: int = 256, k_per_row: np.ndarray | None = None) -> np.ndarray:
    """Drafter simulation: one draw x ~ softmax(l / T) per row via Gumbel-max.
    With k_per_row, a drafter that samples from its own top k: row r draws
    only among its columns at least as large as its k-th largest logit
    (k <= 0 or k >= V: every column)."""
    rows, V = logits_f32.shape
    out = np.empty(rows, dtype=np.int32)
    for r0 in range(0, rows, block):
        n = min(block, rows - r0)
        u = rng.random((n, V), dtype=np.float32)
        with np.errstate(divide="ignore"):
            g = -np.log(-np.log(u))
        z = logits_f32[r0:r0 + n] / temps_per_row[r0:r0 + n, None] + g
        if k_per_row is not None:
            for i in range(n):
                k = int(k_per_row[r0 + i])
                if 0 < k < V:
                    row = logits_f32[r0 + i]
                    z[i, row < np.partition(row, V - k)[V - k]] = -np.inf
        out[r0:r0 + n] = np.argmax(z, axis=1)
    return out


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def sampling_workload(name: str, *, config: int, batch: int, vocab: int, gammas, profile: str,
                      dtype: str, sigma, temps, kv_range=None, block_size: int = 0,
                      ragged: bool = False, pool: int = 1, dataset: int = 0,
                      gauss_std: float = 2.0, top_k=0, top_p=0.0) -> Workload:
    """Generic sampling-verify workload; sigma, temps, top_k and top_p are
    scalars or [B] arrays. With top-k on, the simulated drafter samples from
    its top k (top-p is the verifier's: a draft token outside the nucleus has
    q = 0 there)."""
    rng = _rng(config, dataset)
    gammas = np.asarray(gammas, dtype=np.int32)
    gmax = int(gammas.max()) if gammas.size else 0
    tro, dro = offsets_for(gammas)
    rows_t, rows_d = int(tro[-1]), int(dro[-1])
    V = vocab
    if profile == "gaussian":
        tgt = (gauss_std * rng.standard_normal((rows_t, V), dtype=np.float32)).astype(np.float32)
    else:
        tgt = zipf_rows(rng, rows_t, V)
    sig = np.broadcast_to(np.asarray(sigma, dtype=np.float32), (batch,)).astype(np.float32)
    seq_of_t = np.repeat(np.arange(batch), gammas + 1)
    seq_of_d = np.repeat(np.arange(batch), gammas)
    # draft row (b, i) = target row (b, i) + N(0, sigma_b^2), before rounding
    src = tro[seq_of_d] + (np.arange(rows_d) - dro[seq_of_d])
    dft = np.empty((rows_d, V), dtype=np.float32)
    for r0 in range(0, rows_d, 256):
        n = min(256, rows_d - r0)
        noise = rng.standard_normal((n, V), dtype=np.float32)
        dft[r0:r0 + n] = tgt[src[r0:r0 + n]] + sig[seq_of_d[r0:r0 + n], None] * noise
    target = _store(tgt, dtype)
    draft = _store(dft, dtype)
    del tgt, dft
    if np.ndim(temps) == 0:
        temperatures, temperature = None, float(temps)
        t_rows = np.full(rows_d, float(temps), dtype=np.float32)
    else:
        temperatures = np.asarray(temps, dtype=np.float32)
        temperature = 1.0
        t_rows = temperatures[seq_of_d]
    dvals = stored_f32(draft)
    ks = None if np.ndim(top_k) == 0 else np.asarray(top_k, dtype=np.int32)
    k_rows = None
    if ks is not None:
        k_rows = ks[seq_of_d]
    elif 0 < int(top_k) < V:
        k_rows = np.full(rows_d, int(top_k), dtype=np.int32)
    token_pool = [gumbel_argmax(rng, dvals, t_rows, k_per_row=k_rows) for _ in range(max(1, pool))]
    kv = None
    if kv_range is not None:
        kv = rng.integers(kv_range[0], kv_range[1] + 1, size=batch).astype(np.int32)
    uniform = not ragged and bool(np.all(gammas == gmax))
    return Workload(
        name=name, batch=batch, vocab=V, gamma_max=gmax, gammas=gammas, target=target, draft=draft,
        draft_tokens=token_pool[0], token_pool=token_pool, temperatures=temperatures,
        temperature=temperature, kv_in=kv, block_size=block_size,
        target_row_off=None if uniform else tro, draft_row_off=None if uniform else dro,
        info={"sigma": sig, "config": config, "dataset": dataset, "profile": profile},
        top_k=int(top_k) if ks is None else 0, top_ks=ks,
        top_p=float(top_p) if np.ndim(top_p) == 0 else 0.0,
        top_ps=None if np.ndim(top_p) == 0 else np.asarray(top_p, dtype=np.float32),
    )


# ----------------------------------------------------------------- the five configs
def config1(batch=1, gamma=4, vocab=1000, pool=10000, dataset=0) -> Workload:
    """Sampling, B=1, gamma=4, V=1000, fp32, Gaussian logits, T=1."""
    return sampling_workload("C1 sample B1 g4 V1000 f32", config=1, batch=batch, vocab=vocab,
                             gammas=np.full(batch, gamma), profile="gaussian", dtype="f32",
                             sigma=0.5, temps=1.0, pool=pool, dataset=dataset)


def config2(batch=1, gamma=4, vocab=50257, pool=2000, dataset=0) -> Workload:
    """Sampling, B=1, gamma=4, V=50257, fp32, Zipf logits, sigma tuned to alpha~0.8, T=1."""
    return sampling_workload("C2 sample B1 g4 V50257 f32", config=2, batch=batch, vocab=vocab,
                             gammas=np.full(batch, gamma), profile="zipf", dtype="f32",
                             sigma=C2_SIGMA, temps=1.0, pool=pool, dataset=dataset)


def config3(batch=64, gamma=8, vocab=128256, pool=4, dataset=0, top_k=0, top_p=0.0) -> Workload:
    """Sampling, B=64, gamma=8, V=128256, bf16, Zipf, sigma_b ~ U[0.2,1.5], T=0.8
    (top_k > 0: the same rows, both models truncated to their top k)."""
    rng = _rng(30, dataset)
    sig = rng.uniform(0.2, 1.5, size=batch).astype(np.float32)
    name = "C3 sample B64 g8 V128256 bf16" + (f" top-k {top_k}" if top_k else "") + (f" top-p {top_p}" if top_p else "")
    return sampling_workload(name, config=3, batch=batch, vocab=vocab,
                             gammas=np.full(batch, gamma), profile="zipf", dtype="bf16",
                             sigma=sig, temps=0.8, kv_range=(512, 4096), block_size=16,
                             pool=pool, dataset=dataset, top_k=top_k, top_p=top_p)


def config5(batch=512, gamma_max=8, vocab=128256, pool=2, dataset=0) -> Workload:
    """Ragged sampling, B=512, gamma_b ~ U{1..8}, V=128256, bf16, packed with offsets."""
    rng = _rng(50, dataset)
    gammas = rng.integers(1, gamma_max + 1, size=batch).astype(np.int32)
    temps = rng.uniform(0.5, 1.5, size=batch).astype(np.float32)
    sig = rng.uniform(0.2, 2.0, size=batch).astype(np.float32)
    return sampling_workload("C5 ragged B512 g1..8 V128256 bf16", config=5, batch=batch,
                             vocab=vocab, gammas=gammas, profile="zipf", dtype="bf16", sigma=sig,
                             temps=temps, kv_range=(128, 32768), block_size=16, ragged=True,
                             pool=pool, dataset=dataset)


def config4(batch=256, gamma=5, vocab=152064, dataset=0, tie_every=8) -> Workload:
    """Greedy, B=256, gamma=5, V=152064, bf16 Zipf target; the drafter's logits
    equal the target's w.p. 0.75 per position, else an independent Zipf row."""
    rng = _rng(4, dataset)
    rows_t = batch * (gamma + 1)
    tgt = bf16_bits(zipf_rows(rng, rows_t, vocab))
    vals = bf16_to_f32(tgt)
    # inject explicit ties: copy the row maximum to a second random position
    tie_rows = np.arange(0, rows_t, tie_every)
    for r in tie_rows:
        j_star = int(np.argmax(vals[r]))
        j2 = int(rng.integers(0, vocab))
        if j2 == j_star:
            j2 = (j2 + 1) % vocab
        tgt[r, j2] = tgt[r, j_star]
    vals = bf16_to_f32(tgt)
    same = rng.random((batch, gamma)) < 0.75
    toks = np.empty((batch, gamma), dtype=np.int32)
    for b in range(batch):
        for i in range(gamma):
            if same[b, i]:
                toks[b, i] = int(np.argmax(vals[b * (gamma + 1) + i]))
            else:
                other = bf16_to_f32(bf16_bits(zipf_rows(rng, 1, vocab)))[0]
                toks[b, i] = int(np.argmax(other))
    kv = rng.integers(512, 4097, size=batch).astype(np.int32)
    draft_tokens = toks.reshape(-1)
    return Workload(
        name="C4 greedy B256 g5 V152064 bf16", batch=batch, vocab=vocab, gamma_max=gamma,
        gammas=np.full(batch, gamma, dtype=np.int32), target=tgt, draft=None,
        draft_tokens=draft_tokens, token_pool=[draft_tokens], kv_in=kv, block_size=16,
        greedy=True, info={"config": 4, "dataset": dataset, "tie_rows": tie_rows},
    )


def ngram_contexts(batch=64, doc_len=4096, gen_len=1024, vocab=128256, span=(8, 64), edit_prob=0.05,
                   dataset=0):
    """Contexts for the n-gram drafter: the edit / summarisation / RAG case
    where the output copies the input. Sequence b holds a document of
    doc_len tokens (Zipf-distributed ids, ranks permuted per sequence)
    followed by gen_len generated tokens made of spans copied from random
    places of the document, each token replaced by a fresh one with
    probability edit_prob. Returns (ctx int32, ctx_off int64 [B+1])."""
    rng = _rng(60, dataset)
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    w = 1.0 / ranks
    cdf = np.cumsum(w / w.sum())
    out = []
    for _ in range(batch):
        perm = rng.permutation(vocab).astype(np.int32)
        doc = perm[np.minimum(np.searchsorted(cdf, rng.random(doc_len)), vocab - 1)]
        gen = np.empty(0, np.int32)
        while gen.size < gen_len:
            n = int(rng.integers(span[0], span[1] + 1))
            s0 = int(rng.integers(0, max(1, doc_len - n)))
            piece = doc[s0:s0 + n].copy()
            edit = rng.random(piece.size) < edit_prob
            piece[edit] = perm[np.minimum(np.searchsorted(cdf, rng.random(int(edit.sum()))), vocab - 1)]
            gen = np.concatenate([gen, piece])
        out.append(np.concatenate([doc, gen[:gen_len]]))
    off = np.concatenate([[0], np.cumsum([a.size for a in out])]).astype(np.int64)
    return np.concatenate(out).astype(np.int32), off


@dataclass
class TreeWorkload:
    """Token trees to verify: sequence b owns nodes node_off[b] .. node_off[b+1]
    (node 0 of each the root, the last context token); parent[n] is the
    parent's local index (-1 for a root), tokens[n] the drafted token; one
    target row and one draft row per node (p and q after that node's path)."""
    name: str
    batch: int
    vocab: int
    node_off: np.ndarray
    parent: np.ndarray
    tokens: np.ndarray
    target: np.ndarray
    draft: np.ndarray
    draft_is_probs: bool = False
    temperatures: np.ndarray | None = None
    temperature: float = 1.0
    greedy: bool = False
    info: dict = field(default_factory=dict)

    @property
    def nodes(self) -> int:
        return int(self.node_off[-1])


def tree_shape(rng, branching, depth):
    """Parents (local indices, node 0 the root) of a tree whose nodes at depth
    d < depth have branching[d] children, the children of a node listed
    together, nodes in breadth-first order."""
    parent = [-1]
    level = [0]
    for d in range(depth):
        nxt = []
        for u in level:
            for _ in range(int(branching[d])):
                parent.append(u)
                nxt.append(len(parent) - 1)
        level = nxt
    return np.asarray(parent, np.int32)


def _tree_batch(name, rng, shapes, *, vocab, dtype, sigma, temps, profile, greedy_agree, info):
    """Rows and drafted tokens for trees of the given parent arrays (one per
    sequence): target rows Zipf (or Gaussian) logits per node, draft rows =
    target + N(0, sigma^2); each node's children drafted i.i.d. (with
    replacement) from the draft's softmax(q / T) at their parent by the
    Gumbel-max trick, or, with greedy_agree, a copy of the target's argmax
    at the parent with that probability."""
    batch = len(shapes)
    sizes = np.array([s.shape[0] for s in shapes], np.int64)
    node_off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    N = int(node_off[-1])
    tgt = zipf_rows(rng, N, vocab) if profile == "zipf" else (2.0 * rng.standard_normal((N, vocab))).astype(np.float32)
    dft = (tgt + np.float32(sigma) * rng.standard_normal((N, vocab), dtype=np.float32)).astype(np.float32)
    target, draft = _store(tgt, dtype), _store(dft, dtype)
    tv, dv = stored_f32(target), stored_f32(draft)
    T = np.broadcast_to(np.asarray(temps, np.float32), (batch,)).astype(np.float32)
    parent = np.concatenate(shapes).astype(np.int32)
    tokens = np.full(N, -1, np.int32)
    seq = np.repeat(np.arange(batch), sizes)
    kids = np.nonzero(parent >= 0)[0]
    at = node_off[seq[kids]] + parent[kids]  # each drafted node's parent row
    agree = (rng.random(kids.size) < greedy_agree) if greedy_agree is not None else np.zeros(kids.size, bool)
    tokens[kids[agree]] = np.argmax(tv[at[agree]], axis=1) if agree.any() else []
    rest = np.nonzero(~agree)[0]
    for c0 in range(0, rest.size, 256):
        c = rest[c0:c0 + 256]
        tokens[kids[c]] = gumbel_argmax(rng, dv[at[c]], T[seq[kids[c]]])
    return TreeWorkload(name=name, batch=batch, vocab=vocab, node_off=node_off, parent=parent, tokens=tokens,
                        target=target, draft=draft, temperatures=None if np.ndim(temps) == 0 else T,
                        temperature=float(temps) if np.ndim(temps) == 0 else 1.0, info=info)


def tree_workload(name, *, config, batch, vocab, branching, dtype="bf16", sigma=0.6, temps=1.0, profile="zipf",
                  dataset=0, greedy_agree=None) -> TreeWorkload:
    """The same tree, of the given per-depth branching, for every sequence
    (rows and tokens as _tree_batch)."""
    rng = _rng(70 + config, dataset)
    shape = tree_shape(rng, branching, len(branching))
    return _tree_batch(name, rng, [shape] * batch, vocab=vocab, dtype=dtype, sigma=sigma, temps=temps,
                       profile=profile, greedy_agree=greedy_agree,
                       info={"branching": list(branching), "config": config})


def ragged_tree_workload(name, *, config, batch, vocab, max_nodes, dtype="bf16", sigma=0.6, temps=1.0,
                         profile="zipf", greedy_agree=None) -> TreeWorkload:
    """Trees of different sizes: sequence b has 1..max_nodes nodes (the first
    a lone root, the last max_nodes), the parent of node v uniform over
    0..v-1 (rows and tokens as _tree_batch)."""
    rng = _rng(90 + config, 0)
    sizes = rng.integers(1, max_nodes + 1, size=batch)
    sizes[0], sizes[-1] = 1, max_nodes
    shapes = [np.array([-1] + [int(rng.integers(0, v)) for v in range(1, int(n))], np.int32) for n in sizes]
    return _tree_batch(name, rng, shapes, vocab=vocab, dtype=dtype, sigma=sigma, temps=temps, profile=profile,
                       greedy_agree=greedy_agree, info={"max_nodes": max_nodes, "config": config})


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}
