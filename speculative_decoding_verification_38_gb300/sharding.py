"""Splitting verify work across ranks, one GPU each.

Sequences are independent, so the verify step shards by sequence with no
data-path exchange. Each rank verifies a contiguous range of sequences. The
rank passes that range's first global index as seq_offset, so every sequence
keeps the Philox draws it would get in the unsplit batch: the counter holds
seq_offset + b.

  * weak scaling (bench.py): every rank owns a batch of its own, and the rank
    with index r uses seq_offset = r * batch;
  * splitting one batch: shard() cuts a host Workload into `world` contiguous
    sequence ranges whose sizes differ by at most one.
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np

from .workloads import TreeWorkload, Workload


def seq_offset(rank: int, batch_per_rank: int) -> int:
    """First global sequence index of a rank that owns batch_per_rank sequences."""
    return int(rank) * int(batch_per_rank)


def shard_bounds(batch: int, rank: int, world: int) -> tuple[int, int]:
    """Sequences [b0, b1) of `rank` when `batch` sequences are split over `world` ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must be in [0, world)")
    base, extra = divmod(int(batch), int(world))
    b0 = rank * base + min(rank, extra)
    return b0, b0 + base + (1 if rank < extra else 0)


def shard(w: Workload, rank: int, world: int) -> tuple[Workload, int]:
    """This rank's part of a host workload and its seq_offset."""
    b0, b1 = shard_bounds(w.batch, rank, world)
    g = np.asarray(w.gammas, dtype=np.int64)
    if w.target_row_off is None:
        t0, t1 = b0 * (w.gamma_max + 1), b1 * (w.gamma_max + 1)
        d0, d1 = b0 * w.gamma_max, b1 * w.gamma_max
        tro = dro = None
    else:
        tro_g = np.asarray(w.target_row_off, dtype=np.int64)
        dro_g = np.asarray(w.draft_row_off, dtype=np.int64)
        t0, t1, d0, d1 = int(tro_g[b0]), int(tro_g[b1]), int(dro_g[b0]), int(dro_g[b1])
        tro, dro = tro_g[b0:b1 + 1] - t0, dro_g[b0:b1 + 1] - d0
    part = replace(
        w,
        batch=b1 - b0,
        gammas=np.asarray(g[b0:b1], dtype=np.int32),
        target=w.target[t0:t1],
        draft=None if w.draft is None else w.draft[d0:d1],
        draft_tokens=w.draft_tokens[d0:d1],
        token_pool=[t[d0:d1] for t in w.token_pool],
        temperatures=None if w.temperatures is None else w.temperatures[b0:b1],
        kv_in=None if w.kv_in is None else w.kv_in[b0:b1],
        top_ks=None if w.top_ks is None else w.top_ks[b0:b1],
        top_ps=None if w.top_ps is None else w.top_ps[b0:b1],
        target_row_off=tro,
        draft_row_off=dro,
    )
    return part, b0


def shard_tree(w: TreeWorkload, rank: int, world: int) -> tuple[TreeWorkload, int]:
    """This rank's part of a host tree workload (its trees, node offsets
    rebased to its first node) and its seq_offset."""
    b0, b1 = shard_bounds(w.batch, rank, world)
    off = np.asarray(w.node_off, dtype=np.int64)
    n0, n1 = int(off[b0]), int(off[b1])
    part = replace(
        w,
        batch=b1 - b0,
        node_off=off[b0:b1 + 1] - n0,
        parent=w.parent[n0:n1],
        tokens=w.tokens[n0:n1],
        target=w.target[n0:n1],
        draft=None if w.draft is None else w.draft[n0:n1],
        temperatures=None if w.temperatures is None else w.temperatures[b0:b1],
    )
    return part, b0
