"""The N > 1 path on two gloo ranks (CPU): sequence sharding with seq_offset
and the max-over-ranks timing reduction bench.py uses.

Each rank verifies its shard of one ragged batch with the oracle (standing in
for its GPU) at its seq_offset. Rank 0 gathers every shard's outputs and checks
them against one unsplit oracle call over the whole batch: sharding must not
change any draw or any output.
"""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch(case):
    from speculative_decoding_verification_38_gb300 import workloads as wl

    if case == "plain":
        return wl.config5(batch=7, gamma_max=4, vocab=3001)
    # per-sequence top-k and top-p, top-p alone among them: each shard must
    # carry its own sequences' k and p
    B = 7
    return wl.sampling_workload("sharded truncation", config=401, batch=B, vocab=1500,
                                gammas=np.array([3, 0, 4, 2, 4, 1, 3]), profile="zipf", dtype="bf16",
                                sigma=0.6, temps=np.linspace(0.7, 1.3, B).astype(np.float32), ragged=True, pool=4,
                                top_k=np.array([0, 20, 5, 0, 1500, 40, 0], np.int32),
                                top_p=np.array([0.9, 0.0, 0.5, 0.3, 0.8, 0.95, 0.0], np.float32))


def _worker(rank, world, port, out_path, case="plain"):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    import bench
    import oracle
    from speculative_decoding_verification_38_gb300 import sharding
    from speculative_decoding_verification_38_gb300 import workloads as wl

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = _batch(case)
        part, off = sharding.shard(w, rank, world)
        rnd = 3
        res = oracle.verify_sample(part, seed=11, rnd=rnd, seq_offset=off, draft_tokens=part.tokens_for_round(rnd))
        got = [None] * world
        dist.all_gather_object(got, {k: v.tolist() for k, v in res.items()})
        slowest = bench.max_over_ranks(10.0 + rank, dist, "cpu")
        if rank == 0:
            whole = oracle.verify_sample(w, seed=11, rnd=rnd, seq_offset=0, draft_tokens=w.tokens_for_round(rnd))
            ok = slowest == 10.0 + world - 1
            for k in ("tokens", "accepted", "status", "kv", "blocks"):
                if k not in whole:  # no KV lengths given: no kv or blocks outputs
                    continue
                joined = np.concatenate([np.asarray(g[k]) for g in got])
                ok = ok and np.array_equal(joined, whole[k])
            ok = ok and int(np.asarray(whole["accepted"]).sum()) > 0 and "tokens" in whole
            with open(out_path, "w") as f:
                f.write("ok" if ok else "mismatch")
    finally:
        dist.destroy_process_group()


def _tree_worker(rank, world, port, out_path):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    import oracle
    from speculative_decoding_verification_38_gb300 import sharding
    from speculative_decoding_verification_38_gb300 import workloads as wl

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = wl.ragged_tree_workload("sharded trees", config=11, batch=9, vocab=997, max_nodes=20, dtype="bf16",
                                    sigma=0.7, temps=np.linspace(0.6, 1.4, 9).astype(np.float32))
        part, off = sharding.shard_tree(w, rank, world)
        res = oracle.tree_verify(part, seed=4, rnd=2, seq_offset=off)
        got = [None] * world
        dist.all_gather_object(got, {k: v.tolist() for k, v in res.items()})
        if rank == 0:
            whole = oracle.tree_verify(w, seed=4, rnd=2, seq_offset=0)
            ok = True
            for k in ("tokens", "path", "accepted", "status"):
                ok = ok and np.array_equal(np.concatenate([np.asarray(g[k]) for g in got]), whole[k])
            ok = ok and int(whole["accepted"].max()) >= 1
            with open(out_path, "w") as f:
                f.write("ok" if ok else "mismatch")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_the_unsplit_trees(tmp_path, orc):
    """Tree verification sharded by tree with seq_offset draws what the
    unsplit batch draws (the uniforms are keyed by the global tree index)."""
    mp = pytest.importorskip("torch.multiprocessing")
    out = tmp_path / "result.txt"
    mp.spawn(_tree_worker, args=(2, _free_port(), str(out)), nprocs=2, join=True)
    assert out.read_text() == "ok"


def test_shard_bounds_cover_the_batch():
    from speculative_decoding_verification_38_gb300 import sharding

    for batch in (1, 7, 64):
        for world in (1, 2, 3, 8):
            spans = [sharding.shard_bounds(batch, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == batch
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b1 - b0 for b0, b1 in spans]
            assert max(sizes) - min(sizes) <= 1
    assert sharding.seq_offset(3, 64) == 192


@pytest.mark.parametrize("case", ["plain", "truncated"])
def test_two_gloo_ranks_reproduce_the_unsplit_batch(tmp_path, orc, case):
    mp = pytest.importorskip("torch.multiprocessing")
    out = tmp_path / "result.txt"
    mp.spawn(_worker, args=(2, _free_port(), str(out), case), nprocs=2, join=True)
    assert out.read_text() == "ok"
