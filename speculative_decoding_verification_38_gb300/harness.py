"""Device-resident verify batches for the tests and the benchmark.

DeviceBatch uploads one workloads.Workload to the GPU once, allocates the
outputs and the caller-owned workspace, and issues verify calls through the C
ABI (spec_verify_sample / spec_verify_greedy); DeviceTree does the same for a
workloads.TreeWorkload and spec_tree_verify. Nothing here computes any part
of the verify.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (SpecError, VerifyArgs, Workspace, check, spec_tree_verify, spec_verify_greedy, spec_verify_sample,
               tree_args)
from .workloads import TreeWorkload, Workload


def to_device_rows(a: np.ndarray, device) -> torch.Tensor:
    """float32 rows as-is; uint16 bf16 bit patterns reinterpreted as bfloat16."""
    if a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device)


class DeviceBatch:
    def __init__(self, w: Workload, device="cuda", uniforms: np.ndarray | None = None, seed: int = 0,
                 seq_offset: int = 0, workspace_slack: float = 1.0):
        self.w = w
        self.device = torch.device(device)
        dev = self.device
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)  # noqa: E731
        self.target = to_device_rows(w.target, dev)
        self.draft = to_device_rows(w.draft, dev) if (w.draft is not None and not w.greedy) else None
        pool = w.token_pool if w.token_pool else [w.draft_tokens]
        self.token_pool = [i32(t) for t in pool]
        self.tro = self.dro = None
        if w.target_row_off is not None:
            self.tro = torch.from_numpy(np.asarray(w.target_row_off, dtype=np.int64)).to(dev)
            self.dro = torch.from_numpy(np.asarray(w.draft_row_off, dtype=np.int64)).to(dev)
        self.temps = None if w.temperatures is None else torch.from_numpy(
            np.asarray(w.temperatures, dtype=np.float32)).to(dev)
        self.uniforms = None if uniforms is None else torch.from_numpy(
            np.ascontiguousarray(uniforms, dtype=np.float32)).to(dev)
        self.kv_in = None if w.kv_in is None else i32(w.kv_in)
        self.top_ks = None if w.top_ks is None else i32(w.top_ks)
        self.top_ps = None if getattr(w, "top_ps", None) is None else torch.from_numpy(
            np.asarray(w.top_ps, dtype=np.float32)).to(dev)
        B = w.batch
        self.kv_out = torch.full((B,), -7, dtype=torch.int32, device=dev) if self.kv_in is not None else None
        self.blocks = (torch.full((B,), -7, dtype=torch.int32, device=dev)
                       if (self.kv_in is not None and w.block_size > 0) else None)
        self.out_tokens = torch.full((w.rows_target,), -7, dtype=torch.int32, device=dev)
        self.out_accepted = torch.full((B,), -7, dtype=torch.int32, device=dev)
        self.status = torch.full((B,), -7, dtype=torch.int32, device=dev)
        self.args = VerifyArgs(
            batch=B, gamma_max=w.gamma_max, target=self.target, draft=self.draft, draft_tokens=self.token_pool[0],
            target_row_off=self.tro, draft_row_off=self.dro, draft_is_probs=w.draft_is_probs,
            temperatures=self.temps, temperature=w.temperature, seed=seed, round=0, seq_offset=seq_offset,
            uniforms=self.uniforms, kv_lens_in=self.kv_in, kv_lens_out=self.kv_out,
            block_size=w.block_size if self.blocks is not None else 0, out_num_blocks=self.blocks,
            out_tokens=self.out_tokens, out_accepted=self.out_accepted, seq_status=self.status,
            top_k=w.top_k, top_ks=self.top_ks, top_p=getattr(w, "top_p", 0.0), top_ps=self.top_ps)
        self.ws = Workspace.for_args(self.args, w.greedy, device=dev, slack=workspace_slack)
        self.args.set_workspace(self.ws)

    def call(self, rnd: int = 0, pool_index: int | None = None, stream=None) -> int:
        """Issue one verify call (asynchronous); returns the C status code."""
        self.args.set_round(rnd)
        if pool_index is not None:
            self.args.set_tokens(self.token_pool[pool_index % len(self.token_pool)])
        f = spec_verify_greedy if self.w.greedy else spec_verify_sample
        return f(self.args, stream)

    def run(self, rnd: int = 0, pool_index: int | None = None, stream=None):
        check(self.call(rnd, pool_index, stream), "verify")

    def results(self) -> dict:
        torch.cuda.synchronize(self.device)
        out = {"tokens": self.out_tokens.cpu().numpy(), "accepted": self.out_accepted.cpu().numpy(),
               "status": self.status.cpu().numpy()}
        if self.kv_out is not None:
            out["kv"] = self.kv_out.cpu().numpy()
        if self.blocks is not None:
            out["blocks"] = self.blocks.cpu().numpy()
        return out


class DeviceTree:
    """A TreeWorkload on the device with its outputs; run() is one
    spec_tree_verify launch over every sequence's tree."""

    def __init__(self, w: TreeWorkload, device="cuda", seed: int = 0, seq_offset: int = 0):
        self.w = w
        self.device = dev = torch.device(device)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)  # noqa: E731
        self.node_off = torch.from_numpy(np.ascontiguousarray(w.node_off, dtype=np.int64)).to(dev)
        self.parent = i32(w.parent)
        self.tokens = i32(w.tokens)
        self.target = to_device_rows(w.target, dev)
        self.draft = None if (w.greedy or w.draft is None) else to_device_rows(w.draft, dev)
        self.temps = None if w.temperatures is None else torch.from_numpy(
            np.asarray(w.temperatures, dtype=np.float32)).to(dev)
        n = self.target.shape[0]
        self.out_tokens = torch.full((n,), -7, dtype=torch.int32, device=dev)
        self.out_path = torch.full((n,), -7, dtype=torch.int32, device=dev)
        self.out_accepted = torch.full((w.batch,), -7, dtype=torch.int32, device=dev)
        self.status = torch.full((w.batch,), -7, dtype=torch.int32, device=dev)
        self.seed, self.seq_offset = seed, seq_offset

    def args(self, rnd: int = 0):
        return tree_args(node_off=self.node_off, parent=self.parent, tokens=self.tokens, target=self.target,
                         draft=self.draft, draft_is_probs=self.w.draft_is_probs, temperatures=self.temps,
                         temperature=self.w.temperature, seed=self.seed, rnd=rnd, seq_offset=self.seq_offset,
                         out_tokens=self.out_tokens, out_accepted=self.out_accepted, out_path=self.out_path,
                         seq_status=self.status)

    def call(self, rnd: int = 0, stream=None, args=None) -> int:
        return spec_tree_verify(args if args is not None else self.args(rnd), self.w.greedy, stream)

    def run(self, rnd: int = 0, stream=None):
        check(self.call(rnd, stream), "tree verify")

    def results(self) -> dict:
        torch.cuda.synchronize(self.device)
        return {"tokens": self.out_tokens.cpu().numpy(), "accepted": self.out_accepted.cpu().numpy(),
                "path": self.out_path.cpu().numpy(), "status": self.status.cpu().numpy()}


__all__ = ["DeviceBatch", "DeviceTree", "to_device_rows", "SpecError"]
