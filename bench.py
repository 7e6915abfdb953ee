#!/usr/bin/env python
"""Benchmark of the batched verify step: B=64, gamma=8, V=128256, bf16 logits.

One step = one spec_verify_sample call over the whole batch (the streaming
pass over all 1088 vocabulary rows, the accept scan, the residual / bonus
draw and the KV rollback). Inputs are resident in HBM; consecutive steps
alternate between two resident copies of the 279 MB input (larger than the
129 MB L2 on its own), so no step reads rows the previous step left in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--top-k K]

--top-k K truncates every target and draft row to its top K (the same rows;
the step's first kernel is then the top-k threshold pass).

Under torchrun each rank verifies its own batch of 64 sequences (weak
scaling; no collective on the data path, a barrier and a max-reduce of the
elapsed time only). The reference arm times the float64 CPU oracle on the
host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify rounds/s (B=64, gamma=8, V=128256, bf16 logits)"
UNIT = "rounds/s"
WORKLOAD = "C3 sampling verify B=64 gamma=8 V=128256 bf16 T=0.8 (Zipf logits, per-sequence draft noise)"
FALLBACK_HBM_GBS = 6800.0
HOOK_EVERY = 8  # steps per streaming-kernel timing sample inside the timed region
KERNEL_SAMPLES = 120  # event-bracketed launches of the dominant kernel timed after the timed region
E2E_COPY_STREAMS = 4  # streams the end-to-end measurement spreads its host-to-device copies over


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=60)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--top-k", type=int, default=0,
                    help="truncate every target and draft row to its top k (0: plain sampling, the headline)")
    ap.add_argument("--top-p", type=float, default=0.0,
                    help="keep each row's top-p nucleus (inside the top-k set with --top-k, else of the whole row; 0: off)")
    ap.add_argument("--ngram", action="store_true",
                    help="time the n-gram (prompt lookup) drafter instead of the verify step")
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5],
                    help="the workload: 3 (default) the B=64 headline; 1, 2 small sampling; 4 greedy; 5 ragged")
    ap.add_argument("--tree", action="store_true",
                    help="time tree verification (64 trees of branching 4, 2, 2) instead of the chain verify")
    ap.add_argument("--adaptive", action="store_true",
                    help="each step also updates the running acceptance and chooses the next gamma on the GPU")
    return ap.parse_args()


# The dominant kernel of each mode: its name, the sources whose hash keys the
# committed ncu DRAM summary, and that summary's file.
KERNELS = {
    "stats": {"name": "streaming pass (stats_tma_kernel; stats_kernel where rows are not on 16-byte boundaries)",
              "sources": ("stats.cu", "stream.cuh", "common.cuh", "internal.h", "precise.cuh"),
              "profile": "stats_kernel_c{c}_dram.txt"},
    "topk": {"name": "topk_kernel (top-k threshold pass)", "sources": ("topk.cu", "common.cuh", "internal.h"),
             "profile": "topk_kernel_c3_k{k}_dram.txt"},
    "ngram": {"name": "ngram_kernel (n-gram drafter)", "sources": ("ngram.cu", "common.cuh", "internal.h"),
              "profile": "ngram_kernel_edit_contexts_dram.txt"},
    "tree": {"name": "tree_kernel (tree verification)", "sources": ("tree.cu", "common.cuh", "internal.h", "precise.cuh"),
             "profile": "tree_kernel_bench_trees_dram.txt"},
    "topp": {"name": "topk_kernel (top-k threshold pass, storing each top-p row's kept values for nucleus_kernel)",
             "sources": ("topk.cu", "common.cuh", "internal.h", "precise.cuh"), "profile": "topk_kernel_c3_k{k}_p_dram.txt"},
    "whole": {"name": "whole_nucleus_kernel (top-p without top-k: each bf16 row's pattern counts, nucleus and sum "
                      "in one read of the row)",
              "sources": ("topk.cu", "common.cuh", "internal.h", "precise.cuh"),
              "profile": "whole_nucleus_kernel_c3_p09_dram.txt"},
}


def topp_on(args):
    return 0 < args.top_p < 1


def launches_per_step(greedy, mode, top_k, adaptive):
    """Kernels one timed step launches: the row pass (the streaming pass, the
    top-k pass with truncation, or the whole-row nucleus kernel for top-p
    without top-k) and the finalize; sampling adds the sampler's tile pass and
    the draw; top-p after top-k adds the nucleus kernel (the whole-row and
    alone kernels are not launched when top-k is on for every sequence);
    --adaptive adds the gamma policy."""
    n = 2 if greedy else 4
    if mode == "topp":
        n += 1
    return n + (1 if adaptive else 0)


def kernel_label(mode, args):
    """The roofline's kernel: the mode's dominant kernel."""
    return KERNELS[mode]["name"]


def mode_of(args):
    if topp_on(args):
        return "topp" if args.top_k > 0 else "whole"
    return "topk" if args.top_k > 0 else "stats"


# The other workloads of the scope table (C1, C2, C4, C5): descriptions and metrics.
CONFIGS = {
    1: ("C1 sampling verify B=1 gamma=4 V=1000 f32 T=1 (Gaussian logits, draft = target + N(0, 0.5^2))",
        "verify rounds/s (C1: B=1, gamma=4, V=1000, f32 logits)"),
    2: ("C2 sampling verify B=1 gamma=4 V=50257 f32 T=1 (Zipf logits, draft noise tuned to alpha ~ 0.8)",
        "verify rounds/s (C2: B=1, gamma=4, V=50257, f32 logits)"),
    4: ("C4 greedy verify B=256 gamma=5 V=152064 bf16 (Zipf target; draft token = the target's argmax w.p. 0.75)",
        "verify rounds/s (C4 greedy: B=256, gamma=5, V=152064, bf16 logits)"),
    5: ("C5 ragged sampling verify B=512 gamma_b ~ U{1..8} V=128256 bf16, T_b ~ U[0.5, 1.5], sigma_b ~ U[0.2, 2.0]",
        "verify rounds/s (C5 ragged: B=512, gamma_b in 1..8, V=128256, bf16 logits)"),
}
L2_BYTES = 129 << 20


def metric_of(args):
    if args.config != 3:
        return CONFIGS[args.config][1]
    if args.top_k <= 0 and not topp_on(args):
        return METRIC
    tk = f", top-k {args.top_k}" if args.top_k > 0 else ""
    return METRIC[:-1] + tk + (f", top-p {args.top_p}" if topp_on(args) else "") + ")"


def workload_of(args):
    if args.config != 3:
        return CONFIGS[args.config][0]
    if args.top_k <= 0 and not topp_on(args):
        return WORKLOAD
    if args.top_k <= 0:
        return WORKLOAD + f", both models truncated to their top-p {args.top_p} nucleus (no top-k)"
    w = WORKLOAD + f", both models truncated to top-k {args.top_k}"
    return w + (f" then top-p {args.top_p}" if topp_on(args) else "")


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        return rows

    @staticmethod
    def summarize(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable: nvidia-smi gave no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(mode: str = "stats") -> str:
    h = hashlib.sha256()
    for f in KERNELS[mode]["sources"]:
        with open(os.path.join(ROOT, "speculative_decoding_verification_38_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic_per_launch(mode: str = "stats", top_k: int = 0, config: int = 3):
    """DRAM bytes per launch of the mode's dominant kernel from the committed
    ncu summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", KERNELS[mode]["profile"].format(k=top_k, c=config))
    try:
        kv = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("source_hash") != kernel_source_hash(mode):
            return None
        return int(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def nvtx(name):
    """An NVTX range around one phase of a bench run (seen by a profiler's
    timeline; nothing otherwise)."""
    import contextlib

    import torch

    try:
        return torch.cuda.nvtx.range(name)
    except Exception:  # no NVTX in this build: the phase runs unmarked
        return contextlib.nullcontext()


def realised_acceptance(copies, w):
    """What the last call of each resident copy produced: tokens emitted per
    sequence and pass (accepted drafts + 1; greedy the same), and the fraction
    of accept tests passed (a rejection ends a sequence's tests)."""
    import numpy as np

    acc, tests, emitted, seqs = 0, 0, 0, 0
    g = np.asarray(w.gammas)
    for db in copies:
        r = db.results()
        ok = r["status"] == 0
        a = r["accepted"][ok].astype(np.int64)
        gg = g[ok].astype(np.int64)
        acc += int(a.sum())
        tests += int(np.where(a < gg, a + 1, gg).sum())
        emitted += int((a + 1).sum())
        seqs += int(ok.sum())
    return {"tokens_per_pass": emitted / max(seqs, 1), "accept_rate": acc / max(tests, 1),
            "sequences": seqs, "what": "the last call of each of the two resident copies"}


def draft_agreement(w):
    """The workload's acceptance rates alpha = sum_x min(p(x), q(x)) of each draft
    position against its target row, both at the sequence's temperature (float64,
    host side): the mean over positions, and a histogram of the per-sequence means
    in tenths of [0, 1]. A property of the synthetic inputs, reported beside the
    timing; nothing here runs on the GPU path."""
    import numpy as np
    from speculative_decoding_verification_38_gb300 import workloads as wl

    if w.greedy or w.draft_is_probs or w.rows_draft == 0:
        return None
    tro, dro = (np.asarray(w.target_row_off), np.asarray(w.draft_row_off)) if w.target_row_off is not None \
        else wl.offsets_for(w.gammas)
    temps = np.broadcast_to(np.asarray(w.temperatures if w.temperatures is not None else w.temperature,
                                       dtype=np.float64), (w.batch,))
    per_seq, alphas = [], []
    for b in range(w.batch):
        g = int(dro[b + 1] - dro[b])
        if g == 0:
            continue
        t = wl.stored_f32(w.target[int(tro[b]):int(tro[b]) + g]).astype(np.float64) / temps[b]
        d = wl.stored_f32(w.draft[int(dro[b]):int(dro[b]) + g]).astype(np.float64) / temps[b]
        pt = np.exp(t - t.max(axis=1, keepdims=True))
        pt /= pt.sum(axis=1, keepdims=True)
        qd = np.exp(d - d.max(axis=1, keepdims=True))
        qd /= qd.sum(axis=1, keepdims=True)
        a = np.minimum(pt, qd).sum(axis=1)
        alphas.extend(a.tolist())
        per_seq.append(float(a.mean()))
    hist = np.histogram(per_seq, bins=10, range=(0.0, 1.0))[0].tolist()
    return {"mean": float(np.mean(alphas)), "per_sequence_hist_tenths": hist,
            "what": "sum_x min(p, q) per draft position at the sequence's temperature; histogram of the "
                    "per-sequence means over [0, 1] in tenths"}


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of every rank's value (each rank gets the result)."""
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import numpy as np
    import torch

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    import __graft_entry__

    __graft_entry__.build()
    import speculative_decoding_verification_38_gb300 as sv
    from speculative_decoding_verification_38_gb300 import workloads as wl
    from speculative_decoding_verification_38_gb300.harness import DeviceBatch

    from speculative_decoding_verification_38_gb300.sharding import seq_offset

    mode = mode_of(args)
    if args.config == 3:
        w = wl.config3(top_k=args.top_k, top_p=args.top_p)
    else:
        if args.top_k > 0 or topp_on(args) or args.adaptive:
            raise SystemExit("--top-k, --top-p and --adaptive apply to the C3 workload only")
        w = wl.CONFIGS[args.config]()
    greedy = w.greedy
    small = 2 * w.input_bytes() < L2_BYTES  # C1, C2: both copies would stay in L2
    B = w.batch
    seq_off = seq_offset(rank, B)  # weak scaling: each rank verifies its own batch
    copies = [DeviceBatch(w, seed=0, seq_offset=seq_off) for _ in range(2)]
    gammas_next = None
    if args.adaptive:  # running acceptance per request, updated by every verify call
        for db in copies:
            db.args.set_accept_ema(torch.full((B,), 0.8, dtype=torch.float32, device="cuda"), 0.1)
        gammas_next = torch.zeros(B, dtype=torch.int32, device="cuda")
    algo_bytes = w.input_bytes()  # every logits row read once
    small_io = (w.rows_draft * 4 + B * 4 * 3 + w.rows_target * 4)  # tokens, kv in/out, accepted, out tokens
    torch.cuda.synchronize()

    def step(i, rnd):
        db = copies[i % 2]
        st = db.call(rnd=rnd, pool_index=rnd)
        if st != 0:
            raise sv.SpecError(st, "spec_verify_greedy" if greedy else "spec_verify_sample")
        if gammas_next is not None:  # the next round's gamma per request (the synthetic drafter keeps gamma = 8)
            sv.check(sv.spec_adapt_gamma(db.args.tensors["accept_ema"], w.gamma_max, 0.05, gammas_next),
                     "spec_adapt_gamma")

    W, K = max(3, args.warmup), max(1, args.steps)
    if small:
        K = min(K, 5000)  # each step is timed alone, between L2 flushes
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda") if small else None
    with nvtx("warm-up"):
        for i in range(W):
            step(i, i)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = ClockSampler(local_rank)
    clk.start()
    # every HOOK_EVERY-th step brackets its streaming kernel with events (the
    # events sit between the two kernels and cost that step its programmatic
    # launch overlap, so the other steps run unbracketed)
    hooked = list(range(0, K, HOOK_EVERY))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in hooked]
    for a, b in ev:  # torch creates the CUDA events lazily, on first record
        a.record()
        b.record()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)] \
        if small else []
    torch.cuda.synchronize()
    wall0 = time.time()
    with nvtx("timed steps"):
        t_start.record()
        for i in range(K):
            if small:  # inputs smaller than L2: evict them, then time this step alone
                flush.fill_(i & 255)
                step_ev[i][0].record()
            if i % HOOK_EVERY == 0:
                e0, e1 = ev[i // HOOK_EVERY]
                sv.spec_debug_time_next_stats(e0, e1)  # brackets this step's streaming kernel
            step(i, W + i)
            if small:
                step_ev[i][1].record()
        t_end.record()
        torch.cuda.synchronize()
    wall1 = time.time()
    if dist:
        dist.barrier()
    rows = clk.stop()
    in_window = [r for r in rows]
    clock_window = "timed region"
    if len(in_window) < 3:
        # the timed region was shorter than the sampler's period: sample an
        # adjacent window of the same steps instead
        clk2 = ClockSampler(local_rank)
        clk2.start()
        t0 = time.time()
        i = 0
        while time.time() - t0 < 1.2:
            for _ in range(200):
                step(i, W + K + i)
                i += 1
            torch.cuda.synchronize()
        rows = clk2.stop()
        clock_window = "adjacent 1.2 s window of identical steps (timed region shorter than the 200 ms sampler)"
    clocks = ClockSampler.summarize(rows)
    clocks["window"] = clock_window

    elapsed_ms = t_start.elapsed_time(t_end)
    if small:
        elapsed_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    stats_ms_in_region = [a.elapsed_time(b) for a, b in ev]
    # the dominant kernel alone: KERNEL_SAMPLES more steps after the timed
    # region, each bracketing that kernel with events; the median is reported
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(KERNEL_SAMPLES)]
    for a, b in kev:
        a.record()
        b.record()
    torch.cuda.synchronize()
    with nvtx("dominant kernel samples"):
        for i in range(KERNEL_SAMPLES):
            if small:
                flush.fill_(i & 255)
            sv.spec_debug_time_next_stats(kev[i][0], kev[i][1])
            step(i, W + K + i)
        torch.cuda.synchronize()
    stats_ms = [a.elapsed_time(b) for a, b in kev]
    realised = realised_acceptance(copies, w)
    if dist:
        elapsed_ms = max_over_ranks(elapsed_ms, dist, "cuda")
    ms_per_step = elapsed_ms / K
    rounds_per_s = world * K / (elapsed_ms / 1e3)
    kern_ms = statistics.median(stats_ms)
    peak, peak_kind = measured_hbm_peak()
    achieved = (algo_bytes + small_io) / (kern_ms / 1e3) / 1e9
    traffic = ncu_traffic_per_launch(mode, args.top_k, args.config)
    graph = time_graph(copies[0], W, flush, K) if small else None

    # end to end through the public API with host buffers
    with nvtx("end to end"):
        e2e = run_e2e(copies, w, args, sv) if args.e2e_steps > 0 else None

    out = {
        "metric": metric_of(args), "value": rounds_per_s, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded Zipf logits; no dataset)",
        "config": {"workload": workload_of(args), "batch": B, "gamma": w.gamma_max, "vocab": w.vocab,
                   "top_k": args.top_k, "top_p": args.top_p, "logits_dtype": w.dtype_name,
                   "parallelism": f"replicas x{world} (sequence shards)",
                   "l2": (f"inputs smaller than L2 ({w.input_bytes()} B): each step timed alone after a "
                          f"{2 * L2_BYTES >> 20} MB write that evicts them") if small else
                         (f"inputs larger than L2: {w.input_bytes() / 1e6:.0f} MB per step, "
                          "alternating 2 resident copies")},
        "vocab_rows_per_s": rounds_per_s * w.vocab_rows(),
        "sequence_rounds_per_s": rounds_per_s * B,
        "step_hbm_gbs": rounds_per_s / world * algo_bytes / 1e9,
        "gpu_launches": launches_per_step(greedy, mode, args.top_k, args.adaptive) * K,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": kernel_label(mode, args), "kernel_ms": kern_ms,
                     "kernel_ms_samples": len(stats_ms),
                     "kernel_ms_stat": "median of event-bracketed launches after the timed region",
                     "kernel_ms_in_timed_region": statistics.mean(stats_ms_in_region) if stats_ms_in_region else None,
                     "kernel_ms_in_timed_region_samples": len(stats_ms_in_region),
                     "algorithmic_bytes_per_launch": algo_bytes + small_io,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s"},
        "clocks": clocks,
        "e2e": e2e,
        "wall_s_timed": wall1 - wall0,
        "realised": realised,
    }
    if graph is not None:
        out["cuda_graph"] = graph
    if args.adaptive:
        out["adaptive_gamma"] = time_policy(sv, w.gamma_max)
        out["config"]["adaptive"] = "running acceptance (lambda 0.1) updated in finalize; gamma policy (c = 0.05) each step"
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        with nvtx("cpu baseline"):
            out["cpu_baseline"] = run_cpu_baseline(w, args)
    if rank == 0 and args.config in (2, 3) and args.top_k <= 0 and not topp_on(args):
        # the scope table asks for the C3 acceptance histogram and the C2 draft sigma
        out["config"]["acceptance"] = draft_agreement(w)
        if args.config == 2:
            out["config"]["draft_sigma"] = wl.C2_SIGMA
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


def time_graph(db, rnd, flush, K):
    """One verify call captured in a CUDA graph and replayed, each replay timed
    alone after an L2-evicting write (the launch-bound small workloads)."""
    import torch

    K = min(K, 2000)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st = db.call(rnd=rnd, pool_index=rnd)
        if st != 0:
            return {"unavailable": f"capture: verify returned status {st}"}
        for _ in range(3):
            g.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush.fill_(i & 255)
            ev[i][0].record()
            g.replay()
            ev[i][1].record()
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in ev)
        return {"value": K / (ms / 1e3), "unit": UNIT, "ms_per_step": ms / K, "steps": K,
                "note": "one captured call (fixed round) replayed"}
    except Exception as e:  # a capture the runtime refuses is reported, not fatal
        torch.cuda.synchronize()
        return {"unavailable": f"capture failed: {type(e).__name__}: {str(e)[:160]}"}


def time_policy(sv, gamma_max):
    """spec_adapt_gamma alone, CUDA-event timed over 500 calls per batch size."""
    import torch

    res = {}
    for B in (64, 4096, 65536):
        ema = torch.rand(B, device="cuda", dtype=torch.float32)
        g = torch.zeros(B, dtype=torch.int32, device="cuda")
        for _ in range(10):
            sv.check(sv.spec_adapt_gamma(ema, gamma_max, 0.05, g), "spec_adapt_gamma")
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(500):
            sv.spec_adapt_gamma(ema, gamma_max, 0.05, g)
        b.record()
        torch.cuda.synchronize()
        res[f"policy_us_B{B}"] = a.elapsed_time(b) * 1000 / 500
    res["bound"] = "latency: up to 65 dependent float32 speedups per request (one CTA up to 1024 requests)"
    return res


NGRAM_METRIC = "n-gram drafting rounds/s (B=64, contexts of 5120 tokens, n 3..1, gamma 8)"
NGRAM_WORKLOAD = ("edit-style contexts: 4096-token Zipf document + 1024 generated tokens copied from it in "
                  "8-64-token spans with 5% of tokens replaced; B=64")


def ngram_scanned_bytes(off, pos, mn, n_max, n_min):
    """Context bytes the single backward search must read at least once: one
    token per position from the end back to the continuation of an n_max
    match, or the whole context when no match reaches n_max."""
    total = 0
    for b in range(off.shape[0] - 1):
        L = int(off[b + 1] - off[b])
        if mn[b] == n_max:
            total += 4 * (L - (int(pos[b]) + n_max))
        else:
            total += 4 * L
    return total


def run_ngram(args):
    import numpy as np
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import speculative_decoding_verification_38_gb300 as sv
    from speculative_decoding_verification_38_gb300 import workloads as wl

    n_max, n_min, gamma, B = 3, 1, 8, 64
    ctx, off = wl.ngram_contexts(batch=B)
    copies = 128  # 128 x 1.3 MB: more than L2, and consecutive calls read different copies
    d_ctx = [torch.from_numpy(ctx).cuda() for _ in range(copies)]
    d_off = torch.from_numpy(off).cuda()
    draft = torch.empty(B * gamma, dtype=torch.int32, device="cuda")
    nd = torch.empty(B, dtype=torch.int32, device="cuda")
    pos = torch.empty(B, dtype=torch.int64, device="cuda")
    mn = torch.empty(B, dtype=torch.int32, device="cuda")

    def step(i):
        sv.check(sv.spec_ngram_draft(d_ctx[i % copies], d_off, n_max, n_min, gamma, draft, nd, pos, mn), "ngram")

    W, K = max(3, args.warmup), max(1, args.steps)
    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    clk = ClockSampler(0)
    clk.start()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(K):
        step(W + i)
    b.record()
    torch.cuda.synchronize()
    rows = clk.stop()
    ms = a.elapsed_time(b)
    clocks = ClockSampler.summarize(rows)
    scanned = ngram_scanned_bytes(off, pos.cpu().numpy(), mn.cpu().numpy(), n_max, n_min)
    peak, peak_kind = measured_hbm_peak()
    achieved = scanned / (ms / K / 1e3) / 1e9
    # end to end: contexts copied in from pinned host memory, drafts read back
    h_ctx = torch.from_numpy(ctx).pin_memory()
    h_draft = torch.empty(B * gamma, dtype=torch.int32).pin_memory()
    h_nd = torch.empty(B, dtype=torch.int32).pin_memory()
    n_e2e = max(3, args.e2e_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n_e2e):
        d_ctx[0].copy_(h_ctx, non_blocking=True)
        step(0)
        h_draft.copy_(draft, non_blocking=True)
        h_nd.copy_(nd, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    out = {
        "metric": NGRAM_METRIC, "value": K / (ms / 1e3), "unit": "rounds/s", "n_gpus": 1, "steps": K, "warmup": W,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic (seeded edit-style token contexts; no dataset)",
        "config": {"workload": NGRAM_WORKLOAD, "batch": B, "n_max": n_max, "n_min": n_min, "gamma": gamma,
                   "l2": "128 resident copies of the 1.3 MB contexts (168 MB), rotated"},
        "gpu_launches": K,
        "roofline": {"bound": "latency", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": ncu_traffic_per_launch("ngram"), "kernel": "ngram_kernel", "kernel_ms": ms / K,
                     "algorithmic_bytes_per_launch": scanned,
                     "note": "bytes = context tokens the backward search must read at least once (latest match first)",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
        "clocks": clocks,
        "e2e": {"value": n_e2e / (e2e_ms / 1e3), "unit": "rounds/s", "h2d_bytes_per_step": int(ctx.nbytes),
                "d2h_bytes_per_step": int(B * gamma * 4 + B * 4)},
    }
    if args.cpu_seconds > 0:
        import time as _t

        import oracle

        oracle.build()
        t0, n = _t.time(), 0
        while _t.time() - t0 < min(args.cpu_seconds, 5.0):
            oracle.ngram_draft(ctx, off, n_max, n_min, gamma)
            n += 1
        el = _t.time() - t0
        out["cpu_baseline"] = {"value": n / el, "unit": "rounds/s", "cores": 1, "kind": "oracle",
                               "sample": f"{n} full rounds of the same 64 contexts, C oracle, one thread"}
    print(json.dumps(out), flush=True)


TREE_SHAPE = dict(batch=64, vocab=128256, branching=[4, 2, 2], dtype="bf16", sigma=0.6, temps=0.8)
TREE_METRIC = "tree verify rounds/s (B=64 trees of 29 nodes, branching 4-2-2, V=128256, bf16 logits)"
TREE_WORKLOAD = ("token trees: B=64, branching (4, 2, 2) = 29 nodes per tree, V=128256 bf16, T=0.8; Zipf target "
                 "logits per node, draft = target + N(0, 0.6^2), children drafted i.i.d. from the draft at the parent")


def tree_read_bytes(w, res, row_bytes):
    """Rows the walk must read once: the target row of every visited node
    (the root and the accepted path) and the draft row of each visited node
    that has children."""
    total = 0
    off = w.node_off
    for b in range(w.batch):
        o, n = int(off[b]), int(off[b + 1] - off[b])
        par = w.parent[o:o + n]
        visited = [0] + [int(v) for v in res["path"][o:o + n] if v >= 0]
        has_kids = set(int(x) for x in par[1:])
        total += sum(row_bytes * (2 if u in has_kids else 1) for u in visited)
    return total


def run_tree(args):
    import numpy as np
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import speculative_decoding_verification_38_gb300 as sv
    from speculative_decoding_verification_38_gb300 import workloads as wl
    from speculative_decoding_verification_38_gb300.harness import DeviceTree

    w = wl.tree_workload("bench tree", config=20, **TREE_SHAPE)
    dt = DeviceTree(w, seed=0)
    copies = 4  # 4 x 952 MB resident: consecutive steps read different copies, none left in L2
    tgts = [dt.target] + [dt.target.clone() for _ in range(copies - 1)]
    dfts = [dt.draft] + [dt.draft.clone() for _ in range(copies - 1)]
    arg_sets = []
    for c in range(copies):
        dt.target, dt.draft = tgts[c], dfts[c]
        arg_sets.append([dt.args(rnd) for rnd in range(1)][0])
    dt.target, dt.draft = tgts[0], dfts[0]

    def step(i):
        a = arg_sets[i % copies]
        a.round = i
        sv.check(sv.spec_tree_verify(a, False), "tree verify")

    W, K = max(3, args.warmup), max(1, min(args.steps, 4000))
    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    clk = ClockSampler(0)
    clk.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(K):
        step(W + i)
    e1.record()
    torch.cuda.synchronize()
    rows = clk.stop()
    ms = e0.elapsed_time(e1)
    # the rows each timed round's walk read, from the same rounds replayed
    row_bytes = w.vocab * 2
    read = 0
    for i in range(K):
        step(W + i)
        read += tree_read_bytes(w, dt.results(), row_bytes)
    per_launch = read / K
    peak, peak_kind = measured_hbm_peak()
    achieved = per_launch / (ms / K / 1e3) / 1e9
    # end to end: every step copies the trees in from pinned host memory and reads the outputs back;
    # steps alternate between two of the resident row sets, so a step's row copies (over several copy
    # streams) run while the previous step's walk reads the other set
    host_t, host_d = tgts[0].cpu().pin_memory(), dfts[0].cpu().pin_memory()
    host_meta = [x.cpu().pin_memory() for x in (dt.node_off, dt.parent, dt.tokens)]
    out_h = [torch.empty_like(x, device="cpu").pin_memory() for x in
             (dt.out_tokens, dt.out_path, dt.out_accepted, dt.status)]
    h2d = host_t.numel() * 2 + host_d.numel() * 2 + sum(x.numel() * x.element_size() for x in host_meta)
    d2h = sum(x.numel() * 4 for x in out_h)
    n_e2e = max(3, min(args.e2e_steps, 30))
    cur = torch.cuda.current_stream()
    copy_streams = [torch.cuda.Stream() for _ in range(E2E_COPY_STREAMS)]
    sets = []
    for c in range(2):
        pieces = []
        for d, h in ((tgts[c], host_t), (dfts[c], host_d)):
            dv, hv = d.view(-1), h.view(-1)
            for o in range(0, dv.numel(), 16 << 20):  # 32 MB of bf16 per chunk
                pieces.append((dv[o:o + (16 << 20)], hv[o:o + (16 << 20)]))
        free = torch.cuda.Event()
        free.record(cur)
        sets.append((arg_sets[c], pieces, free))

    def one(i):
        a, pieces, free = sets[i % 2]
        for j, (d, h) in enumerate(pieces):
            cs = copy_streams[j % len(copy_streams)]
            if j < len(copy_streams):
                cs.wait_event(free)
            with torch.cuda.stream(cs):
                d.copy_(h, non_blocking=True)
        for cs in copy_streams:
            e = torch.cuda.Event()
            e.record(cs)
            cur.wait_event(e)
        for d, h in zip((dt.node_off, dt.parent, dt.tokens), host_meta):
            d.copy_(h, non_blocking=True)
        a.round = i
        sv.check(sv.spec_tree_verify(a, False), "tree verify")
        free.record(cur)
        for h, d in zip(out_h, (dt.out_tokens, dt.out_path, dt.out_accepted, dt.status)):
            h.copy_(d, non_blocking=True)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    e0.record()
    for i in range(n_e2e):
        one(i)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    acc = dt.results()["accepted"]
    out = {
        "metric": TREE_METRIC, "value": K / (ms / 1e3), "unit": "rounds/s", "n_gpus": 1, "steps": K, "warmup": W,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32x2",
        "data": "synthetic (seeded Zipf logits and drafted trees; no dataset)",
        "config": {"workload": TREE_WORKLOAD, "batch": w.batch, "nodes_per_tree": int(w.node_off[1]),
                   "vocab": w.vocab, "logits_dtype": "bf16",
                   "l2": "4 resident copies of the 952 MB rows, rotated (inputs larger than L2)",
                   "mean_accepted": float(np.mean(acc))},
        "gpu_launches": K,
        "roofline": {"bound": "latency", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": ncu_traffic_per_launch("tree"), "kernel": "tree_kernel", "kernel_ms": ms / K,
                     "algorithmic_bytes_per_launch": per_launch,
                     "note": "bytes = rows the walks must read once (visited nodes' target rows, draft rows of "
                             "visited nodes with children); a cluster of two CTAs per tree walks node by node",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
        "clocks": ClockSampler.summarize(rows),
        "e2e": {"value": n_e2e / (e2e_ms / 1e3), "unit": "rounds/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": n_e2e, "ms_per_step": e2e_ms / n_e2e,
                "h2d_gbs": h2d / (e2e_ms / n_e2e / 1e3) / 1e9,
                "copies": f"{len(sets[0][1])} chunks of at most 32 MB over {len(copy_streams)} copy streams per step; "
                          "two device row sets, so a step's copies overlap the previous step's walk"},
    }
    if args.cpu_seconds > 0:
        import oracle

        oracle.build()
        t0, n = time.time(), 0
        while time.time() - t0 < args.cpu_seconds and n < 50:
            oracle.tree_verify(w, seed=0, rnd=n)
            n += 1
        el = time.time() - t0
        out["cpu_baseline"] = {"value": n / el, "unit": "rounds/s", "cores": 1, "kind": "oracle",
                               "sample": f"{n} full rounds of the same 64 trees, float64 C oracle, one thread"}
    print(json.dumps(out), flush=True)


def run_e2e(copies, w, args, sv):
    """Same metric through the C ABI with inputs in pinned host memory: every
    step copies that step's inputs host -> device, verifies, and reads the
    outputs back device -> host, all inside the timed region. Steps alternate
    between the two device-resident input sets, so step i + 1's copies run
    while step i verifies (a serving loop's double buffering)."""
    import torch

    host_in = [d.cpu().pin_memory() for d in (copies[0].target, copies[0].draft, copies[0].kv_in) if d is not None]
    host_tok = [t.cpu().pin_memory() for t in copies[0].token_pool]
    h2d = sum(h.numel() * h.element_size() for h in host_in) + host_tok[0].numel() * 4
    n = max(3, args.e2e_steps)
    # The input rows go over in chunks of about 32 MB spread over several
    # copy streams, so that more than one copy engine moves them. The copies
    # into a set start once the verify that last read it is done; the verify
    # waits for all of its own step's copies.
    cur = torch.cuda.current_stream()
    copy_streams = [torch.cuda.Stream() for _ in range(E2E_COPY_STREAMS)]
    sets = []
    for db in copies:
        dev_in = [d for d in (db.target, db.draft, db.kv_in) if d is not None]
        pieces = []
        for d, h in zip(dev_in, host_in):
            dv, hv = d.view(-1), h.view(-1)
            step = max(1, (32 << 20) // dv.element_size())
            for o in range(0, dv.numel(), step):
                pieces.append((dv[o:o + step], hv[o:o + step]))
        outs = [(d, torch.empty_like(d, device="cpu").pin_memory())
                for d in (db.out_tokens, db.out_accepted, db.kv_out, db.status) if d is not None]
        free = torch.cuda.Event()
        free.record(cur)
        sets.append({"db": db, "pieces": pieces, "outs": outs, "free": free})
    d2h = sum(h.numel() * h.element_size() for _, h in sets[0]["outs"])

    def one(i):
        st = sets[i % len(sets)]
        db = st["db"]
        for j, (d, h) in enumerate(st["pieces"]):
            cs = copy_streams[j % len(copy_streams)]
            if j < len(copy_streams):
                cs.wait_event(st["free"])
            with torch.cuda.stream(cs):
                d.copy_(h, non_blocking=True)
        for cs in copy_streams:
            e = torch.cuda.Event()
            e.record(cs)
            cur.wait_event(e)
        tok = db.token_pool[i % len(db.token_pool)]
        tok.copy_(host_tok[i % len(host_tok)], non_blocking=True)
        rc = db.call(rnd=i, pool_index=i)
        if rc != 0:
            raise sv.SpecError(rc, "verify")
        st["free"].record(cur)
        for d, h in st["outs"]:
            h.copy_(d, non_blocking=True)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(n):
        one(i)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    return {"value": n / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": n, "ms_per_step": ms / n, "h2d_gbs": h2d / (ms / n / 1e3) / 1e9,
            "copies": f"{len(sets[0]['pieces'])} chunks of at most 32 MB over {len(copy_streams)} copy streams per "
                      f"step; two device input sets, so a step's copies overlap the previous step's verify"}


# ---------------------------------------------------------------- CPU / oracle
def _oracle_subset(w, nseq):
    """The first nseq sequences of a workload (views, no copies): rows up to
    the (nseq)-th offset, per-sequence arrays cut to nseq."""
    from speculative_decoding_verification_38_gb300 import workloads as wl

    g = w.gamma_max
    if w.target_row_off is None:
        rt, rd, tro, dro = nseq * (g + 1), nseq * g, None, None
    else:
        tro, dro = w.target_row_off[:nseq + 1], w.draft_row_off[:nseq + 1]
        rt, rd = int(tro[-1]), int(dro[-1])
    cut = (lambda a: None if a is None else a[:nseq])
    return wl.Workload(name=w.name, batch=nseq, vocab=w.vocab, gamma_max=g, gammas=w.gammas[:nseq],
                       target=w.target[:rt], draft=None if w.draft is None else w.draft[:rd],
                       draft_tokens=w.draft_tokens[:rd], temperatures=cut(w.temperatures),
                       temperature=w.temperature, kv_in=cut(w.kv_in), block_size=w.block_size,
                       target_row_off=tro, draft_row_off=dro, greedy=w.greedy, draft_is_probs=w.draft_is_probs,
                       top_k=w.top_k, top_ks=cut(w.top_ks), top_p=w.top_p, top_ps=cut(w.top_ps))


def run_cpu_baseline(w, args):
    import oracle

    oracle.build()
    cores = os.cpu_count() or 1
    rounds, t = 0, 0.0
    t0 = time.time()
    while t < args.cpu_seconds and rounds < 200:
        if w.greedy:
            oracle.verify_greedy(w, nthreads=cores)
        else:
            oracle.verify_sample(w, seed=0, rnd=rounds, draft_tokens=w.tokens_for_round(rounds), nthreads=cores)
        rounds += 1
        t = time.time() - t0
    # the same oracle on one host thread, over a bounded subset of one round's sequences
    sub = _oracle_subset(w, max(1, min(w.batch, w.batch // 8 or 1)))
    n1, t1 = 0, 0.0
    t0 = time.time()
    while t1 < min(6.0, args.cpu_seconds) and n1 < 50:
        if sub.greedy:
            oracle.verify_greedy(sub, nthreads=1)
        else:
            oracle.verify_sample(sub, seed=0, rnd=n1, draft_tokens=sub.draft_tokens, nthreads=1)
        n1 += 1
        t1 = time.time() - t0
    one_thread = (n1 * sub.batch / w.batch) / t1
    return {"value": rounds / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{rounds} full rounds of the same workload (all {w.batch} sequences each), float64 C "
                      f"oracle, one thread per sequence slice, {t:.1f} s",
            "value_1thread": one_thread,
            "sample_1thread": f"{n1} calls on the first {sub.batch} of the {w.batch} sequences (counted as "
                              f"{sub.batch}/{w.batch} round each), one host thread, {t1:.1f} s"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return  # rank 0 alone runs the CPU reference
    import oracle
    from speculative_decoding_verification_38_gb300 import workloads as wl

    oracle.build()
    if args.config == 3:
        w = wl.config3(top_k=args.top_k, top_p=args.top_p)
    else:
        w = wl.CONFIGS[args.config]()
    cores = os.cpu_count() or 1
    W, K = max(3, args.warmup), max(1, args.steps)

    def run(x, rnd):
        if x.greedy:
            oracle.verify_greedy(x, nthreads=cores)
        else:
            oracle.verify_sample(x, seed=0, rnd=rnd, draft_tokens=x.draft_tokens, nthreads=cores)

    # size each step so the whole run stays within ~3 minutes
    t0 = time.time()
    run(w, 0)
    t_round = time.time() - t0
    per_step = max(1, min(w.batch, int(w.batch * 150.0 / ((K + W) * max(t_round, 1e-3)))))
    sub = _oracle_subset(w, per_step)
    for i in range(W):
        run(sub, i)
    t0 = time.time()
    for i in range(K):
        run(sub, W + i)
    el = time.time() - t0
    value = (K * per_step / w.batch) / el
    out = {"impl": "reference", "metric": metric_of(args), "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
           "warmup": W, "ms_per_step": el / K * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded Zipf logits; no dataset)",
           "config": {"workload": workload_of(args), "batch": w.batch, "gamma": w.gamma_max, "vocab": w.vocab,
                      "top_k": args.top_k, "top_p": args.top_p, "logits_dtype": w.dtype_name,
                      "parallelism": "host cores"},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                            "sample": f"each step verifies {per_step} of the {w.batch} sequences of one round "
                                      f"(counted as {per_step}/{w.batch} round), float64 C oracle"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.ngram:
        run_ngram(args)
    elif args.tree:
        run_tree(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
