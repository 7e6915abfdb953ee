"""The bench's JSON contract on the host (no GPU): the reference arm's line
on the small workload, and the labels and launch counts the GPU arm reports
for each mode."""
import json
import os
import subprocess
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _ns(**kw):
    d = dict(top_k=0, top_p=0.0, config=3, adaptive=False)
    d.update(kw)
    return types.SimpleNamespace(**d)


def test_reference_arm_line(orc):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["metric"] == bench.CONFIGS[1][1] and d["config"]["workload"] == bench.CONFIGS[1][0]


def test_modes_and_labels():
    assert bench.mode_of(_ns()) == "stats"
    assert bench.mode_of(_ns(top_k=50)) == "topk"
    assert bench.mode_of(_ns(top_k=50, top_p=0.9)) == "topp"
    assert bench.mode_of(_ns(top_p=0.9)) == "whole"  # top-p without top-k
    assert bench.mode_of(_ns(top_p=1.0)) == "stats"  # p = 1 is off
    alone = _ns(top_p=0.9)
    assert "whole_nucleus_kernel" in bench.kernel_label("whole", alone)
    assert "whole_nucleus_kernel" not in bench.kernel_label("topp", _ns(top_k=50, top_p=0.9))
    assert "top-p 0.9" in bench.metric_of(alone) and "top-k" not in bench.metric_of(alone)
    assert "top-k 50" in bench.metric_of(_ns(top_k=50, top_p=0.9))
    assert bench.metric_of(_ns()) == bench.METRIC


def test_launches_per_step():
    L = bench.launches_per_step
    assert L(False, "stats", 0, False) == 4   # streaming pass, finalize, tile pass, draw
    assert L(True, "stats", 0, False) == 2    # greedy: streaming pass, finalize
    assert L(False, "topk", 50, False) == 4   # the top-k pass replaces the streaming pass
    assert L(False, "topp", 50, False) == 5   # + the nucleus kernel
    assert L(False, "whole", 0, False) == 4   # the whole-row nucleus kernel replaces the top-k pass
    assert L(False, "stats", 0, True) == 5    # + the gamma policy


def test_clock_summary_from_nvidia_smi_rows():
    S = bench.ClockSampler.summarize
    row = ["0", "2070", "2070", "900.1", "0x0000000000000000", "Not Active", "Not Active", "Not Active", "Not Active"]
    capped = row[:8] + ["Active"]
    slow = row[:5] + ["Active"] + row[6:]
    na = ["0", "[N/A]", "[N/A]", "[N/A]", "[N/A]", "[N/A]", "[N/A]", "[N/A]", "[N/A]"]
    out = S([row, row, capped])
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0 and out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 3
    low = [row[:1] + ["1200"] + row[2:]] * 3 + [row] * 2
    assert S(low)["sm_mhz"] == 1200.0  # the median under load, not the maximum
    assert S([row, slow])["reasons"] == ["hw_slowdown"]
    assert S([row, na])["sm_mhz"] == 2070.0  # unreadable fields are skipped
    assert S([])["reasons"][0].startswith("unavailable")


def test_traffic_only_while_the_source_hash_matches(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "stats_kernel_c3_dram.txt").write_text(
        "# a capture\nsource_hash: abc123\ndram_bytes_per_launch: 282213376\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda mode="stats": "abc123")
    assert bench.ncu_traffic_per_launch("stats", config=3) == 282213376
    assert bench.ncu_traffic_per_launch("stats", config=4) is None  # no capture for that config
    monkeypatch.setattr(bench, "kernel_source_hash", lambda mode="stats": "changed")
    assert bench.ncu_traffic_per_launch("stats", config=3) is None  # the kernel changed since


def test_committed_summaries_name_their_hash_and_bytes():
    """Every committed DRAM summary carries a hash line and a byte count
    (whether it still matches the sources is the bench's question)."""
    for mode, k in bench.KERNELS.items():
        name = k["profile"].format(k=50, c=3)
        path = os.path.join(ROOT, "profiles", name)
        if not os.path.exists(path):
            continue
        kv = dict(line.split(":", 1) for line in open(path) if ":" in line and not line.startswith("#"))
        assert len(kv["source_hash"].strip()) == 16 and int(kv["dram_bytes_per_launch"]) > 0, name


def test_reference_subset_is_the_batch_prefix(orc):
    """The reference arm times the oracle on the first n sequences: their
    outputs must be the whole batch's first n, per-sequence truncation and
    probability drafts included."""
    import numpy as np

    from speculative_decoding_verification_38_gb300 import workloads as wl

    B = 7
    w = wl.sampling_workload("subset", config=402, batch=B, vocab=700, gammas=np.array([3, 0, 4, 2, 4, 1, 3]),
                             profile="zipf", dtype="bf16", sigma=0.6, temps=np.linspace(0.7, 1.3, B).astype(np.float32),
                             ragged=True, pool=1, top_k=np.array([0, 20, 5, 0, 700, 40, 0], np.int32),
                             top_p=np.array([0.9, 0.0, 0.5, 0.3, 0.8, 0.95, 0.0], np.float32))
    dv = wl.stored_f32(w.draft)
    probs = np.exp(dv - dv.max(axis=1, keepdims=True)).astype(np.float32)
    wp = wl.Workload(**{**w.__dict__, "name": "subset probs", "draft": probs, "draft_is_probs": True})
    n = 4
    rows = int(w.target_row_off[n])
    for ww in (w, wp):
        for rnd in range(4):
            full = orc.verify_sample(ww, seed=3, rnd=rnd)
            part = orc.verify_sample(bench._oracle_subset(ww, n), seed=3, rnd=rnd)
            assert np.array_equal(part["accepted"], full["accepted"][:n])
            assert np.array_equal(part["tokens"], full["tokens"][:rows])
