"""Failure detection without a GPU fault: the bounded wait the fused verify
kernel uses between CTAs, run on a flag nothing sets, gives up within its
limit, reports it, and leaves the context usable; on a set flag it returns the
value at once."""
import time

import numpy as np
import pytest

from tests.test_gpu_parity import _harness, sv  # noqa: F401  (fixture)
from speculative_decoding_verification_38_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_wait_gives_up_on_a_flag_nothing_sets(sv):
    import torch

    flag = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    sv.check(sv.spec_debug_wait_probe(flag, 300_000_000, out), "wait probe")  # 0.3 s limit
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert out.cpu().tolist() == [0, 1]
    assert 0.25 < dt < 5.0, dt
    # the context is still usable: a verify call right after it matches the oracle
    from tests.test_gpu_parity import run_rounds
    w = wl.sampling_workload("after wait", config=402, batch=4, vocab=1031, gammas=np.array([2, 0, 3, 1]),
                             profile="zipf", dtype="bf16", sigma=0.5, temps=1.0, pool=1)
    run_rounds(w, range(2), seed=1, label="after a timed-out wait")


def test_wait_returns_a_set_flag(sv):
    import torch

    flag = torch.tensor([7, 0, 0, 0], dtype=torch.int32, device="cuda")
    out = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    sv.check(sv.spec_debug_wait_probe(flag, 1_000_000_000, out), "wait probe")
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [7, 0]


def test_wait_probe_rejects_bad_arguments(sv):
    import torch

    flag = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert sv.spec_debug_wait_probe(flag, 20_000_000_000, out) == sv.SPEC_ERR_INVALID_ARG
