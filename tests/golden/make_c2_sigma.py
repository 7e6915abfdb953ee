"""Writes tests/golden/c2_sigma.json: the draft-noise sigma of the 50257-vocab
Zipf workload at which the mean acceptance rate alpha = sum_x min(p, q) is 0.80
(alpha is the draft's overlap with the target, "Speculative decoding"
(mhtirogla.ai), Complexity and constants). p and q come from the oracle only.

Run: python tests/golden/make_c2_sigma.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402
from speculative_decoding_verification_38_gb300 import workloads  # noqa: E402


def alpha(sigma: float) -> float:
    w = workloads.sampling_workload("tune", config=2, batch=1, vocab=50257, gammas=[4],
                                    profile="zipf", dtype="f32", sigma=sigma, temps=1.0, pool=1)
    vals = []
    for i in range(4):
        _, p = oracle.softmax_row(w.target[i], 1.0)
        _, q = oracle.softmax_row(w.draft[i], 1.0)
        vals.append(float(np.minimum(p, q).sum()))
    return float(np.mean(vals))


def main():
    lo, hi = 0.01, 3.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if alpha(mid) > 0.8:
            lo = mid
        else:
            hi = mid
    sigma = round(0.5 * (lo + hi) * 1024) / 1024  # a dyadic value, exact in float32
    out = {"sigma": sigma, "alpha_at_sigma": alpha(sigma), "target_alpha": 0.8,
           "workload": "zipf V=50257 fp32, B=1, gamma=4, T=1, PCG64(SeedSequence([0, 2]))"}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c2_sigma.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print(out)


if __name__ == "__main__":
    main()
