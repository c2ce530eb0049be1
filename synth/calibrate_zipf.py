"""Find the router-bias temperature tau of the skewed long-prefill workload.

The workload adds b_e = tau * ln p_e (p_e a Zipf(1.1) popularity over a seeded
permutation of the 896 experts) to the router scores of 4096 tokens.  tau is
chosen by bisection so that the most loaded expert receives between 900 and
1100 of the 65,536 routed (token, slot) pairs.  Loads come from the fp64
oracle's routing only.  Writes synth/zipf_tau.json.

    python -m synth.calibrate_zipf
"""
from __future__ import annotations

import json
import os
import sys
import time

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
import synth  # noqa: E402


def max_load(s0: np.ndarray, logp: np.ndarray, tau: float, k: int, E: int):
    b = (tau * logp).astype(np.float32)
    s = s0 + b.astype(np.float64)[None, :]
    ids, _, _ = oracle.topk(s, k)
    offsets, _ = oracle.bucket(ids, E)
    loads = np.diff(offsets)
    return int(loads.max()), int(loads.min()), loads


def main():
    wl = synth.WORKLOADS["long"]
    t0 = time.time()
    # Inputs without the bias: the oracle adds the fp32 bias to fp64 scores.
    base = synth.Workload(wl.name, wl.T, wl.H, wl.E, wl.k, wl.I, wl.x_dtype, "uniform", wl.shared)
    inp = synth.make_inputs(base)
    s0 = oracle.router_logits(inp.x, inp.wr, None)
    logp = synth.zipf_log_popularity(wl)
    lo, hi = 0.0, 4.0
    target_lo, target_hi = 900, 1100
    tau = None
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        m, _, _ = max_load(s0, logp, mid, wl.k, wl.E)
        if target_lo <= m <= target_hi:
            tau = mid
            break
        if m < target_lo:
            lo = mid
        else:
            hi = mid
    if tau is None:
        raise SystemExit("bisection did not reach the target load window")
    m, mn, loads = max_load(s0, logp, tau, wl.k, wl.E)
    rec = {
        "tau": tau,
        "max_load": m,
        "min_load": mn,
        "active_experts": int(np.count_nonzero(loads)),
        "mean_load_active": float(loads[loads > 0].mean()),
        "alpha": synth.ZIPF_ALPHA,
        "T": wl.T, "E": wl.E, "k": wl.k, "seed": synth.SEED,
        "made_by": "python -m synth.calibrate_zipf (fp64 oracle routing)",
    }
    with open(synth.ZIPF_TAU_FILE, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps(rec), f"{time.time() - t0:.1f}s")


if __name__ == "__main__":
    main()
