"""Find the scale c of the skewed-prefill workload's Zipf bias and store it.

The skewed workload (T=16384, d=7168, E=128, k=2) draws expert_bias[e] = c * ln p_{pi(e)} with
p_r proportional to r^-1.1 over a seeded random permutation pi.  Zipf's own top-3 share is only
~0.40, so c scales the bias until the three most-loaded experts hold ~60% of the T*k
assignments made before any capacity limit.  The share is measured with the oracle router on
the workload's own seeded x and W_g; c is found by bisection and written, with the share it
gives, to workloads/skew_calibration.json.

Run:  python -m oracle.calibrate_skew
This script calls only the oracle and the input generator (no GPU code).
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, _ROOT)

from oracle import moe_oracle as O  # noqa: E402
import workloads as W  # noqa: E402

TARGET = 0.60


def top3_share(logits, bias_unit, c, k):
    s = O.selection_scores(logits, O.BIAS_SELECT, expert_bias=c * bias_unit)
    # top-k via argpartition is enough for a load count (order inside the set is irrelevant)
    idx = np.argpartition(-s, k - 1, axis=1)[:, :k]
    counts = np.bincount(idx.reshape(-1), minlength=s.shape[1])
    return np.sort(counts)[::-1][:3].sum() / idx.size


def main():
    cfg = W.CONFIGS["skewed_cap"]
    inp = W.make_routing_inputs(cfg, zipf_scale=1.0)     # bias drawn with c = 1
    x = O.bf16_bits_to_f64(W.bf16_bits(inp["x"]))
    W_g = O.bf16_bits_to_f64(W.bf16_bits(inp["W_g"]))
    logits = O.router_logits(x, W_g)
    bias_unit = inp["bias"].double().numpy()
    lo, hi = 0.0, 8.0
    assert top3_share(logits, bias_unit, hi, cfg.k) > TARGET
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if top3_share(logits, bias_unit, mid, cfg.k) < TARGET:
            lo = mid
        else:
            hi = mid
    c = round(0.5 * (lo + hi), 6)
    share = float(top3_share(logits, bias_unit, c, cfg.k))
    out = {"c": c, "top3_share": share, "target": TARGET,
           "written_by": "python -m oracle.calibrate_skew",
           "x_sha256": W._sha(inp["x"]), "W_g_sha256": W._sha(inp["W_g"])}
    path = os.path.join(_ROOT, "workloads", "skew_calibration.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")
    print(json.dumps(out))


if __name__ == "__main__":
    main()
