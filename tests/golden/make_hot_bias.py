"""Writes hot_bias.json: the router bias that gives the hot experts their share.

The large workload's hot-expert variant puts 25% of the T*R routing
assignments on 4 seeded experts.  Those experts get +beta added to their
logits; this script finds beta by bisection, routing with the CPU oracle on the
workload's own x and W_g (drawn by the seeded generators).  Only the oracle
computes here.  Run from the repository root:  python tests/golden/make_hot_bias.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from workloads import synth  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402

TARGET_SHARE = 0.25


def share(logits, hot, beta, R):
    l = logits.copy()
    l[:, hot] += np.float32(beta)
    idx, _ = O.route_topk(l, R)
    return float(np.isin(idx, hot).mean())


def main():
    wl = synth.workload("large_hot")
    x, w_gate, _ = synth.router_inputs(synth.workload("large"))   # same seeds, no bias
    logits = O.gate_logits(synth.bf16_bits(x), w_gate.numpy())
    hot = synth.hot_experts(wl).numpy()
    lo, hi = 0.0, 20.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if share(logits, hot, mid, wl.R) < TARGET_SHARE:
            lo = mid
        else:
            hi = mid
    beta = float(np.float32(hi))
    got = share(logits, hot, beta, wl.R)
    out = {"source": "bisection with the CPU oracle's router on the seeded large workload",
           "large_hot": {"beta": beta, "hot_experts": hot.tolist(), "share": got,
                         "target_share": TARGET_SHARE}}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "hot_bias.json"), "w") as fh:
        json.dump(out, fh, indent=1)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
