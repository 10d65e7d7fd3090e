"""Fit the row correlation c of the 8-row 'similar' workload and store it in similar_c.json.

The workload's rows are x_r = c*z0 + sqrt(1-c^2)*z_r (and the same for the residual), so
that the rows pick many of the same experts, as the correlated rows of a verify step do
(the `--similar` option in the Modifications table of the GLM-5.3 long-context indexer
page).  c is chosen by bisection so that the oracle's routing gives a repeat fraction
1 - D/(R*k) as close as possible to 0.40, D the number of distinct experts picked.

Only the oracle's norm, router and top-k are called.  Run:  python tests/golden/fit_similar_c.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from moe_layer_tail_gb300 import inputs as gen  # noqa: E402

TARGET = 0.40


def repeat_fraction(wl, w, c):
    a = gen.make_activations(wl.shape, wl.seed, "similar", c)
    _, n, _ = oracle.add_rmsnorm(a["x"], a["residual"], w["gamma"], wl.shape.eps)
    ids, _ = oracle.topk(oracle.router(n, w["w_r"]), wl.shape.k)
    D = len(np.unique(ids))
    return 1.0 - D / ids.size, D


def main():
    wl = gen.WORKLOADS["r8_h7168_e256k8_similar"]
    w = gen.make_weights(wl.shape, wl.seed, keys=("gamma", "w_r"))
    lo, hi = 0.0, 1.0
    best = None
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        f, D = repeat_fraction(wl, w, mid)
        if best is None or abs(f - TARGET) < abs(best[1] - TARGET):
            best = (mid, f, D)
        if f < TARGET:
            lo = mid
        else:
            hi = mid
    c, f, D = best
    rec = {"workload": wl.name, "c": round(c, 6), "repeat_fraction": f, "distinct_experts": D,
           "picks": wl.shape.R * wl.shape.k, "target": TARGET,
           "made_by": "tests/golden/fit_similar_c.py (oracle norm, router and top-k only)"}
    rec["repeat_fraction"], rec["distinct_experts"] = repeat_fraction(wl, w, rec["c"])
    with open(os.path.join(HERE, "similar_c.json"), "w") as fh:
        json.dump(rec, fh, indent=1)
    print(rec)


if __name__ == "__main__":
    main()
