"""Tune each workload's target-noise scale tau so its mean acceptance probability hits alpha.

Writes ``workloads/tau.json``.  Calls only the oracle (for the row distributions) and the input
generator; nothing here touches the CUDA library.

For a draft position j the acceptance probability of the verify rule (accept with probability
min(1, p/q), cf-1.com §2.2) is alpha_j = sum_x q(x) min(1, p(x)/q(x)) = sum_x min(p(x), q(x)).
tau is found by bisection so that the mean of alpha_j over the draft rows of the first
``--requests`` requests lies within 0.005 of the workload's alpha (alpha falls as tau grows).

Usage:  python oracle/tune_tau.py [--requests 16] [--only c3,c5_a0.8]
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import oracle  # noqa: E402
import workloads as W  # noqa: E402


def mean_alpha(w: W.Workload, tau: float, requests: int) -> float:
    d = W.generate(w, requests=range(min(requests, w.B)), tau=tau)
    vals = []
    for i in range(d["p"].shape[0]):
        for j in range(int(d["k_per_row"][i])):
            P, _, fp = oracle.row_dist(d["p"][i, j], w.temperature, w.top_k, w.top_p)
            Q, _, fq = oracle.row_dist(d["q"][i, j], w.tq, w.top_k, w.top_p)
            assert not (fp | fq) & oracle.FLAG_NONFINITE
            vals.append(np.minimum(P, Q).sum())
    return float(np.mean(vals))


def tune(w: W.Workload, requests: int, lo: float = 0.0, hi: float = 8.0, tol: float = 0.005):
    a = None
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        a = mean_alpha(w, mid, requests)
        if abs(a - w.alpha) <= tol and hi - lo < 1e-3:
            return mid, a
        if a > w.alpha:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi), a


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--requests", type=int, default=16)
    ap.add_argument("--only", default="")
    args = ap.parse_args()
    table = W.load_tau()
    achieved = {}
    if os.path.exists(W.TAU_FILE):
        with open(W.TAU_FILE) as f:
            achieved = json.load(f).get("alpha_on_tuning_subset", {})
    names = [n for n, w in W.WORKLOADS.items() if w.alpha is not None and not w.greedy]
    if args.only:
        names = [n for n in names if n in args.only.split(",")]
    for n in names:
        w = W.WORKLOADS[n]
        t0 = time.time()
        tau, a = tune(w, args.requests)
        table[w.key] = round(tau, 5)
        achieved[w.key] = round(mean_alpha(w, table[w.key], args.requests), 4)
        print(f"{w.key}: tau={table[w.key]} alpha={achieved[w.key]} (target {w.alpha}) "
              f"{time.time() - t0:.1f}s", flush=True)
    with open(W.TAU_FILE, "w") as f:
        json.dump({"written_by": "oracle/tune_tau.py", "requests_per_workload": args.requests,
                   "tau": table, "alpha_on_tuning_subset": achieved}, f, indent=1, sort_keys=True)
        f.write("\n")


if __name__ == "__main__":
    main()
