"""Calibrate the step-to-step query correlation rho that gives a target overlap of
consecutive top-k sets (the "controlled hit rate" of the synthetic workloads).

Calls only the oracle (indexer score and top-k) and the seeded input generator.
For each (context L, k, target overlap) it bisects rho in q_{t+1} = rho*q_t +
sqrt(1-rho^2)*eps, measuring the mean |topk_t & topk_{t+1}| / k over a few
requests and steps, and writes tests/golden/rho_calibration.json.

    python tests/golden/calibrate_rho.py            # all workload points
"""
import json
import multiprocessing as mp
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "rho_calibration.json")
POINTS = [  # (L, k, target overlap)
    (65536, 2048, 0.90),                                             # DeepSeek-V3.2 decode shape
    (32768, 2048, 0.85),                                             # multi-step replay
    (100000, 2048, 0.50),                                            # HBM-pressure / MTP
] + [(L, 2048, h) for L in (16384, 32768, 65536, 131072) for h in (0.5, 0.7, 0.9, 0.99)]   # sweep
REQUESTS, STEPS = 2, 3


def overlap(L, k, rho, seed=7):
    import oracle
    from sparse_attention_kv_fp8_gb300 import workload as wl
    inp = wl.indexer_inputs(REQUESTS, 1, L, L, seed=seed)
    qf = inp.q_float
    prev = None
    vals = []
    q = inp.q
    for step in range(STEPS + 1):
        if step:
            qf, q = wl.next_query(qf, rho, seed, step)
        s = oracle.indexer_score(q, inp.w, inp.k_index, inp.ctx_len)
        sel, _ = oracle.select_topk(s, inp.ctx_len, k)
        cur = [set(sel[b, 0].tolist()) for b in range(REQUESTS)]
        if prev is not None:
            vals += [len(a & b) / k for a, b in zip(prev, cur)]
        prev = cur
    return float(np.mean(vals))


def calibrate(point):
    # bisect x in rho = 1 - 10^-x (overlap grows with x; fine resolution near rho = 1)
    L, k, target = point
    lo, hi = 0.0, 6.0
    best = None
    for _ in range(13):
        mid = 0.5 * (lo + hi)
        rho = 1.0 - 10.0 ** -mid
        ov = overlap(L, k, rho)
        best = (rho, ov)
        if ov < target:
            lo = mid
        else:
            hi = mid
    return {"L": L, "k": k, "target_overlap": target, "rho": round(best[0], 7), "measured_overlap": round(best[1], 4),
            "requests": REQUESTS, "steps": STEPS}


if __name__ == "__main__":
    with mp.get_context("spawn").Pool(min(len(POINTS), os.cpu_count() or 1)) as pool:
        res = pool.map(calibrate, POINTS)
    json.dump({"source": "tests/golden/calibrate_rho.py (oracle indexer score + top-k only)", "points": res},
              open(OUT, "w"), indent=1)
    print(json.dumps(res, indent=1))
