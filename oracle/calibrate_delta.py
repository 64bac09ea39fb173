"""Calibrate the skip scale Delta of each workload on the float64 oracle.

The workloads state a stage-2 budget (the fraction of causal blocks that end up
computed) but the method only exposes the skip scale Delta of the threshold
ln(Delta / N) (CoSA Sec. 3.3 Eq. (5); App. D.1).  This script runs the oracle's
KAP and OSK over a seeded sample of (request, head, query block) items for each
Delta of a grid and keeps the smallest Delta whose realised budget is at or under
the target; if none is, it keeps the largest Delta of the grid below the shortest
request length.  The 2K single-head workload uses Delta = 2000, the paper's
Qwen3-8B operating point (App. D.1), for its skip-on case.

Writes tests/golden/delta_calibration.json.  Calls only the oracle (and the
seeded input generator).  Run:  python -m oracle.calibrate_delta
"""
from __future__ import annotations

import json
import math
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import cosa_oracle as orc  # noqa: E402

GRID = [100, 200, 300, 500, 700, 1000, 1500, 2000, 3000, 4000, 5000, 6000, 7000, 8000, 10000,
        15000, 20000]
PAPER_DELTA_QWEN = 2000.0
PAPER_DELTA_WORKLOAD = "2k_d64_1head"   # the single-head 2K workload takes the paper's Delta
SAMPLE_ITEMS = 384
SAMPLE_SEED = 777


def sample_items(spec):
    b = spec.block_size
    items = [(bi, h, i) for bi, L in enumerate(spec.lengths) for h in range(spec.num_q_heads)
             for i in range(-(-L // b))]
    if len(items) <= 4096:
        return items, "all"
    rng = np.random.default_rng(SAMPLE_SEED)
    pick = rng.choice(len(items), size=SAMPLE_ITEMS, replace=False)
    return sorted(items[k] for k in pick), f"{SAMPLE_ITEMS} items drawn uniformly (seed {SAMPLE_SEED})"


def calibrate(name: str, log=print) -> dict:
    spec = synth.spec_for(name)
    t0 = time.time()
    w = synth.make_workload(spec)
    items, how = sample_items(spec)
    G = spec.num_q_heads // spec.num_kv_heads
    scale = 1.0 / math.sqrt(spec.head_dim)
    min_len = min(spec.lengths)
    grid = [d for d in GRID if d < min_len]
    prm0 = orc.Params(spec.block_size, spec.page_size, spec.stride, spec.budget_ppm, scale, -1.0)
    groups = {}
    for (bi, h, i) in items:
        groups.setdefault((bi, h), []).append(i)
    computed = {d: 0 for d in grid}
    cand = 0
    for (bi, h), qbs in groups.items():
        L = spec.lengths[bi]
        Q = orc.request_queries(w.q, w.cu_seqlens, bi, h)
        K, ex = orc.request_keys(w.k_cache, w.page_table[bi], L, spec.page_size, h // G)
        V, _ = orc.request_keys(w.v_cache, w.page_table[bi], L, spec.page_size, h // G)
        rows = orc.kap_request_head(Q, K, ex, prm0, qbs)
        for i, row in rows.items():
            cand += i + 1
            for d in grid:
                prm = orc.Params(spec.block_size, spec.page_size, spec.stride, spec.budget_ppm, scale, float(d))
                r = orc.osk_qblock(Q, K, V, ex, i, row.order[:row.K], row.K, prm)
                computed[d] += int((r.flags == orc.COMPUTED).sum())
    curve = {str(d): computed[d] / cand for d in grid}
    target = spec.stage2_budget_ppm / 1e6
    ok = [d for d in grid if computed[d] / cand <= target]
    delta = float(min(ok)) if ok else float(max(grid))
    log(f"{name}: delta {delta} realized {curve[str(int(delta))]:.4f} target {target} "
        f"({len(items)} items, {time.time() - t0:.0f}s)")
    return {"delta": delta, "realized_budget": curve[str(int(delta))], "target_budget": target,
            "target_met": bool(ok), "curve": curve, "sample": how, "num_items": len(items)}


def main():
    out = {
        "what": "skip scale Delta per workload, calibrated on the float64 oracle (CoSA Eq. (5), App. D.1)",
        "script": "oracle/calibrate_delta.py",
        "grid": GRID,
        "workloads": {},
    }
    names = sys.argv[1:] or list(synth.WORKLOADS)
    path = os.path.join(ROOT, "tests", "golden", "delta_calibration.json")
    if os.path.exists(path):
        out["workloads"].update(json.load(open(path)).get("workloads", {}))
    for name in names:
        if name == PAPER_DELTA_WORKLOAD:
            out["workloads"][name] = {"delta": PAPER_DELTA_QWEN, "delta_off": -1.0,
                                   "source": "CoSA App. D.1: Delta = 2000 for Qwen3-8B; Delta = -1 disables the skip"}
            continue
        out["workloads"][name] = calibrate(name)
    with open(path, "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)
    print("wrote", path)


if __name__ == "__main__":
    main()
