"""How well the demand signal Delta predicts the next change of demand.

The review of "GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning
Serving" (evolve.pub, "Key claims under review") reports that the dual-
timescale working-set signal Delta_t predicts future demand change (Spearman
rho and sign agreement, the paper's Fig 6).  This module measures the same two
statistics for the decode path on a synthetic request stream:

* at every boundary b of a request: Delta_b = sum over layers and kv heads of
  (W_S - W_L), as the decision saw it;
* the demand D_b = sum over layers and kv heads of W_S (the Top-p working set
  of the short summary, i.e. of recent queries);
* pairs (Delta_b, D_{b+1} - D_b) over consecutive boundaries of the same
  request (the next boundary comes P steps later);
* Spearman's rho of the pairs and the fraction of pairs with nonzero entries
  whose signs agree.

Reading (the pages define neither the demand measure nor the horizon): the
demand is the short summary's working set and the horizon is the next
boundary.  The traces come from the library's own outputs (the per-request
Delta and the per-(layer, head) working sets it writes at a boundary); the
statistics are plain NumPy on the host.

Usage: python -m demand_paged_kv_gqa_b300.signal_quality [--workload W]
       [--steps N] [--batch B] [--layers L]
"""
from __future__ import annotations

import argparse
import json
from typing import Dict, List, Sequence, Tuple

import numpy as np


def rank_average(x: Sequence[float]) -> np.ndarray:
    """Ranks 1..n with tied values sharing the mean of their ranks."""
    x = np.asarray(x, dtype=np.float64)
    order = np.argsort(x, kind="mergesort")
    ranks = np.empty(len(x), dtype=np.float64)
    xs = x[order]
    i = 0
    while i < len(x):
        j = i
        while j + 1 < len(x) and xs[j + 1] == xs[i]:
            j += 1
        ranks[order[i:j + 1]] = 0.5 * (i + j) + 1.0
        i = j + 1
    return ranks


def spearman(x: Sequence[float], y: Sequence[float]) -> float:
    """Spearman's rank correlation: Pearson correlation of the average ranks."""
    rx, ry = rank_average(x), rank_average(y)
    rx -= rx.mean()
    ry -= ry.mean()
    den = np.sqrt(np.sum(rx * rx) * np.sum(ry * ry))
    return float(np.sum(rx * ry) / den) if den > 0 else float("nan")


def pairs_from_traces(traces: Dict[int, List[Tuple[int, int]]]) -> Tuple[np.ndarray, np.ndarray]:
    """traces: request id -> [(Delta_b, D_b)] in boundary order.  Returns the
    arrays (Delta_b, D_{b+1} - D_b) over consecutive boundaries."""
    xs, ys = [], []
    for seq in traces.values():
        for (d0, dem0), (_, dem1) in zip(seq[:-1], seq[1:]):
            xs.append(d0)
            ys.append(dem1 - dem0)
    return np.asarray(xs, dtype=np.float64), np.asarray(ys, dtype=np.float64)


def statistics(traces: Dict[int, List[Tuple[int, int]]]) -> dict:
    x, y = pairs_from_traces(traces)
    nz = (x != 0) & (y != 0)
    agree = float(np.mean(np.sign(x[nz]) == np.sign(y[nz]))) if nz.any() else float("nan")
    return {"pairs": int(len(x)), "spearman_rho": spearman(x, y) if len(x) > 1 else float("nan"),
            "sign_agreement": agree, "sign_pairs": int(nz.sum()),
            "delta_positive": float(np.mean(x > 0)) if len(x) else float("nan"),
            "change_positive": float(np.mean(y > 0)) if len(y) else float("nan")}


def collect(engine, steps: int) -> Dict[int, List[Tuple[int, int]]]:
    """Run ``steps`` decode steps of an Engine and record, at every boundary,
    the request's Delta and its demand D = sum of W_S (read back after each
    step; this is an analysis run, not a timed one)."""
    import torch
    pool = engine.pool
    req = pool.region("req")
    wset = pool.region("wset")
    traces: Dict[int, List[Tuple[int, int]]] = {}
    seen = torch.zeros(engine.batch, dtype=torch.int32)
    engine.fill()
    for _ in range(steps):
        act = engine.active()
        rids = {s: engine.slots[s].rid for s in act}
        engine.prepare_inputs()
        engine.step()
        meta = req[: engine.batch].cpu()
        ws = wset[: engine.batch].sum(dim=(1, 2)).cpu()          # [R][2]
        nb = meta[:, 10]
        delta = (meta[:, 9].to(torch.int64) << 32) | (meta[:, 8].to(torch.int64) & 0xFFFFFFFF)
        for s in act:
            if int(nb[s]) > int(seen[s]):
                traces.setdefault(rids[s], []).append((int(delta[s]), int(ws[s, 0])))
        seen = nb.clone()
        for s in range(engine.batch):   # a refilled slot starts again from 0
            if engine.slots[s] is None or (s in rids and engine.slots[s].rid != rids[s]):
                seen[s] = 0
        engine.fill()
    return traces


def main(argv=None):
    from . import growpage as gpb
    from . import synth
    from .engine import Engine
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama8b_32layer")
    ap.add_argument("--steps", type=int, default=1536)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None)
    a = ap.parse_args(argv)
    w = synth.WORKLOADS[a.workload]
    if a.layers:
        w = w.replace(num_layers=a.layers)
    eng = Engine(w, mode=gpb.GP_MODE_GROWPAGE, batch=a.batch)
    st = statistics(collect(eng, a.steps))
    st.update({"workload": w.name, "steps": a.steps, "batch": eng.batch, "layers": w.num_layers})
    print(json.dumps(st))


if __name__ == "__main__":
    main()
