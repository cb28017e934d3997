"""Offline slot-policy report over recorded routing traces (the moe_policy_* C ABI).

    python -m hbm_slot_cache_gb300.policy TRACE.npy --experts 256 --budget 7360

TRACE.npy: int32 [layers, steps, picks] of routed expert ids (picks = rows *
top_k per layer-step).  Prints, per layer and in total, the host-link expert
reads and hit rate of the cache's LRU at a uniform ring size, of a hindsight
static pin and of hybrids, and the per-layer ring sizes that minimise the link
reads within the slot budget (pass them to the cache as slots_per_layer).
"""
from __future__ import annotations

import argparse
import json

import numpy as np

from ._lib import (moe_policy_hybrid, moe_policy_lru, moe_policy_lru_curve,
                   moe_policy_size_layers, moe_policy_static)


def report(traces: np.ndarray, experts: int, budget: int, min_slots: int = 1,
           hybrid_fracs=(0.5, 0.75)) -> dict:
    traces = np.asarray(traces, np.int32)
    L = traces.shape[0]
    uniform = max(min_slots, budget // L)
    rows = []
    for l in range(L):
        t = traces[l]
        r = {"lru": moe_policy_lru(t, experts, uniform),
             "static": moe_policy_static(t, experts, uniform)}
        for f in hybrid_fracs:
            r[f"hybrid{int(round(100 * f))}"] = moe_policy_hybrid(t, experts, uniform,
                                                                  int(round(f * uniform)))
        rows.append(r)
    curves = np.stack([moe_policy_lru_curve(traces[l], experts, experts) for l in range(L)])
    sizes = moe_policy_size_layers(curves, budget, min_slots)
    sized = [moe_policy_lru(traces[l], experts, int(sizes[l])) for l in range(L)]

    def total(key, recs):
        picks = sum(x["picks"] for x in recs)
        return {"host_experts": int(sum(x["host_experts"] for x in recs)),
                "hit_rate": (sum(x["hits"] for x in recs) / picks) if picks else None}

    out = {"layers": L, "uniform_slots": uniform, "budget": budget,
           "per_layer_slots": sizes.tolist(),
           "uniform": {k: total(k, [r[k] for r in rows]) for k in rows[0]},
           "sized_lru": total("lru", sized)}
    return out


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("trace", help="int32 .npy [layers, steps, picks]")
    ap.add_argument("--experts", type=int, required=True)
    ap.add_argument("--budget", type=int, required=True, help="total slots over all layers")
    ap.add_argument("--min-slots", type=int, default=1)
    a = ap.parse_args()
    print(json.dumps(report(np.load(a.trace), a.experts, a.budget, a.min_slots), indent=1))


if __name__ == "__main__":
    main()
