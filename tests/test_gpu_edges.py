"""GPU parity for the one-row path's degenerate shapes, through the C ABI.

- slots == top_k: every step's picks hold every slot, so each miss must evict
  a slot no pick of this step uses (the LRU's untouched-this-step rule at its
  limit);
- top-1: one pick, router weight exactly 1;
- inter 4096 (I/32 = 128 blocks of h a row): the down pass keeps g * w * h in
  shared memory instead of registers, a branch no shipped config reaches;
- hidden = inter = MOE_MAX_DIM (8192): the largest gate/up rows (544-thread
  CTAs) and a one-stage down ring; outputs checked every third step (the
  oracle takes seconds a step at this size).

Each runs from an empty ring against the oracle (trace bit for bit, outputs
within max |d|/max|ref| <= 2e-2 and mean |d| <= 1e-3), and the wide case
also cached against all-resident, bit for bit.  The multi-row cached path at
its row-count ends: 2 rows, and 16 (the most a cached step takes) on a ring
large enough that no step bypasses.
"""
import dataclasses

import numpy as np
import pytest
import torch

import workload
from harness import (Banks, assert_within_tolerance, check_record_against_sim, make_cache,
                     record_ids)
from test_gpu_decode import _check_trace_and_outputs, _run_outputs

pytestmark = pytest.mark.gpu

TINY = workload.CONFIGS["tiny"]
EDGES = {
    # 16 experts, top-4, 4 slots
    "slots_eq_topk": dataclasses.replace(TINY, name="slots_eq_topk", top_k=4, slots=4,
                                         steps=48, seed=5),
    # 8 experts, top-1, 2 slots
    "top1": dataclasses.replace(TINY, name="top1", experts=8, top_k=1, slots=2, steps=48,
                                seed=6),
    # H256 / I4096, 6 experts, top-2, 3 slots
    "wide_inter": dataclasses.replace(TINY, name="wide_inter", inter=4096, experts=6, slots=3,
                                      steps=24, seed=7),
    # H8192 / I8192 (113 MB an expert), 3 experts, top-2, 2 slots
    "max_dims": dataclasses.replace(TINY, name="max_dims", hidden=8192, inter=8192, experts=3,
                                    slots=2, steps=6, seed=8),
}
OUT_EVERY = {"max_dims": 3}


@pytest.fixture(scope="module")
def lib():
    import hbm_slot_cache_gb300 as m
    m.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


@pytest.mark.parametrize("name", sorted(EDGES))
def test_edge_shape_trace_and_outputs(lib, orc, name):
    cfg = EDGES[name]
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, trace_capacity=cfg.steps)
    sim, worst = _check_trace_and_outputs(orc, cache, cfg, banks, 0, cfg.steps,
                                          out_every=OUT_EVERY.get(name, 1))
    print(name, "worst", worst, "misses", sim.stats["misses"])
    assert sim.stats["misses"] > cfg.slots  # the ring churned
    if cfg.top_k == 1:  # one pick: its weight is exactly 1
        assert all(rec.weights[0] == 1.0 for rec in cache.trace(0))
    if cfg.top_k == cfg.slots:  # every slot is used by some pick of every step
        for rec in cache.trace(0):
            assert sorted(rec.slot[:cfg.top_k]) == list(range(cfg.slots))
    cache.close()
    banks.close()


def test_wide_inter_cached_equals_all_resident_bitwise(lib):
    cfg = EDGES["wide_inter"]
    banks = Banks(cfg)
    a = make_cache(cfg, banks, layers=1)
    outs_a = _run_outputs(a, cfg, 0, cfg.steps)
    assert a.stats(0)["misses"] > 0
    a.close()
    b = make_cache(cfg, banks, layers=1, all_resident=True)
    outs_b = _run_outputs(b, cfg, 0, cfg.steps)
    assert b.stats(0)["misses"] == 0
    b.close()
    banks.close()
    for t, (x, y) in enumerate(zip(outs_a, outs_b)):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32)), f"step {t}"


@pytest.mark.parametrize("rows,slots", [(2, 4), (16, 16)])
def test_multirow_row_count_edges(lib, orc, rows, slots):
    cfg = dataclasses.replace(TINY, name=f"rows{rows}", slots=slots, rows=rows, steps=24,
                              seed=9)
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, trace_capacity=cfg.steps)
    rt = workload.Routing(cfg)
    xs = workload.activations(cfg.seed, 0, cfg.steps, rows, cfg.hidden)
    sim = orc.LRUSim(cfg.experts, cfg.slots)
    w, s, g = banks.layer_arrays(0)
    lg_d = torch.empty((rows, cfg.experts), dtype=torch.float32, device="cuda")
    x_d = torch.empty((rows, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    out_d = torch.empty((rows, cfg.hidden), dtype=torch.float32, device="cuda")
    ids_ref, worst = [], {}
    for t in range(cfg.steps):
        lg = rt.step(rows)
        lg_d.copy_(torch.from_numpy(np.ascontiguousarray(lg)))
        x_d.copy_(torch.from_numpy(np.ascontiguousarray(xs[t]).view(np.int16)).view(torch.bfloat16))
        cache.step(0, lg_d, x_d, out_d)
        ref, ids, _, _ = orc.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k,
                                      lg, xs[t])
        m = assert_within_tolerance(out_d.cpu().numpy(), ref, f"rows {rows} step {t}")
        worst = {k: max(worst.get(k, 0.0), v) for k, v in m.items()}
        ids_ref.append(ids)
    print(f"rows {rows} worst", worst)
    for t, rec in enumerate(cache.trace(0)):
        assert np.array_equal(record_ids(rec, rows, cfg.top_k), ids_ref[t]), f"ids step {t}"
        sr = sim.step(ids_ref[t].ravel())
        assert not sr["bypass"]  # the union always fits the ring: the cached path ran
        check_record_against_sim(rec, sr, rows, cfg.top_k)
    st = cache.stats(0)
    assert st["misses"] == sim.stats["misses"] > 0 and st["hits"] == sim.stats["hits"]
    assert st["bypass_calls"] == 0 and st["error_flags"] == 0
    cache.close()
    banks.close()
