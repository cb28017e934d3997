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
also cached against all-resident, bit for bit.
"""
import dataclasses

import numpy as np
import pytest
import torch

import workload
from harness import Banks, make_cache
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
