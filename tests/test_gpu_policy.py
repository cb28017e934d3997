"""Per-layer ring sizes end to end: the offline policy tool sizes each layer's
ring from that layer's routing trace for a slot budget; a cache built with
those sizes then replays the traces, and every layer's device counters equal
the policy simulator's prediction, and its slot trace the oracle LRU's, bit
for bit."""
import numpy as np
import pytest
import torch

import workload
from harness import Banks, assert_within_tolerance, check_record_against_sim, make_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import hbm_slot_cache_gb300 as m
    m.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def test_per_layer_rings_sized_by_policy(lib, orc):
    cfg = workload.CONFIGS["tiny"]
    L, steps, budget = 3, 48, 12
    banks = Banks(cfg)
    # layers with different popularity skews, so their curves differ
    traces, logits = [], []
    for l in range(L):
        rt = workload.Routing(cfg, layer=l)
        rt.bias = rt.bias * (0.5 + l)
        lg = [rt.step(1) for _ in range(steps)]
        logits.append(lg)
        traces.append(np.stack([orc.route(x[0], cfg.top_k)[0] for x in lg]).astype(np.int32))
    curves = np.stack([lib.moe_policy_lru_curve(t, cfg.experts, cfg.experts) for t in traces])
    sizes = lib.moe_policy_size_layers(curves, budget, min_slots=cfg.top_k)
    assert sizes.sum() <= budget and (sizes >= cfg.top_k).all()
    cache = make_cache(cfg, banks, layers=L, trace_capacity=steps, slots_per_layer=sizes)
    assert [cache.layer_slots(l) for l in range(L)] == sizes.tolist()
    xs = workload.activations(cfg.seed, 9, steps, 1, cfg.hidden)
    lg_d = torch.empty((1, cfg.experts), dtype=torch.float32, device="cuda")
    x_d = torch.empty((1, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    out_d = torch.empty((1, cfg.hidden), dtype=torch.float32, device="cuda")
    for t in range(steps):
        for l in range(L):
            lg_d.copy_(torch.from_numpy(logits[l][t]))
            x_d.copy_(torch.from_numpy(xs[t].view(np.int16)).view(torch.bfloat16))
            cache.step(l, lg_d, x_d, out_d)
            if t == steps - 1 and l == L - 1:
                w, s, g = banks.layer_arrays(l)
                ref, _, _, _ = orc.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter,
                                            cfg.top_k, logits[l][t], xs[t])
                assert_within_tolerance(out_d.cpu().numpy(), ref)
    for l in range(L):
        pred = lib.moe_policy_lru(traces[l], cfg.experts, int(sizes[l]))
        st = cache.stats(l)
        assert (st["hits"], st["misses"], st["evictions"], st["bypass_calls"]) == \
            (pred["hits"], pred["misses"], pred["evictions"], pred["bypass_steps"]), l
        sim = orc.LRUSim(cfg.experts, int(sizes[l]))
        for t, rec in enumerate(cache.trace(l)):
            check_record_against_sim(rec, sim.step(traces[l][t]), 1, cfg.top_k)
        assert len(cache.slot_map(l)) == sizes[l]
        assert st["error_flags"] == 0
    cache.close()
    banks.close()
