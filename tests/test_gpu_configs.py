"""GPU parity on the remaining workload shapes.

- Flash-shaped stack: 16 MoE layers (hidden 4096, inter 2048, 288 experts,
  top-8, 54 slots), 512 decode steps per layer with independent routing per
  layer; every layer's trace bit-exact, outputs sampled.  The 16 layers alias
  one host bank (the routing and the caches stay independent per layer).
- Slot sweep: GLM shape at S = 32, 64, 128, 192, 300 steps each; trace
  bit-exact, hit rate rising with S, outputs sampled.
- A full 512-row prefill chunk bypassing the cache, sampled rows.
- Host-side error handling: unpinned backing, too many rows, bad arguments.
"""
import numpy as np
import pytest
import torch

import workload
from harness import (Banks, assert_within_tolerance, check_record_against_sim, make_cache,
                     record_ids)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import hbm_slot_cache_gb300 as m
    m.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _dev(cfg, rows=1):
    return (torch.empty((rows, cfg.experts), dtype=torch.float32, device="cuda"),
            torch.empty((rows, cfg.hidden), dtype=torch.bfloat16, device="cuda"),
            torch.empty((rows, cfg.hidden), dtype=torch.float32, device="cuda"))


def _put(lg_d, x_d, lg, xb):
    lg_d.copy_(torch.from_numpy(np.ascontiguousarray(lg)))
    x_d.copy_(torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16))


def test_flash_stack_16_layers(lib, orc):
    cfg = workload.CONFIGS["flash"]
    steps = cfg.steps
    banks = Banks(cfg, distinct=1)
    cache = make_cache(cfg, banks, trace_capacity=steps)
    rts = [workload.Routing(cfg, l) for l in range(cfg.layers)]
    lg_d, x_d, out_d = _dev(cfg)
    ids_ref = [[] for _ in range(cfg.layers)]
    w, s, g = banks.layer_arrays(0)
    xs = workload.activations(cfg.seed, 0, 4, 1, cfg.hidden)
    for t in range(steps):
        for l in range(cfg.layers):  # a decode round walks the layers in order
            lg = rts[l].step()
            xb = xs[(t + l) % 4]
            _put(lg_d, x_d, lg, xb)
            cache.step(l, lg_d, x_d, out_d)
            ids_ref[l].append(orc.route(lg[0], cfg.top_k)[0])
            if (t, l) in ((steps - 1, 0), (steps // 2, cfg.layers - 1)):
                ref, _, _, _ = orc.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter,
                                            cfg.top_k, lg, xb)
                print("flash", t, l, assert_within_tolerance(out_d.cpu().numpy(), ref))
    hits = []
    for l in range(cfg.layers):
        sim = orc.LRUSim(cfg.experts, cfg.slots, check_list=False)
        recs = cache.trace(l)
        assert len(recs) == steps
        for t, rec in enumerate(recs):
            assert np.array_equal(record_ids(rec, 1, cfg.top_k)[0], ids_ref[l][t])
            check_record_against_sim(rec, sim.step(ids_ref[l][t]), 1, cfg.top_k)
        st = cache.stats(l)
        assert st["misses"] == sim.stats["misses"] and st["error_flags"] == 0
        hits.append(sim.stats["hits"] / sim.stats["picks"])
    print("flash per-layer hit rates", np.round(hits, 3))
    assert 0.45 < float(np.mean(hits)) < 0.8
    cache.close()
    banks.close()


def test_glm_slot_sweep(lib, orc):
    cfg = workload.CONFIGS["prefill"]
    steps = cfg.steps
    banks = Banks(cfg)
    w, s, g = banks.layer_arrays(0)
    rates = []
    for S in workload.SWEEP_SLOTS:
        cache = make_cache(cfg, banks, layers=1, slots=S, trace_capacity=steps)
        rt = workload.Routing(cfg)
        xs = workload.activations(cfg.seed, 0, steps, 1, cfg.hidden)
        lg_d, x_d, out_d = _dev(cfg)
        ids_ref = []
        for t in range(steps):
            lg = rt.step(1)
            _put(lg_d, x_d, lg, xs[t])
            cache.step(0, lg_d, x_d, out_d)
            ids_ref.append(orc.route(lg[0], cfg.top_k)[0])
            if t == steps - 1:
                ref, _, _, _ = orc.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter,
                                            cfg.top_k, lg, xs[t])
                assert_within_tolerance(out_d.cpu().numpy(), ref, f"S={S}")
        sim = orc.LRUSim(cfg.experts, S, check_list=False)
        for t, rec in enumerate(cache.trace(0)):
            check_record_against_sim(rec, sim.step(ids_ref[t]), 1, cfg.top_k)
        st = cache.stats(0)
        assert st["misses"] == sim.stats["misses"]
        rates.append(st["hits"] / st["picks"])
        cache.close()
    print("slot sweep hit rates", dict(zip(workload.SWEEP_SLOTS, np.round(rates, 3))))
    assert all(a < b for a, b in zip(rates, rates[1:]))
    banks.close()


def test_glm_prefill_512_rows(lib, orc):
    cfg = workload.CONFIGS["prefill"]
    rows = cfg.rows
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, layers=1, max_rows=rows)
    lg = workload.prefill_logits(cfg, 0, rows)
    xb = workload.activations(cfg.seed, 2, 1, rows, cfg.hidden)[0]
    lg_d, x_d, out_d = _dev(cfg, rows)
    _put(lg_d, x_d, lg, xb)
    cache.step(0, lg_d, x_d, out_d)
    got = out_d.cpu().numpy()
    assert np.isfinite(got).all()
    w, s, g = banks.layer_arrays(0)
    for m in (0, 257, 511):
        ref, _, _, _ = orc.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k,
                                    lg[m:m + 1], xb[m:m + 1])
        assert_within_tolerance(got[m:m + 1], ref, f"row {m}")
    st = cache.stats(0)
    assert st["bypass_calls"] == 1 and st["misses"] == 0
    cache.close()
    banks.close()


def test_host_side_errors(lib):
    import ctypes
    from hbm_slot_cache_gb300 import _lib as L
    cfg = workload.CONFIGS["tiny"]
    Bw, Bs = workload.storage_bytes(cfg.hidden, cfg.inter)
    # unpinned (pageable) backing is refused
    w = np.zeros(cfg.experts * Bw + 64, np.uint8)
    s = np.zeros(cfg.experts * Bs + 64, np.uint8)
    g = workload.global_scales(cfg.experts)
    wp = (w.ctypes.data + 15) // 16 * 16
    sp = (s.ctypes.data + 15) // 16 * 16
    with pytest.raises(L.MoeError) as e:
        L.moe_cache_create(1, cfg.experts, cfg.slots, cfg.hidden, cfg.inter, cfg.top_k,
                           [(wp, sp, g.ctypes.data)])
    assert e.value.code == L.MOE_ERR_NOT_PINNED
    banks = Banks(cfg)
    # S < top_k and S > E are argument errors
    for S in (1, cfg.experts + 1):
        with pytest.raises(L.MoeError) as e:
            make_cache(cfg, banks, slots=S)
        assert e.value.code == L.MOE_ERR_ARG
    dflt = make_cache(cfg, banks)   # default: a decode-only handle (no bypass rows)
    lg_d, x_d, out_d = _dev(cfg, 33)
    with pytest.raises(L.MoeError) as e:
        L.moe_cache_step(dflt.h, 0, 17, lg_d.data_ptr(), x_d.data_ptr(), out_d.data_ptr(), 0)
    assert e.value.code == L.MOE_ERR_UNSUPPORTED
    dflt.close()
    cache = make_cache(cfg, banks, max_rows=32)
    with pytest.raises(L.MoeError) as e:   # more rows than the handle was sized for
        L.moe_cache_step(cache.h, 0, 33, lg_d.data_ptr(), x_d.data_ptr(), out_d.data_ptr(), 0)
    assert e.value.code == L.MOE_ERR_UNSUPPORTED
    with pytest.raises(L.MoeError) as e:   # layer out of range
        L.moe_cache_step(cache.h, 1, 1, lg_d.data_ptr(), x_d.data_ptr(), out_d.data_ptr(), 0)
    assert e.value.code == L.MOE_ERR_ARG
    with pytest.raises(L.MoeError) as e:   # misaligned activations
        L.moe_cache_step(cache.h, 0, 1, lg_d.data_ptr(), x_d.data_ptr() + 2, out_d.data_ptr(), 0)
    assert e.value.code == L.MOE_ERR_ARG
    with pytest.raises(L.MoeError) as e:   # misaligned output
        L.moe_cache_step(cache.h, 0, 1, lg_d.data_ptr(), x_d.data_ptr(), out_d.data_ptr() + 4, 0)
    assert e.value.code == L.MOE_ERR_ARG
    assert cache.stats(0)["steps"] == 0
    cache.close()
    banks.close()
    del ctypes
