"""GPU parity for multi-row steps (grouped tcgen05 path) and the prefill bypass.

Multi-row cached steps (2 <= M <= 16): every row's router ids equal the
oracle's, the union's slot/hit/miss/eviction record equals the oracle LRU bit
for bit (a union larger than S bypasses on the device), outputs are within the
stated tolerance of the oracle, and a cached run is bit-identical to an
all-resident run.  Bypass steps (M > 16): outputs within tolerance, the cache
untouched (no fills, slot map unchanged).
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


def _dev(cfg, rows):
    return (torch.empty((rows, cfg.experts), dtype=torch.float32, device="cuda"),
            torch.empty((rows, cfg.hidden), dtype=torch.bfloat16, device="cuda"),
            torch.empty((rows, cfg.hidden), dtype=torch.float32, device="cuda"))


def _put(lg_d, x_d, lg, xb):
    lg_d.copy_(torch.from_numpy(np.ascontiguousarray(lg)))
    x_d.copy_(torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16))


def _oracle_rows(orc, banks, cfg, lg, xb, rows):
    w, s, g = banks.layer_arrays(0)
    out = np.zeros((len(rows), cfg.hidden))
    for i, m in enumerate(rows):
        o, _, _, _ = orc.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k,
                                  lg[m:m + 1], xb[m:m + 1])
        out[i] = o[0]
    return out


@pytest.mark.parametrize("name,wide_x", [("tiny", False), ("tiny_wide", False),
                                         ("tiny_wide", True), ("small", False),
                                         ("small", True), ("small_wide_i", False),
                                         ("small_wide_h", False)])
def test_tiny_multirow_trace_outputs_and_device_bypass(lib, orc, name, wide_x):
    cfg = workload.CONFIGS[name]
    M, steps = 4, 40
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, trace_capacity=steps)
    rt = workload.Routing(cfg)
    act = workload.activations_wide if wide_x else workload.activations
    xs = act(cfg.seed, 0, steps, M, cfg.hidden)
    sim = orc.LRUSim(cfg.experts, cfg.slots)
    lg_d, x_d, out_d = _dev(cfg, M)
    ids_ref, worst = [], {}
    for t in range(steps):
        lg = rt.step(M)
        _put(lg_d, x_d, lg, xs[t])
        cache.step(0, lg_d, x_d, out_d)
        w, s, g = banks.layer_arrays(0)
        ref, ids, _, _ = orc.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k,
                                      lg, xs[t])
        m = assert_within_tolerance(out_d.cpu().numpy(), ref, f"step {t}", scale_free=wide_x)
        worst = {k: max(worst.get(k, 0.0), v) for k, v in m.items()}
        ids_ref.append(ids)
    print(name, "multirow worst", "(wide x)" if wide_x else "", worst)
    recs = cache.trace(0)
    n_bypass = 0
    for t, rec in enumerate(recs):
        assert np.array_equal(record_ids(rec, M, cfg.top_k), ids_ref[t])
        sr = sim.step(ids_ref[t].ravel())
        check_record_against_sim(rec, sr, M, cfg.top_k)
        n_bypass += sr["bypass"]
    st = cache.stats(0)
    assert st["misses"] == sim.stats["misses"] and st["hits"] == sim.stats["hits"]
    assert st["bypass_calls"] == sim.stats["bypass"]
    assert 0 < n_bypass < steps      # both the cached and the union > S path ran
    cache.close()
    banks.close()


def test_glm_multirow_wide_x(lib, orc):
    """GLM shape, one 16-row round of x with a wide dynamic range (elements up to
    6e4 and below 1e-5): sampled rows within the scale-free tolerance."""
    cfg = workload.CONFIGS["multirow"]
    M = cfg.rows
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, layers=1)
    lg = workload.Routing(cfg).step()
    xb = workload.activations_wide(cfg.seed, 0, 1, M, cfg.hidden)[0]
    lg_d, x_d, out_d = _dev(cfg, M)
    _put(lg_d, x_d, lg, xb)
    cache.step(0, lg_d, x_d, out_d)
    rows = [0, 7, 15]
    ref = _oracle_rows(orc, banks, cfg, lg, xb, rows)
    print("glm multirow wide x", assert_within_tolerance(out_d.cpu().numpy()[rows], ref,
                                                          scale_free=True))
    assert cache.stats(0)["error_flags"] == 0
    cache.close()
    banks.close()


def test_glm_multirow_rounds(lib, orc):
    """GLM shape, M = 16 rows per round (4 streams x 4 rows): trace on every step,
    outputs on sampled rows, and cached == all-resident bitwise."""
    cfg = workload.CONFIGS["multirow"]
    M, steps = cfg.rows, 24
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, layers=1, trace_capacity=steps)
    rt = workload.Routing(cfg)
    xs = workload.activations(cfg.seed, 0, steps, M, cfg.hidden)
    sim = orc.LRUSim(cfg.experts, cfg.slots, check_list=False)
    lg_d, x_d, out_d = _dev(cfg, M)
    lgs, outs = [], []
    for t in range(steps):
        lg = rt.step()
        lgs.append(lg)
        _put(lg_d, x_d, lg, xs[t])
        cache.step(0, lg_d, x_d, out_d)
        outs.append(out_d.cpu().numpy().copy())
        if t in (0, steps - 1):
            rows = [0, 5, 15]
            ref = _oracle_rows(orc, banks, cfg, lg, xs[t], rows)
            m = assert_within_tolerance(outs[-1][rows], ref, f"step {t}")
            print("glm multirow step", t, m)
    recs = cache.trace(0)
    unions = []
    for t, rec in enumerate(recs):
        ids = np.stack([orc.route(lgs[t][m], cfg.top_k)[0] for m in range(M)])
        assert np.array_equal(record_ids(rec, M, cfg.top_k), ids)
        check_record_against_sim(rec, sim.step(ids.ravel()), M, cfg.top_k)
        unions.append(rec.n_union)
    st = cache.stats(0)
    assert st["picks"] == steps * M * cfg.top_k
    # union fetch: far fewer experts than picks (shared draft ids, popular experts)
    assert np.mean(unions) < 0.6 * M * cfg.top_k
    cache.close()
    # same steps, every expert resident: identical bits
    full = make_cache(cfg, banks, layers=1, all_resident=True)
    for t in range(steps):
        _put(lg_d, x_d, lgs[t], xs[t])
        full.step(0, lg_d, x_d, out_d)
        got = out_d.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), outs[t].view(np.uint32)), f"step {t}"
    full.close()
    banks.close()


@pytest.mark.parametrize("name,rows", [("tiny", 17), ("tiny", 64), ("tiny_wide", 64)])
def test_tiny_prefill_bypass(lib, orc, name, rows):
    cfg = workload.CONFIGS[name]
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, max_rows=rows)
    # warm the ring with a few decode steps, then bypass
    lg1, x1, o1 = _dev(cfg, 1)
    rt = workload.Routing(cfg)
    xs = workload.activations(cfg.seed, 0, 6, 1, cfg.hidden)
    for t in range(6):
        _put(lg1, x1, rt.step(), xs[t])
        cache.step(0, lg1, x1, o1)
    before = cache.slot_map(0).copy()
    st0 = cache.stats(0)
    lg = workload.prefill_logits(cfg, 0, rows)
    xb = workload.activations(cfg.seed, 1, 1, rows, cfg.hidden)[0]
    lg_d, x_d, out_d = _dev(cfg, rows)
    _put(lg_d, x_d, lg, xb)
    cache.step(0, lg_d, x_d, out_d)
    w, s, g = banks.layer_arrays(0)
    ref, _, _, _ = orc.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, lg, xb)
    print("tiny bypass", rows, assert_within_tolerance(out_d.cpu().numpy(), ref))
    st1 = cache.stats(0)
    assert st1["bypass_calls"] == st0["bypass_calls"] + 1
    assert st1["misses"] == st0["misses"] and st1["bytes_copied"] == st0["bytes_copied"]
    assert np.array_equal(cache.slot_map(0), before)
    cache.close()
    banks.close()


def test_glm_prefill_bypass_sampled_rows(lib, orc):
    cfg = workload.CONFIGS["prefill"]
    rows = 64
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, layers=1, max_rows=rows)
    lg = workload.prefill_logits(cfg, 0, rows)
    xb = workload.activations(cfg.seed, 0, 1, rows, cfg.hidden)[0]
    lg_d, x_d, out_d = _dev(cfg, rows)
    _put(lg_d, x_d, lg, xb)
    cache.step(0, lg_d, x_d, out_d)
    got = out_d.cpu().numpy()
    sample = [0, 31, 63]
    ref = _oracle_rows(orc, banks, cfg, lg, xb, sample)
    print("glm bypass", assert_within_tolerance(got[sample], ref))
    st = cache.stats(0)
    assert st["bypass_calls"] == 1 and st["misses"] == 0
    cache.close()
    banks.close()


@pytest.mark.parametrize("name", ["tiny", "tiny_wide", "small", "small_wide_i", "small_wide_h"])
def test_tiny_prefill_staged_equals_zero_copy(lib, orc, name):
    """Staged prefill (experts copied into HBM a chunk at a time, two chunks held)
    gives the same bits as reading host memory directly, for chunk sizes that
    cover the union in one chunk, in several, and with a ragged last chunk.
    At the small shape the staged chunks run the TMA-tiled kernel and the
    zero-copy path the cp.async one."""
    cfg = workload.CONFIGS[name]
    rows = 64
    banks = Banks(cfg)
    lg = workload.prefill_logits(cfg, 0, rows)
    xb = workload.activations(cfg.seed, 3, 1, rows, cfg.hidden)[0]
    lg_d, x_d, out_d = _dev(cfg, rows)
    _put(lg_d, x_d, lg, xb)
    outs = {}
    for chunk in (-1, 0, 4, 3, 1):
        cache = make_cache(cfg, banks, prefill_chunk=chunk, max_rows=rows)
        for _ in range(2):   # twice: the staging halves are reused across steps
            cache.step(0, lg_d, x_d, out_d)
        outs[chunk] = out_d.cpu().numpy().copy()
        st = cache.stats(0)
        assert st["bypass_calls"] == 2 and st["misses"] == 0 and st["error_flags"] == 0
        cache.close()
    w, s, g = banks.layer_arrays(0)
    ref, _, _, _ = orc.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, lg, xb)
    assert_within_tolerance(outs[-1], ref)
    for chunk, o in outs.items():
        assert np.array_equal(o.view(np.uint32), outs[-1].view(np.uint32)), f"chunk {chunk}"
    banks.close()


def test_glm_prefill_staged_graph_and_zero_copy(lib, orc):
    """GLM prefill, 128 rows: the staged path (8 chunks of 32 experts) replayed
    from a CUDA graph equals its eager run and the zero-copy path bit for bit."""
    cfg = workload.CONFIGS["prefill"]
    rows = 128
    banks = Banks(cfg)
    lg = workload.prefill_logits(cfg, 1, rows)
    xb = workload.activations(cfg.seed, 4, 1, rows, cfg.hidden)[0]
    lg_d, x_d, out_d = _dev(cfg, rows)
    _put(lg_d, x_d, lg, xb)
    zc = make_cache(cfg, banks, layers=1, prefill_chunk=-1, max_rows=rows)
    zc.step(0, lg_d, x_d, out_d)
    ref_bits = out_d.cpu().numpy().copy()
    zc.close()
    cache = make_cache(cfg, banks, layers=1, max_rows=rows)
    cache.step(0, lg_d, x_d, out_d)
    eager = out_d.cpu().numpy().copy()
    assert np.array_equal(eager.view(np.uint32), ref_bits.view(np.uint32))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    out_d.zero_()
    with torch.cuda.graph(g, stream=s):
        cache.step(0, lg_d, x_d, out_d)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(out_d.cpu().numpy().view(np.uint32), ref_bits.view(np.uint32))
    sample = [0, 64, 127]
    assert_within_tolerance(eager[sample], _oracle_rows(orc, banks, cfg, lg, xb, sample))
    assert cache.stats(0)["error_flags"] == 0
    cache.close()
    banks.close()


@pytest.mark.parametrize("name", ["tiny", "tiny_wide", "small", "multirow"])
def test_batch_invariant_rows(lib, orc, name):
    """Batch-invariant mode: every row of a round (M = 16, cached) is bit-identical
    to the same row stepped alone through another cached handle.  Both handles'
    caches evolve differently, which caching must not show in any output bit."""
    cfg = workload.CONFIGS[name]
    M = 16
    steps = 3
    banks = Banks(cfg)
    rt = workload.Routing(cfg)
    lgs = [rt.step(M) for _ in range(steps)]
    xs = workload.activations(cfg.seed, 5, steps, M, cfg.hidden)
    rounds = make_cache(cfg, banks, layers=1, batch_invariant=True)
    single = make_cache(cfg, banks, layers=1, batch_invariant=True)
    lgM, xM, oM = _dev(cfg, M)
    lg1, x1, o1 = _dev(cfg, 1)
    rows = range(M) if name in ("tiny", "tiny_wide", "small") else (0, 5, 15)
    for t in range(steps):
        _put(lgM, xM, lgs[t], xs[t])
        rounds.step(0, lgM, xM, oM)
        got = oM.cpu().numpy()
        for m in rows:
            _put(lg1, x1, lgs[t][m:m + 1], xs[t][m:m + 1])
            single.step(0, lg1, x1, o1)
            alone = o1.cpu().numpy()[0]
            assert np.array_equal(alone.view(np.uint32), got[m].view(np.uint32)), (t, m)
    ref = _oracle_rows(orc, banks, cfg, lgs[-1], xs[-1], [0])
    assert_within_tolerance(got[[0]], ref)
    for c in (rounds, single):
        assert c.stats(0)["error_flags"] == 0
        c.close()
    banks.close()
