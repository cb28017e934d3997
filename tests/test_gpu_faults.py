"""Failure detection on the GPU without a fault: a bounded device wait that runs out.

Every device wait in the library gives up after a limit and sets a sticky
flag instead of trapping or hanging.  moe_cache_set_wait_timeout shortens the
limit of the one-row expert kernels' copy waits to 1 us, so on a GLM-shaped
step (hundreds of CTAs waiting for HBM and host-link copies) some wait runs
out: the step still returns, MOE_FLAG_WAIT_TIMEOUT is set, and after the limit
is restored and the cache reset, steps are clean again (trace equal to the
oracle LRU from an empty ring, outputs within tolerance, no flag).  No GPU
fault, trap or unbounded wait is involved: copies still in flight are drained
under the default limit before any kernel exits.
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


def _put(lg_d, x_d, lg, xb):
    lg_d.copy_(torch.from_numpy(np.ascontiguousarray(lg)))
    x_d.copy_(torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16))


def test_wait_timeout_flag_then_reset_recovers(lib, orc):
    from hbm_slot_cache_gb300 import _lib
    cfg = workload.CONFIGS["glm"]
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, layers=1, trace_capacity=32)
    lg_d = torch.empty((1, cfg.experts), dtype=torch.float32, device="cuda")
    x_d = torch.empty((1, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    out_d = torch.empty((1, cfg.hidden), dtype=torch.float32, device="cuda")
    rt = workload.Routing(cfg)
    xs = workload.activations(cfg.seed, 0, 40, 1, cfg.hidden)
    for t in range(8):                     # normal steps first: the ring fills
        _put(lg_d, x_d, rt.step(), xs[t])
        cache.step(0, lg_d, x_d, out_d)
    assert cache.stats(0)["error_flags"] == 0
    with pytest.raises(_lib.MoeError):
        cache.set_wait_timeout(-1)

    cache.set_wait_timeout(1)
    flagged = 0
    for t in range(8, 18):
        _put(lg_d, x_d, rt.step(), xs[t])
        cache.step(0, lg_d, x_d, out_d)      # returns: no trap, no hang
        flagged = cache.stats(0)["error_flags"]
        if flagged & _lib.MOE_FLAG_WAIT_TIMEOUT:
            break
    assert flagged & _lib.MOE_FLAG_WAIT_TIMEOUT, f"no wait ran out (flags {flagged:#x})"

    cache.set_wait_timeout(0)
    cache.reset()
    assert cache.stats(0)["error_flags"] == 0
    # clean steps from an empty ring: trace, outputs and flags
    rt = workload.Routing(cfg, 3)
    steps = 12
    xs = workload.activations(cfg.seed, 3, steps, 1, cfg.hidden)
    sim = orc.LRUSim(cfg.experts, cfg.slots)
    w, s, g = banks.layer_arrays(0)
    ids_ref = []
    for t in range(steps):
        lg = rt.step()
        ids_ref.append(orc.route(lg[0], cfg.top_k)[0])
        _put(lg_d, x_d, lg, xs[t])
        cache.step(0, lg_d, x_d, out_d)
        if t in (0, steps - 1):
            ref, ids, _, _ = orc.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter,
                                          cfg.top_k, lg, xs[t])
            assert_within_tolerance(out_d.cpu().numpy(), ref, f"step {t} after reset")
    recs = cache.trace(0)
    assert len(recs) == steps            # the reset cleared the trace too
    for t, rec in enumerate(recs):
        ids = record_ids(rec, 1, cfg.top_k)
        assert np.array_equal(ids[0], ids_ref[t])
        check_record_against_sim(rec, sim.step(ids_ref[t]), 1, cfg.top_k)
    st = cache.stats(0)
    assert st["error_flags"] == 0 and st["misses"] == sim.stats["misses"]
    cache.close()
    banks.close()
