"""The no-allocation expert pass (moe_expert_pass_noalloc) against the regular step.

Some callers cannot allocate device memory (an engine that already owns all
free HBM, a decode loop that cannot take an allocation's synchronisation); for
them the library offers an expert pass whose scratch is a fixed file-scope
device array.  This test drives it through the C ABI on the experts and router
weights that a regular all-resident moe_cache_step chose, two calls in a row
with different inputs, and checks that each output equals that step's output
bit for bit (both run the same expert kernels over the same picks in rank
order) and that the call reports clean error flags.  It covers the GLM shape
and the scratch's largest shape (top-16, hidden = inter = 8192), where h and the
per-expert outputs fill their whole fixed extents.  It runs alone in a fresh
process or after the rest of the suite (this file sorts last so a failure here
comes after every other test has run).
"""
import numpy as np
import pytest
import torch

import workload
from harness import Banks, make_cache, record_ids

pytestmark = pytest.mark.gpu

CASES = {
    # GLM-shaped layer, top-8 of 16 experts
    "glm": workload.Config("noalloc", 1, 6144, 2048, 16, 8, 16, 1, 2, 1.1, 0.1, 7),
    # the scratch's limits: top-16, hidden = inter = 8192
    "max": workload.Config("noalloc_max", 1, 8192, 8192, 16, 16, 16, 1, 2, 1.1, 0.1, 8),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_pass_matches_cache_step_twice(name):
    import hbm_slot_cache_gb300 as hsc
    from hbm_slot_cache_gb300 import _lib
    hsc.build()
    assert torch.cuda.is_available()
    cfg = CASES[name]
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, all_resident=True, trace_capacity=4, max_rows=1)
    w, s, g = banks.layer_arrays(0)
    rt = workload.Routing(cfg)
    xs = workload.activations(cfg.seed, 0, 2, 1, cfg.hidden)
    lg_d = torch.empty((1, cfg.experts), dtype=torch.float32, device="cuda")
    x_d = torch.empty((1, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    out_step = torch.empty((1, cfg.hidden), dtype=torch.float32, device="cuda")
    out_na = torch.empty((1, cfg.hidden), dtype=torch.float32, device="cuda")
    flags = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for t in range(2):
        lg_d.copy_(torch.from_numpy(rt.step()))
        x_d.copy_(torch.from_numpy(xs[t].view(np.int16)).view(torch.bfloat16))
        cache.step(0, lg_d, x_d, out_step)
        rec = cache.trace(0)[-1]
        ids = record_ids(rec, 1, cfg.top_k)[0].tolist()
        wts = np.array(rec.weights[:cfg.top_k], np.float32)
        # the caller's own device copies of the chosen experts
        wd = [torch.from_numpy(w[e * cache.Bw:(e + 1) * cache.Bw].copy()).cuda() for e in ids]
        sd = [torch.from_numpy(s[e * cache.Bs:(e + 1) * cache.Bs].copy()).cuda() for e in ids]
        out_na.fill_(float("nan"))
        flags.fill_(0xFFFF)
        _lib.moe_expert_pass_noalloc(cfg.top_k, cfg.hidden, cfg.inter,
                                     [t_.data_ptr() for t_ in wd], [t_.data_ptr() for t_ in sd],
                                     g[ids], wts, x_d.data_ptr(), out_na.data_ptr(), stream,
                                     flags_out=flags.data_ptr())
        torch.cuda.synchronize()
        got, ref = out_na.cpu().numpy(), out_step.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"call {t}"
        assert int(flags.item()) == 0, f"call {t}: flags {int(flags.item()):#x}"
        del wd, sd
    assert cache.stats(0)["error_flags"] == 0
    # sizes beyond the fixed scratch are refused with a clear error
    with pytest.raises(_lib.MoeError) as e:
        _lib.moe_expert_pass_noalloc(cfg.top_k, 16384, cfg.inter, [1] * cfg.top_k,
                                     [1] * cfg.top_k, g[:cfg.top_k],
                                     np.ones(cfg.top_k, np.float32), x_d.data_ptr(),
                                     out_na.data_ptr(), stream)
    assert e.value.code == _lib.MOE_ERR_UNSUPPORTED
    cache.close()
    banks.close()
