"""GPU: the host-buffer entry point (moe_cache_step_host) against the device one.

A twin cache stepped through moe_cache_step on device buffers is the
reference: every step's output must be bit-identical and the layer counters
equal, over several layers (each one-row layer replays its own captured
graph from its second step), a mid-run multi-row round (eager path), the
tiny and GLM shapes, page-locked buffers (moved by kernels, also unaligned)
and pageable ones (copies).  The device path itself is checked against the oracle
in test_gpu_decode.py.
"""
import numpy as np
import pytest
import torch

import workload
from harness import Banks, make_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import hbm_slot_cache_gb300 as m
    m.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _host(a, pinned, offset=0):
    """A CPU tensor holding a's values: page-locked or pageable, its data
    starting `offset` elements into a larger buffer (so not 16-byte aligned)."""
    flat = a.reshape(-1)
    buf = torch.empty(flat.numel() + offset, dtype=a.dtype)
    if pinned:
        buf = buf.pin_memory()
    t = buf[offset:].view(a.shape)
    t.copy_(a)
    return t


@pytest.mark.parametrize("name,layers,steps,pinned,offset", [
    ("tiny", 3, 20, True, 0), ("glm", 2, 12, True, 0),
    ("tiny", 2, 10, False, 0),     # pageable: the copy path
    ("tiny", 2, 10, True, 1)])     # page-locked, not 16-byte aligned: the narrow kernel words
def test_step_host_equals_device_step(lib, name, layers, steps, pinned, offset):
    cfg = workload.CONFIGS[name]
    banks = Banks(cfg, distinct=1)
    E, H = cfg.experts, cfg.hidden
    dev = make_cache(cfg, banks, layers=layers, max_rows=4)
    host = make_cache(cfg, banks, layers=layers, max_rows=4)
    rts = [workload.Routing(cfg, l) for l in range(layers)]
    xs = [workload.activations(cfg.seed, l, steps, 4, H) for l in range(layers)]
    s = torch.cuda.Stream()
    for t in range(steps):
        rows = 3 if t == steps // 2 else 1     # one multi-row round in the middle
        for l in range(layers):
            lg = np.ascontiguousarray(rts[l].step(rows), np.float32)
            xb = np.ascontiguousarray(xs[l][t][:rows])
            lg_d = torch.from_numpy(lg).cuda()
            x_d = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
            out_d = torch.empty((rows, H), dtype=torch.float32, device="cuda")
            dev.step(l, lg_d, x_d, out_d)
            lg_h = _host(torch.from_numpy(lg), pinned, offset)
            x_h = _host(torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16), pinned, offset)
            out_h = _host(torch.zeros((rows, H), dtype=torch.float32), pinned, offset)
            with torch.cuda.stream(s):
                host.step_host(l, lg_h, x_h, out_h, s)
            s.synchronize()
            ref = out_d.cpu().numpy()
            got = out_h.numpy()
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (name, t, l, rows)
    for l in range(layers):
        a, b = dev.stats(l), host.stats(l)
        for key in ("steps", "picks", "hits", "misses", "evictions", "bytes_copied", "error_flags"):
            assert a[key] == b[key], (l, key)
    dev.close()
    host.close()
    banks.close()


def test_step_host_rejects_too_many_rows(lib):
    """max_rows below the cached-row limit is raised to it (every cached step
    fits the workspaces); more rows than that are refused."""
    cfg = workload.CONFIGS["tiny"]
    banks = Banks(cfg, distinct=1)
    cache = make_cache(cfg, banks, layers=1, max_rows=2)
    rows = lib._lib.MOE_MAX_CACHED_ROWS + 1
    lg = torch.zeros((rows, cfg.experts), dtype=torch.float32).pin_memory()
    x = torch.zeros((rows, cfg.hidden), dtype=torch.bfloat16).pin_memory()
    out = torch.zeros((rows, cfg.hidden), dtype=torch.float32).pin_memory()
    with pytest.raises(lib.MoeError):
        cache.step_host(0, lg, x, out)
    cache.close()
    banks.close()
