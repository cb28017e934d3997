"""hbm_slot_cache_gb300: decode-time routed-MoE layer with an HBM expert slot cache.

Python face of the C ABI in include/moe_slot_cache.h.  ``_lib`` mirrors the C
functions one to one; the two classes below only marshal torch tensors and
pinned host buffers into those calls.  PyTorch provides device memory and
streams; every step of the layer runs in the library's sm_103a kernels.
"""
from __future__ import annotations

import numpy as np

from . import _lib
from ._lib import (MoeError, moe_cache_create, moe_cache_destroy, moe_cache_reset,  # noqa: F401
                   moe_cache_slot_bytes, moe_cache_slot_map, moe_cache_stats, moe_cache_step,
                   moe_cache_trace, moe_expert_bytes, moe_host_alloc, moe_host_free,
                   moe_probe_host_link, moe_cache_set_timing_events, moe_policy_hybrid,
                   moe_policy_lru, moe_policy_lru_curve, moe_policy_size_layers,
                   moe_policy_static)

__all__ = ["HostBank", "MoeCache", "MoeError", "build"]


def build(**kw) -> str:
    from .builder import build as _b
    return _b(**kw)


class HostBank:
    """Exact-size pinned, mapped host buffer (moe_host_alloc) with a numpy view."""

    def __init__(self, nbytes: int):
        self.nbytes = int(nbytes)
        self.ptr = moe_host_alloc(self.nbytes)
        import ctypes
        buf = (ctypes.c_uint8 * self.nbytes).from_address(self.ptr)
        self.array = np.frombuffer(buf, dtype=np.uint8)

    def close(self) -> None:
        if self.ptr:
            self.array = None
            moe_host_free(self.ptr)
            self.ptr = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _dev_ptr(t, dtype, what):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise TypeError(f"{what}: expected a contiguous CUDA tensor of {dtype}")
    return t.data_ptr()


class MoeCache:
    """One slot cache over `layers` MoE layers (moe_cache_create ... moe_cache_destroy).

    host_layers: per layer (w_bank, s_bank, gscale) where the banks are HostBank
    (or pinned torch CPU uint8 tensors) and gscale a float32 array [E, 3]."""

    def __init__(self, layers, experts, slots, hidden, inter, top_k, host_layers, *,
                 all_resident=False, trace_capacity=0, bypass_rows=0, max_rows=0,
                 prefill_chunk=0, batch_invariant=False, slots_per_layer=None):
        self.layers, self.experts, self.hidden, self.inter, self.top_k = (
            layers, experts, hidden, inter, top_k)
        self.slots = experts if all_resident else slots
        self.Bw, self.Bs = moe_expert_bytes(hidden, inter)
        self._keep = []
        ptrs = []
        for (w, s, g) in host_layers:
            g = np.ascontiguousarray(g, np.float32)
            self._keep.append((w, s, g))
            ptrs.append((self._host_ptr(w), self._host_ptr(s), g.ctypes.data))
        self.h = moe_cache_create(layers, experts, slots, hidden, inter, top_k, ptrs,
                                  all_resident=all_resident, trace_capacity=trace_capacity,
                                  bypass_rows=bypass_rows, max_rows=max_rows,
                                  prefill_chunk=prefill_chunk, batch_invariant=batch_invariant,
                                  slots_per_layer=slots_per_layer)
        self.trace_capacity = trace_capacity

    @staticmethod
    def _host_ptr(b) -> int:
        if isinstance(b, HostBank):
            return b.ptr
        if isinstance(b, int):
            return b
        import torch
        if isinstance(b, torch.Tensor):
            return b.data_ptr()
        raise TypeError("host bank must be HostBank, int address or pinned torch tensor")

    def step(self, layer: int, logits, x, out, stream=None) -> None:
        """logits fp32 [rows, E], x bf16 [rows, H], out fp32 [rows, H] (CUDA tensors)."""
        import torch
        rows = logits.shape[0]
        if x.shape != (rows, self.hidden) or out.shape != (rows, self.hidden) or \
                logits.shape != (rows, self.experts):
            raise ValueError("shape mismatch")
        st = (stream or torch.cuda.current_stream()).cuda_stream
        moe_cache_step(self.h, layer, rows, _dev_ptr(logits, torch.float32, "logits"),
                       _dev_ptr(x, torch.bfloat16, "x"), _dev_ptr(out, torch.float32, "out"), st)

    def step_host(self, layer: int, logits, x, out, stream=None) -> None:
        """The same step with host buffers (moe_cache_step_host): logits fp32 [rows, E],
        x bf16 [rows, H], out fp32 [rows, H], CPU tensors (pinned for asynchronous
        copies).  Enqueued on `stream`; the buffers must live until the stream
        passes the step."""
        import torch
        rows = logits.shape[0]
        if x.shape != (rows, self.hidden) or out.shape != (rows, self.hidden) or \
                logits.shape != (rows, self.experts):
            raise ValueError("shape mismatch")
        for t, dt, nm in ((logits, torch.float32, "logits"), (x, torch.bfloat16, "x"),
                          (out, torch.float32, "out")):
            if t.device.type != "cpu" or t.dtype != dt or not t.is_contiguous():
                raise ValueError(f"{nm}: expected a contiguous CPU {dt} tensor")
        st = (stream or torch.cuda.current_stream()).cuda_stream
        _lib.moe_cache_step_host(self.h, layer, rows, logits.data_ptr(), x.data_ptr(),
                                 out.data_ptr(), st)

    def stats(self, layer: int = -1) -> dict:
        return moe_cache_stats(self.h, layer)

    def slot_map(self, layer: int) -> np.ndarray:
        """Expert in each slot of `layer`'s ring (-1: empty)."""
        return moe_cache_slot_map(self.h, layer)

    def layer_slots(self, layer: int) -> int:
        return _lib.moe_cache_layer_slots(self.h, layer)

    def slot_bytes(self, layer: int, slot: int):
        return moe_cache_slot_bytes(self.h, layer, slot, self.Bw, self.Bs)

    def trace(self, layer: int, max_recs: int | None = None):
        return moe_cache_trace(self.h, layer, max_recs or self.trace_capacity)

    def reset(self) -> None:
        moe_cache_reset(self.h)

    def set_wait_timeout(self, microseconds: int) -> None:
        """Failure-detection hook: bound the one-row expert kernels' copy waits
        (0: the default limit).  See moe_cache_set_wait_timeout."""
        _lib.moe_cache_set_wait_timeout(self.h, microseconds)

    def close(self) -> None:
        if getattr(self, "h", None):
            moe_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
