"""ctypes binding of libmoe_slot_cache.so: the C ABI of include/moe_slot_cache.h.

Argument marshalling only.  Every step of the layer runs in the library's CUDA
kernels; there is no Python or CPU path.  Loading fails loudly when the shared
library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_SO = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_slot_cache.so")

MOE_OK = 0
MOE_ERR_ARG = -1
MOE_ERR_NOT_PINNED = -2
MOE_ERR_OOM = -3
MOE_ERR_CUDA = -4
MOE_ERR_UNSUPPORTED = -5
MOE_FLAG_NONFINITE_LOGIT = 0x1
MOE_FLAG_WAIT_TIMEOUT = 0x2
MOE_FLAG_BAD_PLAN = 0x4
MOE_MAX_EXPERTS = 1024
MOE_MAX_TOPK = 16
MOE_MAX_CACHED_ROWS = 16
MOE_MAX_PICKS = MOE_MAX_CACHED_ROWS * MOE_MAX_TOPK
MOE_MAX_DIM = 8192
MOE_COPY_SM = 0

EXPORTS = ("moe_cache_create", "moe_cache_step", "moe_cache_step_host", "moe_cache_stats",
           "moe_cache_slot_map",
           "moe_cache_slot_bytes", "moe_cache_trace", "moe_cache_reset", "moe_cache_destroy",
           "moe_cache_strerror", "moe_expert_bytes", "moe_host_alloc", "moe_host_free",
           "moe_probe_host_link", "moe_cache_set_timing_events", "moe_expert_pass_noalloc",
           "moe_policy_lru", "moe_policy_static", "moe_policy_hybrid", "moe_policy_lru_curve",
           "moe_policy_size_layers", "moe_cache_layer_slots", "moe_feed_inputs",
           "moe_cache_set_wait_timeout")


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


class HostLayer(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("s", ctypes.c_void_p), ("gscale", ctypes.c_void_p)]


class Opts(ctypes.Structure):
    _fields_ = [("copy_backend", ctypes.c_int), ("bypass_rows", ctypes.c_int),
                ("all_resident", ctypes.c_int), ("trace_capacity", ctypes.c_int),
                ("max_rows", ctypes.c_int), ("prefill_chunk", ctypes.c_int),
                ("batch_invariant", ctypes.c_int), ("slots_per_layer", ctypes.c_void_p)]


class PolicyResult(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("steps", "picks", "hits", "misses", "evictions",
                                               "bypass_steps", "host_experts")]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


class Stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_uint64), ("picks", ctypes.c_uint64), ("hits", ctypes.c_uint64),
                ("misses", ctypes.c_uint64), ("evictions", ctypes.c_uint64),
                ("bytes_copied", ctypes.c_uint64), ("bypass_calls", ctypes.c_uint64),
                ("error_flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_ if f != "reserved"}


_P = MOE_MAX_PICKS


class StepRecord(ctypes.Structure):
    _fields_ = [("clock", ctypes.c_uint32), ("rows", ctypes.c_int32), ("n_union", ctypes.c_int32),
                ("n_miss", ctypes.c_int32), ("bypass", ctypes.c_int32),
                ("ids", ctypes.c_int32 * _P), ("weights", ctypes.c_float * _P),
                ("slot", ctypes.c_int32 * _P), ("hit", ctypes.c_int32 * _P),
                ("miss_expert", ctypes.c_int32 * _P), ("miss_slot", ctypes.c_int32 * _P),
                ("miss_evicted", ctypes.c_int32 * _P)]


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            raise RuntimeError(f"{_SO} is missing: build it with hbm_slot_cache_gb300.build() "
                               "(needs nvcc); there is no fallback implementation")
        L = ctypes.CDLL(_SO)
        P, I, U64P = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)
        L.moe_cache_create.argtypes = [ctypes.POINTER(P), I, I, I, I, I, I, P, P]
        L.moe_cache_step.argtypes = [P, I, I, P, P, P, P]
        L.moe_cache_step_host.argtypes = [P, I, I, P, P, P, P]
        L.moe_cache_stats.argtypes = [P, I, ctypes.POINTER(Stats)]
        L.moe_cache_slot_map.argtypes = [P, I, P]
        L.moe_cache_layer_slots.argtypes = [P, I, ctypes.POINTER(I)]
        L.moe_cache_slot_bytes.argtypes = [P, I, I, P, P]
        L.moe_cache_trace.argtypes = [P, I, P, I, ctypes.POINTER(ctypes.c_int)]
        L.moe_cache_reset.argtypes = [P]
        L.moe_cache_destroy.argtypes = [P]
        L.moe_cache_set_wait_timeout.argtypes = [P, I]
        L.moe_cache_strerror.argtypes = [I]
        L.moe_cache_strerror.restype = ctypes.c_char_p
        L.moe_expert_bytes.argtypes = [I, I, U64P, U64P]
        L.moe_host_alloc.argtypes = [ctypes.POINTER(P), ctypes.c_size_t]
        L.moe_host_free.argtypes = [P]
        L.moe_probe_host_link.argtypes = [P, P, ctypes.c_size_t, I, I,
                                          ctypes.POINTER(ctypes.c_double)]
        L.moe_cache_set_timing_events.argtypes = [P, P]
        L.moe_expert_pass_noalloc.argtypes = [I, I, I, P, P, P, P, P, P, P, P]
        L.moe_feed_inputs.argtypes = [P, P, ctypes.c_size_t, ctypes.c_size_t, I, P, P, P, P]
        PR = ctypes.POINTER(PolicyResult)
        L.moe_policy_lru.argtypes = [P, I, I, I, I, PR]
        L.moe_policy_static.argtypes = [P, I, I, I, I, PR]
        L.moe_policy_hybrid.argtypes = [P, I, I, I, I, I, PR]
        L.moe_policy_lru_curve.argtypes = [P, I, I, I, I, P]
        L.moe_policy_size_layers.argtypes = [P, I, I, I, I, P]
        for name in EXPORTS:
            if name != "moe_cache_strerror":
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().moe_cache_strerror(code).decode()


def _check(rc: int, what: str) -> None:
    if rc != MOE_OK:
        raise MoeError(rc, what)


# ------------------------------------------------------------------- C ABI

def moe_expert_bytes(hidden: int, inter: int) -> tuple[int, int]:
    bw, bs = ctypes.c_uint64(), ctypes.c_uint64()
    _check(lib().moe_expert_bytes(hidden, inter, ctypes.byref(bw), ctypes.byref(bs)),
           "moe_expert_bytes")
    return bw.value, bs.value


def moe_cache_create(layers: int, experts: int, slots: int, hidden: int, inter: int, top_k: int,
                     host_layers, copy_backend: int = MOE_COPY_SM, bypass_rows: int = 0,
                     all_resident: bool = False, trace_capacity: int = 0,
                     max_rows: int = 0, prefill_chunk: int = 0,
                     batch_invariant: bool = False, slots_per_layer=None) -> int:
    """host_layers: sequence of (w_ptr, s_ptr, gscale_ptr) per layer. Returns the handle."""
    arr = (HostLayer * layers)(*[HostLayer(int(w), int(s), int(g)) for (w, s, g) in host_layers])
    spl = None
    if slots_per_layer is not None:
        spl = np.ascontiguousarray(slots_per_layer, np.int32)
        if spl.shape != (layers,):
            raise ValueError("slots_per_layer must have one entry per layer")
    o = Opts(copy_backend, bypass_rows, int(all_resident), trace_capacity, max_rows, prefill_chunk,
             int(batch_invariant), spl.ctypes.data if spl is not None else None)
    h = ctypes.c_void_p()
    _check(lib().moe_cache_create(ctypes.byref(h), layers, experts, slots, hidden, inter, top_k,
                                  ctypes.cast(arr, ctypes.c_void_p), ctypes.byref(o)),
           "moe_cache_create")
    return h.value


def moe_cache_step(h: int, layer: int, rows: int, router_logits: int, x: int, out: int,
                   stream: int = 0) -> None:
    _check(lib().moe_cache_step(h, layer, rows, router_logits, x, out, stream), "moe_cache_step")


def moe_cache_step_host(h: int, layer: int, rows: int, router_logits: int, x: int, out: int,
                        stream: int = 0) -> None:
    _check(lib().moe_cache_step_host(h, layer, rows, router_logits, x, out, stream),
           "moe_cache_step_host")


def moe_cache_stats(h: int, layer: int = -1) -> dict:
    st = Stats()
    _check(lib().moe_cache_stats(h, layer, ctypes.byref(st)), "moe_cache_stats")
    return st.as_dict()


def moe_cache_layer_slots(h: int, layer: int) -> int:
    n = ctypes.c_int()
    _check(lib().moe_cache_layer_slots(h, layer, ctypes.byref(n)), "moe_cache_layer_slots")
    return n.value


def moe_cache_slot_map(h: int, layer: int, slots: int | None = None) -> np.ndarray:
    if slots is None:
        slots = moe_cache_layer_slots(h, layer)
    out = np.empty(slots, np.int32)
    _check(lib().moe_cache_slot_map(h, layer, out.ctypes.data), "moe_cache_slot_map")
    return out


def moe_cache_slot_bytes(h: int, layer: int, slot: int, bw: int, bs: int):
    w = np.empty(bw, np.uint8)
    s = np.empty(bs, np.uint8)
    _check(lib().moe_cache_slot_bytes(h, layer, slot, w.ctypes.data, s.ctypes.data),
           "moe_cache_slot_bytes")
    return w, s


def moe_cache_trace(h: int, layer: int, max_recs: int) -> list[StepRecord]:
    recs = (StepRecord * max_recs)()
    n = ctypes.c_int()
    _check(lib().moe_cache_trace(h, layer, ctypes.cast(recs, ctypes.c_void_p), max_recs,
                                 ctypes.byref(n)), "moe_cache_trace")
    return list(recs[:n.value])


def moe_cache_reset(h: int) -> None:
    _check(lib().moe_cache_reset(h), "moe_cache_reset")


def moe_cache_set_wait_timeout(h: int, microseconds: int) -> None:
    _check(lib().moe_cache_set_wait_timeout(h, microseconds), "moe_cache_set_wait_timeout")


def moe_cache_destroy(h: int) -> None:
    _check(lib().moe_cache_destroy(h), "moe_cache_destroy")


MOE_TIMING_EVENTS = 8


def moe_cache_set_timing_events(h: int, events) -> None:
    """events: MOE_TIMING_EVENTS cudaEvent_t handles (ints), or None to stop recording."""
    if events is None:
        _check(lib().moe_cache_set_timing_events(h, None), "moe_cache_set_timing_events")
        return
    if len(events) != MOE_TIMING_EVENTS:
        raise ValueError(f"need {MOE_TIMING_EVENTS} events")
    arr = (ctypes.c_void_p * MOE_TIMING_EVENTS)(*[int(e) for e in events])
    _check(lib().moe_cache_set_timing_events(h, ctypes.cast(arr, ctypes.c_void_p)),
           "moe_cache_set_timing_events")


def moe_expert_pass_noalloc(k: int, hidden: int, inter: int, expert_w, expert_s, gscale,
                            weights, x: int, out: int, stream: int = 0,
                            flags_out: int = 0) -> None:
    """One-row expert pass without any device allocation (see the header).

    expert_w / expert_s: k device addresses; gscale float32 [k, 3]; weights float32 [k];
    flags_out: device address of a uint32 that receives the call's error flags (0: none)."""
    wa = (ctypes.c_void_p * k)(*[int(p) for p in expert_w])
    sa = (ctypes.c_void_p * k)(*[int(p) for p in expert_s])
    g = np.ascontiguousarray(gscale, np.float32).reshape(k, 3)
    w = np.ascontiguousarray(weights, np.float32).reshape(k)
    _check(lib().moe_expert_pass_noalloc(k, hidden, inter, ctypes.cast(wa, ctypes.c_void_p),
                                         ctypes.cast(sa, ctypes.c_void_p), g.ctypes.data,
                                         w.ctypes.data, x, out, flags_out or None, stream),
           "moe_expert_pass_noalloc")


def moe_feed_inputs(logits_trace: int, x_trace: int, logits_bytes: int, x_bytes: int,
                    steps: int, logits_dst: int, x_dst: int, cursor: int,
                    stream: int = 0) -> None:
    """Copy entry cursor[0] mod steps of the device traces into the fixed buffers and
    advance the device cursor (see the header)."""
    _check(lib().moe_feed_inputs(logits_trace, x_trace, logits_bytes, x_bytes, steps, logits_dst,
                                 x_dst, cursor, stream), "moe_feed_inputs")


def moe_host_alloc(nbytes: int) -> int:
    p = ctypes.c_void_p()
    _check(lib().moe_host_alloc(ctypes.byref(p), nbytes), "moe_host_alloc")
    return p.value


def moe_host_free(p: int) -> None:
    _check(lib().moe_host_free(p), "moe_host_free")


def moe_probe_host_link(host_src: int, dev_dst: int, nbytes: int, method: int = 0,
                        iters: int = 5) -> float:
    g = ctypes.c_double()
    _check(lib().moe_probe_host_link(host_src, dev_dst, nbytes, method, iters, ctypes.byref(g)),
           "moe_probe_host_link")
    return g.value


# ------------------------------------------------------------ offline slot policy

def _trace(trace) -> tuple[np.ndarray, int, int]:
    t = np.ascontiguousarray(trace, np.int32)
    if t.ndim != 2:
        raise ValueError("trace must be [steps, picks]")
    return t, t.shape[0], t.shape[1]


def moe_policy_lru(trace, experts: int, slots: int) -> dict:
    """LRU ring of `slots` slots over one layer's trace [steps, picks] (see the header)."""
    t, n, p = _trace(trace)
    r = PolicyResult()
    _check(lib().moe_policy_lru(t.ctypes.data, n, p, experts, slots, ctypes.byref(r)),
           "moe_policy_lru")
    return r.as_dict()


def moe_policy_static(trace, experts: int, slots: int) -> dict:
    t, n, p = _trace(trace)
    r = PolicyResult()
    _check(lib().moe_policy_static(t.ctypes.data, n, p, experts, slots, ctypes.byref(r)),
           "moe_policy_static")
    return r.as_dict()


def moe_policy_hybrid(trace, experts: int, slots: int, pinned: int) -> dict:
    t, n, p = _trace(trace)
    r = PolicyResult()
    _check(lib().moe_policy_hybrid(t.ctypes.data, n, p, experts, slots, pinned, ctypes.byref(r)),
           "moe_policy_hybrid")
    return r.as_dict()


def moe_policy_lru_curve(trace, experts: int, max_slots: int) -> np.ndarray:
    """host_experts of an S-slot LRU ring for S = 1 .. max_slots (uint64 [max_slots])."""
    t, n, p = _trace(trace)
    out = np.zeros(max_slots, np.uint64)
    _check(lib().moe_policy_lru_curve(t.ctypes.data, n, p, experts, max_slots, out.ctypes.data),
           "moe_policy_lru_curve")
    return out


def moe_policy_size_layers(curves, budget: int, min_slots: int = 1) -> np.ndarray:
    """Per-layer ring sizes (int32 [layers]) minimising the summed host-link experts
    of the layers' LRU curves (uint64 [layers, max_slots]) within a total budget."""
    c = np.ascontiguousarray(curves, np.uint64)
    out = np.zeros(c.shape[0], np.int32)
    _check(lib().moe_policy_size_layers(c.ctypes.data, c.shape[0], c.shape[1], budget, min_slots,
                                        out.ctypes.data), "moe_policy_size_layers")
    return out
