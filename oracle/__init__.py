"""CPU oracle for the slot-cache MoE layer (test infrastructure only).

Loads ``oracle/liboracle.so`` (plain C, one thread, double precision; built
from ``oracle.c`` by :func:`build`) and wraps it for numpy callers.  Only the
tests, the package smoke check and the benchmark's CPU-baseline leg may import
this module; the library under ``hbm_slot_cache_gb300`` never does, and this
module imports nothing from it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

FLAG_NONFINITE_LOGIT = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with the host C compiler."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        i64, i32, u32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_double
        L.orc_e2m1.argtypes, L.orc_e2m1.restype = [ctypes.c_uint], dbl
        L.orc_e4m3.argtypes, L.orc_e4m3.restype = [ctypes.c_uint], dbl
        L.orc_bf16.argtypes, L.orc_bf16.restype = [ctypes.c_uint], dbl
        L.orc_expert_bytes.argtypes = [i64, i64, P, P]
        L.orc_route.argtypes, L.orc_route.restype = [P, i32, i32, P, P], ctypes.c_uint
        L.orc_nvfp4_matvec.argtypes = [P, P, dbl, i64, i64, P, P]
        L.orc_expert_ffn.argtypes = [P, P, P, i64, i64, P, P, P]
        L.orc_moe_rows.argtypes = [P, P, P, i64, i64, i64, i32, i32, P, P, P, P, P]
        L.orc_moe_rows.restype = ctypes.c_uint
        L.orc_lru_step.argtypes = [i32, i32, P, P, P, u32, i32, P, P, P, P, P, P, P]
        L.orc_lru_step.restype = i32
        L.orc_lru_list_step.argtypes = [i32, i32, P, P, P, i32, P, P, P, P, P, P, P]
        L.orc_lru_list_step.restype = i32
        _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def e2m1(code: int) -> float:
    return lib().orc_e2m1(code)


def e4m3(code: int) -> float:
    return lib().orc_e4m3(code)


def bf16(bits: int) -> float:
    return lib().orc_bf16(bits)


def expert_bytes(H: int, I: int) -> tuple[int, int]:
    bw, bs = ctypes.c_int64(), ctypes.c_int64()
    lib().orc_expert_bytes(H, I, ctypes.byref(bw), ctypes.byref(bs))
    return bw.value, bs.value


def route(logits: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray, int]:
    """Top-k ids (rank order), renormalised weights (float64) and flags for one row."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    ids = np.zeros(k, np.int32)
    w = np.zeros(k, np.float64)
    flags = lib().orc_route(_p(lg), lg.size, k, _p(ids), _p(w))
    return ids, w, flags


def nvfp4_matvec(codes: np.ndarray, scales: np.ndarray, gscale: float, rows: int, K: int,
                 v: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes, np.uint8)
    s = np.ascontiguousarray(scales, np.uint8)
    vv = np.ascontiguousarray(v, np.float64)
    assert c.size >= rows * K // 2 and s.size >= rows * K // 16 and vv.size >= K
    out = np.zeros(rows, np.float64)
    lib().orc_nvfp4_matvec(_p(c), _p(s), float(gscale), rows, K, _p(vv), _p(out))
    return out


def expert_ffn(w_e: np.ndarray, s_e: np.ndarray, gs3: np.ndarray, H: int, I: int,
               x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(y[H], h[I]) for one expert applied to x (float64)."""
    w = np.ascontiguousarray(w_e, np.uint8)
    s = np.ascontiguousarray(s_e, np.uint8)
    g = np.ascontiguousarray(gs3, np.float32)
    xx = np.ascontiguousarray(x, np.float64)
    bw, bs = expert_bytes(H, I)
    assert w.size >= bw and s.size >= bs and g.size >= 3 and xx.size >= H
    y = np.zeros(H, np.float64)
    h = np.zeros(I, np.float64)
    lib().orc_expert_ffn(_p(w), _p(s), _p(g), H, I, _p(xx), _p(y), _p(h))
    return y, h


def moe_rows(w: np.ndarray, s: np.ndarray, gscale: np.ndarray, E: int, H: int, I: int,
             k: int, logits: np.ndarray, x_bf16: np.ndarray):
    """Layer result for M rows: (out float64 [M,H], ids int32 [M,k], wts float64 [M,k], flags).

    ``w``/``s`` may be any buffer-like with E experts back to back (uint8 view)."""
    lg = np.ascontiguousarray(logits, np.float32).reshape(-1, E)
    M = lg.shape[0]
    xb = np.ascontiguousarray(x_bf16, np.uint16).reshape(M, H)
    gs = np.ascontiguousarray(gscale, np.float32)
    bw, bs = expert_bytes(H, I)
    assert w.size >= E * bw and s.size >= E * bs and gs.size >= 3 * E
    out = np.zeros((M, H), np.float64)
    ids = np.zeros((M, k), np.int32)
    wts = np.zeros((M, k), np.float64)
    flags = lib().orc_moe_rows(_p(w), _p(s), _p(gs), E, H, I, k, M, _p(lg), _p(xb),
                               _p(out), _p(ids), _p(wts))
    return out, ids, wts, flags


class LRUSim:
    """Per-layer slot-cache trace (O-2) in both formulations, checked against each other."""

    def __init__(self, E: int, S: int, check_list: bool = True):
        self.E, self.S = E, S
        self.map = np.full(E, -1, np.int32)
        self.owner = np.full(S, -1, np.int32)
        self.stamp = np.zeros(S, np.uint32)
        self.t = 0
        self.check_list = check_list
        if check_list:
            self.lmap = np.full(E, -1, np.int32)
            self.lowner = np.full(S, -1, np.int32)
            self.order = np.arange(S, dtype=np.int32)
        self.stats = dict(steps=0, picks=0, hits=0, misses=0, evictions=0, bypass=0)

    def step(self, ids: np.ndarray) -> dict:
        """One layer-step over all picks (flattened row-major [M*k]); returns the record."""
        picks = np.ascontiguousarray(ids, np.int32).ravel()
        n = picks.size
        outs = [np.zeros(n, np.int32) for _ in range(5)] + [np.zeros(1, np.int32)]
        slot, hit, me, mv, mev, nu = outs
        self.t += 1
        nm = lib().orc_lru_step(self.E, self.S, _p(self.map), _p(self.owner), _p(self.stamp),
                                self.t, n, _p(picks), _p(slot), _p(hit), _p(me), _p(mv),
                                _p(mev), _p(nu))
        if self.check_list:
            louts = [np.zeros(n, np.int32) for _ in range(5)] + [np.zeros(1, np.int32)]
            nm2 = lib().orc_lru_list_step(self.E, self.S, _p(self.lmap), _p(self.lowner),
                                          _p(self.order), n, _p(picks), *[_p(a) for a in louts])
            k = max(nm, 0)
            if nm2 != nm or not (np.array_equal(louts[0], slot) and np.array_equal(louts[1], hit)
                                 and np.array_equal(louts[2][:k], me[:k])
                                 and np.array_equal(louts[3][:k], mv[:k])
                                 and np.array_equal(louts[4][:k], mev[:k])):
                raise AssertionError("stamp and recency-list LRU formulations disagree")
        self.stats["steps"] += 1
        if nm < 0:
            self.t -= 1  # a bypassed step does not advance the layer's clock
            self.stats["bypass"] += 1
            return dict(bypass=True, n_union=int(nu[0]), hit=hit.copy(), slot=slot.copy(),
                        miss_e=me[:0].copy(), miss_v=mv[:0].copy(), miss_evicted=mev[:0].copy())
        self.stats["picks"] += n
        self.stats["hits"] += int(hit.sum())
        self.stats["misses"] += nm
        self.stats["evictions"] += int((mev[:nm] >= 0).sum())
        return dict(bypass=False, n_union=int(nu[0]), hit=hit.copy(), slot=slot.copy(),
                    miss_e=me[:nm].copy(), miss_v=mv[:nm].copy(), miss_evicted=mev[:nm].copy())
