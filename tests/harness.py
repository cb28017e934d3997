"""Test/bench helpers: build seeded host banks, drive the library, compare with the oracle.

Imports the library and (for comparisons) the oracle; the library never imports this.
"""
from __future__ import annotations

import numpy as np

import workload


def tolerance_metrics(got: np.ndarray, ref: np.ndarray) -> dict:
    """Errors of a layer output against the oracle: max |d| / max |ref| (the stated
    'max relative error') and mean |d| (absolute), plus both normalised by RMS(ref)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) or 1.0
    return dict(max_rel=float(d.max() / max(np.abs(ref).max(), 1e-30)), mae=float(d.mean()),
                max_over_rms=float(d.max() / rms), mae_over_rms=float(d.mean() / rms))


MAX_REL_TOL = 2e-2   # max |gpu - oracle| / max |oracle|
MAE_TOL = 1e-3       # mean |gpu - oracle|, absolute, fp32 output


# Inputs far outside the configurations' output scale (the wide-range x, whose
# outputs reach ~1e8) take the scale-free form of the mean bound: 1e-3 absolute
# at the GLM layer's output RMS of ~12 is ~8e-5 of the RMS.
MAE_OVER_RMS_TOL = 1e-4


def assert_within_tolerance(got, ref, what="", scale_free=False):
    m = tolerance_metrics(got, ref)
    if scale_free:
        ok = m["max_rel"] <= MAX_REL_TOL and m["mae_over_rms"] <= MAE_OVER_RMS_TOL
    else:
        ok = m["max_rel"] <= MAX_REL_TOL and m["mae"] <= MAE_TOL
    assert ok, f"{what}: {m}"
    return m


class PlainBank:
    """Ordinary host memory with HostBank's interface (.array, .close()), for
    users that only read the bytes on the CPU."""

    def __init__(self, nbytes: int):
        self.array = np.empty(int(nbytes), np.uint8)

    def close(self) -> None:
        self.array = None


class Banks:
    """Host banks for `distinct` layers of a config (layers beyond that alias
    bank l % distinct; routing stays independent per layer): pinned, mapped
    memory the library can read, or (pinned=False) ordinary memory for the
    oracle alone."""

    def __init__(self, cfg: workload.Config, distinct: int = 1, pinned: bool = True):
        if pinned:
            from hbm_slot_cache_gb300 import HostBank as Bank
        else:
            Bank = PlainBank
        self.cfg = cfg
        self.Bw, self.Bs = workload.storage_bytes(cfg.hidden, cfg.inter)
        self.w, self.s, self.g = [], [], []
        for l in range(distinct):
            w = Bank(cfg.experts * self.Bw)
            s = Bank(cfg.experts * self.Bs)
            workload.fill_bank(w.array, s.array, cfg.experts, cfg.hidden, cfg.inter, cfg.seed, l,
                               scales=cfg.scales)
            self.w.append(w)
            self.s.append(s)
            self.g.append(workload.global_scales(cfg.experts, cfg.scales, cfg.seed, l))
        self.distinct = distinct

    def host_layers(self, layers: int):
        return [(self.w[l % self.distinct], self.s[l % self.distinct], self.g[l % self.distinct])
                for l in range(layers)]

    def layer_arrays(self, layer: int):
        d = layer % self.distinct
        return self.w[d].array, self.s[d].array, self.g[d]

    def close(self):
        for b in self.w + self.s:
            b.close()


def make_cache(cfg: workload.Config, banks: Banks, layers: int | None = None, slots=None, **kw):
    from hbm_slot_cache_gb300 import MoeCache
    L = cfg.layers if layers is None else layers
    return MoeCache(L, cfg.experts, cfg.slots if slots is None else slots, cfg.hidden, cfg.inter,
                    cfg.top_k, banks.host_layers(L), **kw)


def record_ids(rec, rows: int, k: int) -> np.ndarray:
    return np.array(rec.ids[:rows * k], np.int32).reshape(rows, k)


def check_record_against_sim(rec, sim_rec, rows: int, k: int) -> None:
    """GPU step record vs oracle LRU record: bit-exact."""
    n = rows * k
    assert bool(rec.bypass) == sim_rec["bypass"]
    assert rec.n_union == sim_rec["n_union"]
    assert list(rec.hit[:n]) == [int(v) for v in sim_rec["hit"]]
    if not sim_rec["bypass"]:
        assert list(rec.slot[:n]) == [int(v) for v in sim_rec["slot"]]
        m = rec.n_miss
        assert m == len(sim_rec["miss_e"])
        assert list(rec.miss_expert[:m]) == sim_rec["miss_e"].tolist()
        assert list(rec.miss_slot[:m]) == sim_rec["miss_v"].tolist()
        assert list(rec.miss_evicted[:m]) == sim_rec["miss_evicted"].tolist()
