"""Offline slot-policy analysis (moe_policy_*), host only.

The library's LRU policy simulator is pinned to the oracle's LRU (O-2) step by
step on random traces, with multi-row picks and bypassed steps; the static,
hybrid and sizing functions are pinned to brute force on small cases."""
import itertools

import numpy as np
import pytest

import workload


@pytest.fixture(scope="module")
def pol():
    import hbm_slot_cache_gb300 as m
    m.build()
    return m


def _oracle_lru(orc, trace, E, S):
    sim = orc.LRUSim(E, S)
    host = 0
    for ids in trace:
        r = sim.step(ids)
        host += r["n_union"] if r["bypass"] else len(r["miss_e"])
    st = sim.stats
    return dict(picks=st["picks"], hits=st["hits"], misses=st["misses"],
                evictions=st["evictions"], bypass_steps=st["bypass"], host_experts=host)


@pytest.mark.parametrize("E,S,picks,seed", [(8, 2, 2, 0), (8, 3, 4, 1), (16, 4, 8, 2),
                                             (16, 8, 6, 3), (32, 5, 16, 4)])
def test_lru_policy_matches_oracle(pol, orc, E, S, picks, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    trace = rng.choice(E, size=(120, picks), p=p / p.sum()).astype(np.int32)
    got = pol.moe_policy_lru(trace, E, S)
    ref = _oracle_lru(orc, trace, E, S)
    assert got["steps"] == 120
    for key, v in ref.items():
        assert got[key] == v, (key, got, ref)


def test_lru_policy_glm_trace_matches_oracle(pol, orc):
    cfg = workload.CONFIGS["glm"]
    rt = workload.Routing(cfg)
    trace = np.stack([orc.route(rt.step()[0], cfg.top_k)[0] for _ in range(150)])
    got = pol.moe_policy_lru(trace, cfg.experts, cfg.slots)
    ref = _oracle_lru(orc, trace, cfg.experts, cfg.slots)
    for key, v in ref.items():
        assert got[key] == v, key


def test_static_policy_brute_force(pol):
    rng = np.random.default_rng(5)
    E, picks = 12, 3
    trace = rng.integers(0, E, size=(40, picks)).astype(np.int32)
    counts = np.bincount(trace.ravel(), minlength=E)
    order = sorted(range(E), key=lambda e: (-counts[e], e))
    for S in (0, 1, 4, 12):
        pinned = set(order[:S])
        hits = sum(int(e in pinned) for e in trace.ravel())
        host = sum(len(set(row) - pinned) for row in trace.tolist())
        got = pol.moe_policy_static(trace, E, S)
        assert got["hits"] == hits and got["host_experts"] == host and got["picks"] == trace.size


def test_hybrid_reduces_to_lru_and_static(pol):
    rng = np.random.default_rng(6)
    E = 20
    trace = rng.integers(0, E, size=(80, 4)).astype(np.int32)
    for S in (4, 7):
        assert pol.moe_policy_hybrid(trace, E, S, 0) == pol.moe_policy_lru(trace, E, S)
        assert pol.moe_policy_hybrid(trace, E, S, S) == pol.moe_policy_static(trace, E, S)
        h = pol.moe_policy_hybrid(trace, E, S, 2)
        assert h["picks"] + 0 <= trace.size and h["hits"] <= h["picks"]


def test_lru_curve_matches_single_runs(pol):
    rng = np.random.default_rng(7)
    E = 24
    trace = rng.integers(0, E, size=(60, 5)).astype(np.int32)
    curve = pol.moe_policy_lru_curve(trace, E, 10)
    for S in range(1, 11):
        assert curve[S - 1] == pol.moe_policy_lru(trace, E, S)["host_experts"]


def test_size_layers_brute_force(pol):
    rng = np.random.default_rng(8)
    L, max_s = 3, 5
    curves = np.sort(rng.integers(0, 100, size=(L, max_s)), axis=1)[:, ::-1].astype(np.uint64)
    curves[1, 2] += 7                                     # a non-convex curve too
    for budget, lo in ((3, 1), (7, 1), (9, 2), (15, 1)):
        got = pol.moe_policy_size_layers(curves, budget, lo)
        best = min(sum(int(curves[l, s[l] - 1]) for l in range(L))
                   for s in itertools.product(range(lo, max_s + 1), repeat=L) if sum(s) <= budget)
        assert sum(got) <= budget and all(lo <= v <= max_s for v in got)
        assert sum(int(curves[l, got[l] - 1]) for l in range(L)) == best


def test_policy_errors(pol):
    from hbm_slot_cache_gb300 import _lib
    t = np.zeros((4, 2), np.int32)
    with pytest.raises(_lib.MoeError):
        pol.moe_policy_lru(t, 8, 0)
    with pytest.raises(_lib.MoeError):
        pol.moe_policy_lru(np.full((4, 2), 9, np.int32), 8, 2)   # id out of range
    with pytest.raises(_lib.MoeError):
        pol.moe_policy_size_layers(np.zeros((2, 4), np.uint64), 1, 1)  # budget < layers


def test_policy_report_cli(pol, orc, tmp_path):
    import json
    import subprocess
    import sys
    cfg = workload.CONFIGS["flash"]
    L, steps = 4, 80
    tr = []
    for l in range(L):
        rt = workload.Routing(cfg, layer=l)
        tr.append(np.stack([orc.route(rt.step(1)[0], cfg.top_k)[0] for _ in range(steps)]))
    p = tmp_path / "trace.npy"
    np.save(p, np.stack(tr).astype(np.int32))
    budget = L * cfg.slots
    r = subprocess.run([sys.executable, "-m", "hbm_slot_cache_gb300.policy", str(p),
                        "--experts", str(cfg.experts), "--budget", str(budget)],
                       capture_output=True, text=True, check=True)
    rep = json.loads(r.stdout)
    assert sum(rep["per_layer_slots"]) <= budget
    # sizing by the curves never reads more over the link than the uniform ring
    assert rep["sized_lru"]["host_experts"] <= rep["uniform"]["lru"]["host_experts"]
    assert 0.0 <= rep["uniform"]["static"]["hit_rate"] <= 1.0
