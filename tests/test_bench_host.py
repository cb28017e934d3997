"""bench.py's host-side arithmetic on synthetic measurements (no GPU): the
serial and overlapped rooflines, the per-kernel table built from event times
(algorithmic bytes over event-timed durations, the read-through's fit against
the miss count), the committed DRAM-traffic lookup, and the run count."""
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workload  # noqa: E402

GLM = workload.CONFIGS["glm"]
BEXP = 21233664  # GLM expert: 18,874,368 B of codes + 2,359,296 B of scales


def test_glm_expert_bytes_match_the_pages():
    # "GLM 5.3 Testing: HBM Expert Allocation", "What the slot cache is":
    # 18.874 MB of weights + 2.359 MB of scales = 21.234 MB per expert
    H, I = GLM.hidden, GLM.inter
    assert 3 * H * I // 2 + 3 * H * I // 16 == BEXP


def test_run_count_bounds():
    assert bench.n_runs(3000) == 5          # one run already covers 1,500 layer-steps
    assert bench.n_runs(300) == 5
    assert bench.n_runs(100) == 15
    assert bench.n_runs(20) == 50           # capped
    assert bench.n_runs(20, 16) == 5        # 16 layers a round
    assert bench.n_runs(0) == 50


def test_serial_and_overlapped_roofline_on_a_hand_case():
    res = {"Bexp": BEXP, "ms_total": 1.5, "K": 10, "L": 1, "misses_per_step": 1.0,
           "hit_rate": 0.875, "ev_n_miss": np.array([0, 1, 2])}
    r = bench.roofline_terms(GLM, res, hbm_peak=6800.0, link_peak=200.0)
    # 8 experts over HBM at 6.8 TB/s: 24.98 us; one expert over the link at
    # 200 GB/s: 106.17 us; measured 150 us a step
    assert r["t_measured_us"] == pytest.approx(150.0)
    assert r["t_roofline_us"] == pytest.approx(24.9808 + 106.1683, abs=1e-3)
    assert r["frac"] == pytest.approx((24.9808 + 106.1683) / 150.0, abs=1e-5)
    # overlapped: per step max(hit bytes / HBM, miss bytes / link) =
    # 24.98, 106.17, 212.34 us -> mean 114.50 us
    assert r["overlapped_bound"]["t_us"] == pytest.approx(
        (24.9808 + 106.1683 + 212.3366) / 3, abs=1e-3)
    assert r["hbm_bytes_per_step"] == 8 * BEXP
    assert r["link_bytes_per_step"] == BEXP


def _events(n_miss):
    """Event times (ms from the step's first event) of one-row steps: route
    10 us, resident gate/up 40 us, resident down 30 us, read-through 25 us +
    100 us per missed expert on the second stream, join 3 us after the later
    of the two paths."""
    rows = []
    for n in n_miss:
        t1 = 0.010
        t2 = t1 + 0.002
        t3 = t2 + (0.025 + 0.100 * n if n else 0.008)
        t4 = t3
        t5 = t1 + 0.040
        t6 = t5 + 0.030
        t7 = max(t4, t6) + 0.003
        rows.append([0.0, t1, t2, t3, t4, t5, t6, t7])
    return np.array(rows)


def test_kernel_table_bytes_over_event_times_and_read_through_fit(monkeypatch):
    monkeypatch.setattr(bench, "_src_sha", lambda: "not-the-profiled-source")
    n_miss = np.array([0, 1, 2, 3, 0, 1])
    res = {"Bexp": BEXP, "ev_ms": _events(n_miss), "ev_n_miss": n_miss}
    kern, split = bench.kernel_table(GLM, res, hbm_peak=6800.0, link_peak=200.0)
    H, I, k = GLM.hidden, GLM.inter, GLM.top_k
    gu_pick = 2 * I * (H // 2 + H // 16)   # 14,155,776 B
    dn_pick = H * (I // 2 + I // 16)       # 7,077,888 B
    assert gu_pick + dn_pick == BEXP
    n_hit = k - n_miss
    gu = kern["gemv_gateup[resident picks]"]
    assert gu["achieved"] == pytest.approx(
        (n_hit * gu_pick).sum() / (0.040e-3 * len(n_miss)) / 1e9)
    assert gu["frac"] == pytest.approx(gu["achieved"] / 6800.0)
    # steps without a miss: 8 picks in 40 us
    assert gu["steps_without_miss"]["achieved"] == pytest.approx(8 * gu_pick / 40e-6 / 1e9)
    dn = kern["gemv_down[resident picks]"]
    assert dn["steps_without_miss"]["achieved"] == pytest.approx(8 * dn_pick / 30e-6 / 1e9)
    rt = kern["gemv_readthrough[missed picks]"]
    # only steps with a miss: 7 experts in 3 * 25 + 7 * 100 us
    assert rt["achieved"] == pytest.approx(7 * BEXP / ((4 * 25 + 7 * 100) * 1e-6) / 1e9)
    assert rt["ms_per_launch"] == pytest.approx((4 * 0.025 + 0.7) / 4)
    assert rt["us_by_misses"] == {1: 125.0, 2: 225.0, 3: 325.0}
    assert rt["fit"]["fixed_us"] == pytest.approx(25.0, abs=0.05)
    assert rt["fit"]["per_miss_us"] == pytest.approx(100.0, abs=0.05)
    assert rt["fit"]["marginal_link_gbs"] == pytest.approx(BEXP / 100e-6 / 1e9, abs=0.1)
    # counters from another source are not reported
    assert gu["traffic"] is None and dn["traffic"] is None and rt["traffic"] is None
    assert split["frac_steps_with_miss"] == pytest.approx(4 / 6)
    assert split["no_miss_breakdown_ms"]["resident_gateup"] == pytest.approx(0.040)
    assert split["no_miss_breakdown_ms"]["resident_down"] == pytest.approx(0.030)
    assert split["ms_step_no_miss"] == pytest.approx(0.083)


def test_traffic_lookup_scales_the_committed_bytes_per_pick(monkeypatch):
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    monkeypatch.setattr(bench, "_src_sha", lambda: d["src_sha"])
    per = d["kernels"]["gemv_gateup"]["dram_bytes_per_pick"]
    assert bench._traffic("gemv_gateup", 6.5) == pytest.approx(per * 6.5)
    assert bench._traffic("no_such_kernel", 1.0) is None
    monkeypatch.setattr(bench, "_src_sha", lambda: "0" * 16)
    assert bench._traffic("gemv_gateup", 6.5) is None


def test_committed_traffic_is_close_to_the_algorithmic_bytes():
    # the captures behind the roofline's traffic field: DRAM bytes per pick
    # within a few percent of the bytes the kernels must move (no re-reads)
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for name, k in d["kernels"].items():
        ratio = k["dram_bytes_per_pick"] / k["algorithmic_bytes_per_pick"]
        assert 0.99 < ratio < 1.06, (name, ratio)


def test_job_rate_single_process():
    v, ms = bench.job_rate(2.0, 300, 1, "cpu")
    assert ms == 2.0 and v == pytest.approx(150000.0)
