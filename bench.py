"""Benchmark: GLM-shape slot-cache MoE decode layer-steps/s (M=1, S=128).

One step = one layer-step of the whole hot path (route + remap/LRU, miss copy
over the host link, NVFP4 gate/up + SwiGLU, down + combine) on one row, GLM
shape (hidden 6144, inter 2048, 256 experts, top-8, 128 slots), seeded
synthetic routing (Zipf(1.1) popularity, ~0.27 step-to-step overlap) and
weights.  The cache is warmed to steady state first (300 eager steps); every
timed step then routes a row no earlier step has seen, so misses are real and
counted, whatever K is.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
                  [--workload glm|flash|sweep|multirow|prefill]

Our arm: the per-step inputs are resident in HBM; a CUDA graph of a few steps
is captured once, and its first node (moe_feed_inputs, a device step cursor)
copies the next step's logits and x into the fixed buffers the step reads, so
every replay runs on fresh inputs.  The plain graph (programmatic launches on)
is timed in runs of K fresh steps each (at least 5, and enough to cover about
1,500 layer-steps, at most 50); the value is the median run.  Per-kernel
times come from an event-instrumented graph on further fresh steps after the
timed runs, and the end-to-end leg (moe_cache_step_host with pinned host
buffers) runs on steps after those.  N > 1 (torchrun): independent replicas,
one per GPU ("replicas only": the layer has no exchange step), value = all
ranks' steps / max time.  The reference arm (--impl reference) times the CPU
oracle as it stands on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

METRIC = "GLM-shape MoE decode layer-steps/s (M=1, S=128); % of HBM+host-link roofline"
UNIT = "layer-steps/s"
GLM_MOE_LAYERS = 75  # tok/s-equivalent = layer-steps/s / 75 MoE layers


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return 6800.0, "fallback (6.8 TB/s)"


def job_rate(ms_local: float, units_local: int, world: int, device) -> tuple[float, float]:
    """Whole-job rate of `world` replicas that each processed `units_local` units:
    the job's time is the slowest rank's (max over ranks, an all-reduce when
    world > 1).  Returns (units per second over all ranks, that time in ms)."""
    import torch
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms = float(t.item())
    return world * units_local / (ms * 1e-3), ms


def _src_sha() -> str:
    h = hashlib.sha256()
    cs = os.path.join(ROOT, "hbm_slot_cache_gb300", "csrc")
    for f in sorted(os.listdir(cs)):
        h.update(open(os.path.join(cs, f), "rb").read())
    return h.hexdigest()[:16]


def _traffic(kernel: str, picks: float):
    """dram bytes per launch of `picks` picks, from the committed ncu summary's bytes
    per pick, if that summary was taken on this source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("src_sha") != _src_sha():
        return None
    k = d.get("kernels", {}).get(kernel)
    return None if k is None else k["dram_bytes_per_pick"] * picks


def _breakdown(ev):
    """Mean event intervals of some one-row steps (events 0..7, see the header)."""
    if len(ev) == 0:
        return None
    m = ev.mean(axis=0)
    return {"route": m[1], "read_through": m[3] - m[2],
            "resident_gateup": m[5] - m[1],
            "resident_down": m[6] - m[5], "join_to_end": m[7] - max(m[6], m[4]), "step": m[7]}


class ClockSampler:
    def __init__(self, uuid: str | None):
        self.proc = None
        self.path = None
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "50"]
            if uuid:
                cmd += ["-i", uuid]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------- CPU oracle

def oracle_layer_steps(cfg, banks, seconds: float, max_steps: int) -> dict:
    """Full oracle layer-steps (route, LRU, 8-expert FFN, combine), one thread."""
    import oracle
    import workload
    rt = workload.Routing(cfg)
    xs = workload.activations(cfg.seed, 0, max_steps, 1, cfg.hidden)
    sim = oracle.LRUSim(cfg.experts, cfg.slots, check_list=False)
    w, s, g = banks.layer_arrays(0)
    n, t0 = 0, time.perf_counter()
    while n < max_steps and (n == 0 or time.perf_counter() - t0 < seconds):
        lg = rt.step()
        _, ids, _, _ = oracle.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k,
                                       lg, xs[n])
        sim.step(ids)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} full GLM layer-steps (route, LRU, 8 experts x 3 NVFP4 matvecs in "
                      f"double, combine) in {dt:.1f} s, single-threaded C"}


def oracle_sampled_step(cfg, banks, sim, rt, x, frac: float) -> float:
    """One reference-arm step: route + LRU in full, then for each of the k picked
    experts the NVFP4 matvecs on a fraction `frac` of the gate/up rows (K = hidden)
    and of the down rows (K = inter); returns the time scaled to a full layer-step."""
    import oracle
    t0 = time.perf_counter()
    lg = rt.step()
    ids, _, _ = oracle.route(lg[0], cfg.top_k)
    sim.step(ids)
    t1 = time.perf_counter()
    H, I = cfg.hidden, cfg.inter
    w, s, _ = banks.layer_arrays(0)
    bw, bs = banks.Bw, banks.Bs
    xd = (x[0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    hv = np.tanh(xd[:I])
    n_gu = max(1, int(round(2 * I * frac)))
    n_dn = max(1, int(round(H * frac)))
    for e in ids.tolist():
        we, se = w[e * bw:(e + 1) * bw], s[e * bs:(e + 1) * bs]
        oracle.nvfp4_matvec(we, se, 1 / 64, n_gu, H, xd)
        oracle.nvfp4_matvec(we[I * H:], se[I * H // 8:], 1 / 64, n_dn, I, hv)
    t2 = time.perf_counter()
    return (t1 - t0) + (t2 - t1) / frac


def run_reference(args) -> None:
    """The CPU oracle as it stands, single-threaded, on the glm workload.  Every
    step is the oracle's full layer-step (route, LRU, the k experts' NVFP4 FFN in
    double, combine) when warm-up + steps fit in about three minutes at ~2.7 s a
    step; otherwise each step runs the FFN on a fraction of every matrix's rows
    and its time is scaled to a full step (the line then says "extrapolated")."""
    import workload
    from harness import Banks
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    cfg = workload.CONFIGS["glm"]
    banks = Banks(cfg, pinned=False)  # the oracle reads the bytes on the CPU only
    rt = workload.Routing(cfg)
    sim = oracle.LRUSim(cfg.experts, cfg.slots, check_list=False)
    n = args.steps + args.warmup
    full = n * 2.7 <= 180.0
    xs = workload.activations(cfg.seed, 0, n, 1, cfg.hidden)
    w, s, g = banks.layer_arrays(0)

    def full_step(i):
        t0 = time.perf_counter()
        lg = rt.step()
        _, ids, _, _ = oracle.moe_rows(w, s, g, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k,
                                       lg, xs[i])
        sim.step(ids)
        return time.perf_counter() - t0

    frac = 1.0
    if full:
        for i in range(args.warmup):
            full_step(i)
        t = [full_step(args.warmup + i) for i in range(args.steps)]
        sample = "every step in full: route, LRU, 8 experts x 3 NVFP4 matvecs in double, combine"
    else:
        frac = min(1.0, max(1.0 / 2048, 60.0 / (7.0 * n)))
        for i in range(args.warmup):
            oracle_sampled_step(cfg, banks, sim, rt, xs[i], frac)
        t = [oracle_sampled_step(cfg, banks, sim, rt, xs[args.warmup + i], frac)
             for i in range(args.steps)]
        sample = (f"per step: route + LRU in full, expert FFN on {frac:.5f} of each matrix's "
                  "rows, time scaled to a full layer-step")
    sec = float(np.sum(t))
    value = args.steps / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "extrapolated": not full,
            "config": {"workload": "glm-layer M=1 S=128 (hidden 6144, inter 2048, 256 experts, top-8)",
                       "global_batch": 1, "parallelism": "cpu oracle, 1 thread"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample, "extrapolated": not full,
                             "fraction_of_rows_computed": frac},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    banks.close()


# ---------------------------------------------------------------- our arm

# Timed runs of K rounds each, over distinct fresh rounds; the median run is
# reported.  At least 5 runs, and enough that the runs cover ~RUN_LAYER_STEPS
# layer-steps together (at most 50 runs), so a short K still samples the
# workload's miss mix instead of a handful of steps.
RUNS_MIN, RUNS_MAX, RUN_LAYER_STEPS = 5, 50, 1500


def n_runs(K: int, L: int = 1) -> int:
    return max(RUNS_MIN, min(RUNS_MAX, -(-RUN_LAYER_STEPS // max(K * L, 1))))
# Untimed fresh rounds replayed right before the timed runs, about this long: after
# even a fraction of a second idle (graph capture, the clock sampler's start) the
# first ~100 ms of steps ran up to 2-3x slower (the host link and memory come back
# from idle), so the timed runs start on a busy GPU.
PRERUN_S = 0.25
PRERUN_EST_ROUND_S = 1.7e-4  # per layer-step, to size the pre-run's slice of the trace


class Feeder:
    """Seeded per-round inputs held in device memory, the fixed buffers a captured
    round reads, and the device step cursor (moe_feed_inputs) that copies the next
    round's inputs into those buffers as the round's first node, so one graph
    replays over rounds it has never seen."""

    def __init__(self, lgs: np.ndarray, xs: np.ndarray):
        import torch
        # lgs: fp32 [T, L, E]; xs: bf16 bits [T, L, H]
        self.T = lgs.shape[0]
        self.lg_tr = torch.from_numpy(np.ascontiguousarray(lgs, np.float32)).cuda()
        self.x_tr = torch.from_numpy(np.ascontiguousarray(xs).view(np.int16)).cuda()
        self.lg = torch.empty_like(self.lg_tr[0])
        self.x = torch.empty_like(self.x_tr[0]).view(torch.bfloat16)
        self.cursor = torch.zeros(2, dtype=torch.int32, device="cuda")

    def feed(self, stream) -> None:
        from hbm_slot_cache_gb300 import _lib
        _lib.moe_feed_inputs(self.lg_tr.data_ptr(), self.x_tr.data_ptr(),
                             self.lg.numel() * 4, self.x.numel() * 2, self.T,
                             self.lg.data_ptr(), self.x.data_ptr(), self.cursor.data_ptr(),
                             stream.cuda_stream)

    def position(self) -> int:
        return int(self.cursor[0].item())

    def seek(self, t: int) -> None:
        import torch
        torch.cuda.synchronize()
        self.cursor.zero_()
        self.cursor[0] = t
        torch.cuda.synchronize()


def decode_bench(cfg, *, layers: int, slots: int, K: int, W: int, prewarm: int,
                 ev_rounds: int, e2e_rounds: int, cold_rounds: int, world: int, rank: int,
                 banks=None, seed_layers_from: int = 0) -> dict:
    """One-row decode rounds (each round steps `layers` layers once) of config `cfg`
    with `slots` slots a layer.  Every timed round consumes fresh inputs.

    Sequence: `prewarm` eager rounds from an empty ring (steady state), W warm-up
    rounds through the graphs, n_runs(K) timed runs of K rounds (the plain graph with
    programmatic launches; the value is the median run), then, on further fresh
    rounds, an event-instrumented graph for per-kernel times, the end-to-end leg
    through moe_cache_step_host with pinned host buffers, and a cold start (the
    first rounds again from an empty ring).  Returns the measurements."""
    import torch
    import torch.distributed as dist

    import workload
    from harness import Banks, make_cache
    import hbm_slot_cache_gb300 as hsc

    E, H, I, k, L = cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, layers
    own_banks = banks is None
    if own_banks:
        banks = Banks(cfg)
    cache = make_cache(cfg, banks, layers=L, slots=slots, trace_capacity=max(ev_rounds, 8))
    B = max(1, min(10, W - 1))            # rounds in the multi-round graph
    prerun = max(2 * B, min(2000, int(PRERUN_S / (PRERUN_EST_ROUND_S * L))))
    RUNS = n_runs(K, L)
    T_dev = prewarm + W + prerun + RUNS * K + ev_rounds
    T = T_dev + e2e_rounds
    rts = [workload.Routing(cfg, layer=seed_layers_from + l) for l in range(L)]
    lgs = np.empty((T, L, E), np.float32)
    for t in range(T):
        for l in range(L):
            lgs[t, l] = rts[l].step(1)[0]
    xs = np.stack([workload.activations(cfg.seed, seed_layers_from + l, T, 1, H)[:, 0]
                   for l in range(L)], axis=1)                      # [T, L, H] bf16 bits
    fd = Feeder(lgs[:T_dev], xs[:T_dev])
    out = torch.empty((L, 1, H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    evs = None

    def one_round(with_events=False, r=0):
        fd.feed(stream)
        for l in range(L):
            if with_events:
                hsc.moe_cache_set_timing_events(cache.h, [e.cuda_event for e in evs[r * L + l]])
            cache.step(l, fd.lg[l:l + 1], fd.x[l:l + 1], out[l], stream)
        if with_events:
            hsc.moe_cache_set_timing_events(cache.h, None)

    def capture(n, with_events=False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(n):
                one_round(with_events, r)
        return g

    def replay(g1, gB, n):
        for _ in range(n // B):
            gB.replay()
        for _ in range(n % B):
            g1.replay()

    with torch.cuda.stream(stream):
        for _ in range(prewarm):           # eager: fills the rings to steady state
            one_round()
    stream.synchronize()
    g1, gB = capture(1), capture(B)
    with torch.cuda.stream(stream):       # warm-up: uploads both graphs (W = B + (W - B))
        gB.replay()
        for _ in range(W - B):
            g1.replay()
    stream.synchronize()
    assert fd.position() == prewarm + W, fd.position()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    with torch.cuda.stream(stream):       # pre-run: fresh rounds, untimed, no idle gap after
        replay(g1, gB, prerun)
    s0 = cache.stats(-1)                  # (synchronizes)
    run_ms = []
    for _ in range(RUNS):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            replay(g1, gB, K)
            b.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        run_ms.append(a.elapsed_time(b))
    clocks = sampler.stop()
    s1 = cache.stats(-1)
    assert s1["error_flags"] == 0, s1
    rates = [job_rate(ms, K * L, world, "cuda") for ms in run_ms]   # (units/s, max ms)
    order = np.argsort([r[1] for r in rates])
    med = rates[order[len(order) // 2]]
    ls = RUNS * K * L
    misses = (s1["misses"] - s0["misses"]) / ls
    hits, picks = s1["hits"] - s0["hits"], s1["picks"] - s0["picks"]

    # per-kernel times: an event-instrumented graph over fresh rounds (events
    # between kernels break programmatic launch, so this graph is slower)
    nev = ev_rounds * L
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(hsc._lib.MOE_TIMING_EVENTS)]
           for _ in range(nev)]
    for row in evs:
        for e in row:
            e.record(stream)
    stream.synchronize()
    g_ev = capture(ev_rounds, with_events=True)
    with torch.cuda.stream(stream):
        g_ev.replay()
    stream.synchronize()
    ev_ms = np.array([[row[0].elapsed_time(row[i]) for i in range(8)] for row in evs])
    recs = []
    for l in range(L):
        recs.append(cache.trace(l)[-ev_rounds:])
    n_miss = np.array([recs[l][r].n_miss for r in range(ev_rounds) for l in range(L)], np.float64)
    del g_ev

    # end to end through the public API on further fresh rounds: moe_cache_step_host
    # with pinned host buffers (H2D of logits and x, the step, D2H of out), every
    # layer-step inside the timed region
    e2e = None
    if e2e_rounds > 0:
        lg_h = torch.from_numpy(lgs[T_dev:].copy()).pin_memory()
        x_h = torch.from_numpy(xs[T_dev:].view(np.int16).copy()).pin_memory().view(torch.bfloat16)
        out_h = torch.empty((e2e_rounds, L, 1, H), dtype=torch.float32).pin_memory()
        bufs = [(l, lg_h[t, l:l + 1], x_h[t, l:l + 1], out_h[t, l])
                for t in range(e2e_rounds) for l in range(L)]
        with torch.cuda.stream(stream):   # untimed: each layer's eager step, then its capture
            for l, lg_t, x_t, o_t in bufs[:2 * L]:
                cache.step_host(l, lg_t, x_t, o_t, stream)
        stream.synchronize()
        bufs = bufs[2 * L:]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        se0 = cache.stats(-1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            h0 = time.perf_counter()
            for l, lg_t, x_t, o_t in bufs:
                cache.step_host(l, lg_t, x_t, o_t, stream)
            h1 = time.perf_counter()
            e1.record(stream)
        stream.synchronize()
        n = len(bufs)
        e2e_value, _ = job_rate(e0.elapsed_time(e1), n, world, "cuda")
        e2e = {"value": e2e_value, "unit": UNIT, "host_us_per_call": 1e6 * (h1 - h0) / n,
               "misses_per_step": (cache.stats(-1)["misses"] - se0["misses"]) / n,
               "h2d_bytes_per_step": E * 4 + H * 2, "d2h_bytes_per_step": H * 4, "steps": n,
               "note": "fresh rounds after the device-resident ones; pinned host buffers"}

    # cold: the first rounds again from an empty ring, through the same graphs
    cold = None
    if cold_rounds > 0:
        cache.reset()
        fd.seek(0)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            c0.record(stream)
            replay(g1, gB, cold_rounds)
            c1.record(stream)
        stream.synchronize()
        sc = cache.stats(-1)
        cold = {"value": cold_rounds * L / (c0.elapsed_time(c1) * 1e-3), "unit": UNIT,
                "rounds": cold_rounds, "misses_per_step": sc["misses"] / (cold_rounds * L),
                "note": "rounds 0..n from an empty ring, the same graphs (the value is steady "
                        f"state after a {prewarm}-round pre-warm)"}
    del g1, gB
    cache.close()
    if own_banks:
        banks.close()
    return {"run_ms": run_ms, "value": med[0], "ms_total": med[1], "misses_per_step": misses,
            "hit_rate": hits / picks if picks else None, "clocks": clocks, "ev_ms": ev_ms,
            "ev_n_miss": n_miss, "e2e": e2e, "cold": cold, "K": K, "L": L, "B": B,
            "prerun": prerun, "runs": RUNS,
            "Bexp": banks.Bw + banks.Bs}


def link_probe() -> tuple[float, float]:
    """Host-link bandwidth in the same session: SM 16-byte loads and cudaMemcpyAsync,
    1 GiB pinned -> HBM, best of 5 each."""
    import torch
    from hbm_slot_cache_gb300 import HostBank, moe_probe_host_link
    nb = 1 << 30
    hb = HostBank(nb)
    hb.array[::4096] = 1
    dst = torch.empty(nb, dtype=torch.uint8, device="cuda")
    try:
        return (moe_probe_host_link(hb.ptr, dst.data_ptr(), nb, 0, 5),
                moe_probe_host_link(hb.ptr, dst.data_ptr(), nb, 1, 5))
    finally:
        del dst
        hb.close()


def roofline_terms(cfg, res: dict, hbm_peak: float, link_peak: float) -> dict:
    """Serial path roofline of the timed rounds (k experts' bytes over HBM + the
    counted miss bytes over the host link, per layer-step) and the overlapped
    bound over the instrumented layer-steps."""
    k, Bexp = cfg.top_k, res["Bexp"]
    ms_step = res["ms_total"] / (res["K"] * res["L"])
    hbm_bytes = k * Bexp
    link_bytes = res["misses_per_step"] * Bexp
    t_roof = hbm_bytes / (hbm_peak * 1e9) + link_bytes / (link_peak * 1e9)
    nm = res["ev_n_miss"]
    t_max = float(np.mean(np.maximum((k - nm) * Bexp / (hbm_peak * 1e9),
                                     nm * Bexp / (link_peak * 1e9))))
    return {"frac": t_roof / (ms_step * 1e-3), "t_roofline_us": t_roof * 1e6,
            "t_measured_us": ms_step * 1e3, "hbm_bytes_per_step": hbm_bytes,
            "link_bytes_per_step": link_bytes, "hbm_peak_gbs": hbm_peak,
            "link_peak_gbs": link_peak, "misses_per_step": res["misses_per_step"],
            "hit_rate": res["hit_rate"],
            "overlapped_bound": {"t_us": t_max * 1e6, "frac": t_max / (ms_step * 1e-3),
                                 "note": "mean over the instrumented steps of max(hit bytes / "
                                         "HBM peak, miss bytes / link peak)"}}


def kernel_table(cfg, res: dict, hbm_peak: float, link_peak: float) -> tuple[dict, dict]:
    """Per-kernel rooflines from the event-instrumented layer-steps: algorithmic
    bytes of each launch over its event-timed duration."""
    H, I, k, Bexp = cfg.hidden, cfg.inter, cfg.top_k, res["Bexp"]
    ev, n_miss = res["ev_ms"], res["ev_n_miss"]
    n_hit = k - n_miss
    G = len(ev)
    t_route = ev[:, 1]
    t_rt = ev[:, 3] - ev[:, 2]
    t_gu_hit = ev[:, 5] - ev[:, 1]
    t_dn_hit = ev[:, 6] - ev[:, 5]
    gu_pick = 2 * I * (H // 2 + H // 16)
    dn_pick = H * (I // 2 + I // 16)

    def entry(bytes_total, ms_total, peak, bound, launches):
        ach = bytes_total / (ms_total * 1e-3) / 1e9 if ms_total > 0 else None
        return {"bound": bound, "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak if ach else None,
                "algorithmic_bytes_per_launch": bytes_total / launches,
                "ms_per_launch": ms_total / launches}
    hm = n_miss > 0
    nm = max(int(hm.sum()), 1)
    kern = {
        "gemv_gateup[resident picks]": entry(float((n_hit * gu_pick).sum()), float(t_gu_hit.sum()),
                                             hbm_peak, "hbm", G),
        "gemv_down[resident picks]": entry(float((n_hit * dn_pick).sum()), float(t_dn_hit.sum()),
                                           hbm_peak, "hbm", G),
        "gemv_readthrough[missed picks]": entry(float((n_miss * Bexp).sum()),
                                                float(t_rt[hm].sum()), link_peak, "host-link", nm),
        "route_remap": {"ms_per_launch": float(t_route.mean())},
    }
    # the resident passes alone: on steps without a miss nothing shares their SMs
    if (~hm).any():
        for n, t_k, per in (("gemv_gateup[resident picks]", t_gu_hit, gu_pick),
                             ("gemv_down[resident picks]", t_dn_hit, dn_pick)):
            b = float((n_hit[~hm] * per).sum())
            a = b / (float(t_k[~hm].sum()) * 1e-3) / 1e9
            kern[n]["steps_without_miss"] = {"achieved": a, "frac": a / hbm_peak,
                                             "ms_per_launch": float(t_k[~hm].mean())}
    for n in kern:
        if "resident" in n:
            kern[n]["traffic"] = _traffic(n.split("[")[0], float(n_hit.mean()))
        elif "missed" in n:
            kern[n]["traffic"] = _traffic(n.split("[")[0],
                                          float(n_miss[hm].mean()) if hm.any() else 0.0)
            kern[n]["note"] = "steps with at least one miss"
    kern["gemv_readthrough[missed picks]"]["note"] += (
        "; whole missed experts over the host link, written to their slots, gate/up and "
        "down computed on the way in; traffic = its DRAM bytes (the slot write-through)")
    if hm.any():
        # read-through time against the step's miss count: mean per count, and a
        # least-squares line t = fixed + n * per_miss (the per-miss slope is the
        # marginal link rate, the intercept the launch's fixed part)
        by = {int(n): round(float(t_rt[n_miss == n].mean()) * 1e3, 1)
              for n in np.unique(n_miss[hm])}
        fit = None
        if len(by) >= 2:
            slope, icpt = np.polyfit(n_miss[hm].astype(float), t_rt[hm] * 1e-3, 1)
            fit = {"fixed_us": round(float(icpt) * 1e6, 1),
                   "per_miss_us": round(float(slope) * 1e6, 1),
                   "marginal_link_gbs": round(Bexp / slope / 1e9, 1) if slope > 0 else None}
        kern["gemv_readthrough[missed picks]"]["us_by_misses"] = by
        kern["gemv_readthrough[missed picks]"]["fit"] = fit
    split = {"ms_per_step_event_graph": float(ev[:, 7].mean()),
             "ms_miss_path": float(np.mean(ev[:, 4] - ev[:, 1])),
             "ms_hit_path": float(np.mean(ev[:, 6] - ev[:, 1])),
             "ms_route": float(np.mean(t_route)),
             "ms_step_with_miss": float(np.mean(ev[hm, 7])) if hm.any() else None,
             "ms_step_no_miss": float(np.mean(ev[~hm, 7])) if (~hm).any() else None,
             "frac_steps_with_miss": float(np.mean(hm)),
             "no_miss_breakdown_ms": _breakdown(ev[~hm]),
             "with_miss_breakdown_ms": _breakdown(ev[hm]),
             "instrumented_steps": G}
    return kern, split


def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    import workload
    import hbm_slot_cache_gb300 as hsc

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    hsc.build()
    cfg = workload.CONFIGS["glm"]
    K, W = args.steps, args.warmup
    res = decode_bench(cfg, layers=1, slots=cfg.slots, K=K, W=W, prewarm=300, ev_rounds=200,
                       e2e_rounds=max(min(K, 1000), 300) + 2, cold_rounds=300, world=world, rank=rank)
    # sanity: the timed rounds must exercise the miss path at S = 128
    if not 0.3 <= res["misses_per_step"] <= 4.0:
        raise SystemExit(f"timed rounds saw {res['misses_per_step']:.3f} misses per layer-step at "
                         f"S={cfg.slots}: outside the workload's band, measurement invalid")
    link_sm, link_ce = link_probe()
    link_peak = max(link_sm, link_ce)
    hbm_peak, hbm_src = _peaks()
    path = roofline_terms(cfg, res, hbm_peak, link_peak)
    path.update(hbm_peak_source=hbm_src, link_probe_sm_gbs=link_sm, link_probe_memcpy_gbs=link_ce)
    kern, split = kernel_table(cfg, res, hbm_peak, link_peak)
    split["ms_per_step_plain_graph_runs"] = [m / K for m in res["run_ms"]]
    nm = max(int((res["ev_n_miss"] > 0).sum()), 1)
    G = len(res["ev_ms"])
    share = {n: v["ms_per_launch"] * (nm if "missed" in n else G) for n, v in kern.items()}
    dom = max(share, key=share.get)
    roofline = dict(kern[dom])
    roofline["kernel"] = dom
    roofline["peak_source"] = (hbm_src if roofline.get("bound") == "hbm"
                               else "moe_probe_host_link, same session (best of SM copy / cudaMemcpyAsync)")
    banks_cpu = None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from harness import Banks
        banks_cpu = Banks(cfg, pinned=False)
        cpu = oracle_layer_steps(cfg, banks_cpu, seconds=12.0, max_steps=8)
        banks_cpu.close()
    if rank == 0:
        ms_step = res["ms_total"] / K
        line = {
            "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "nvfp4 weights, fp32 accumulate", "data": "synthetic",
            "config": {"workload": "glm-layer M=1 S=128: hidden 6144, inter 2048, 256 experts, "
                                   "top-8, 128 HBM slots, Zipf(1.1) routing, steady state",
                       "global_batch": world, "seq_len": 1,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2: 170 MB of expert bytes per step > 126 MB L2; "
                             "2.7 GB slot ring",
                       "graph": f"one CUDA graph of {res['B']} rounds (and a one-round graph) "
                                "replayed; its first node feeds each round fresh inputs from a "
                                "device trace (moe_feed_inputs); programmatic launches on",
                       "timing": f"{res['runs']} runs of K fresh steps each after a 300-step pre-warm "
                                 f"and an untimed pre-run of {res['prerun']} fresh steps; "
                                 "value = median run"},
            "tok_s_equivalent": res["value"] / GLM_MOE_LAYERS,
            "path_roofline": path, "roofline": roofline, "kernels": kern, "timing_split": split,
            "cold": res["cold"], "cpu_baseline": cpu, "e2e": res["e2e"],
            "gpu_launches": K * 5, "launches_per_step": "feeder + route/remap + read-through + "
                                                        "gate/up + resident down",
            "clocks": res["clocks"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_flash_or_sweep(args) -> None:
    """The Flash-shaped 16-layer stack, or the GLM slot sweep over S: their own
    JSON line (not the headline)."""
    import torch

    import workload
    import hbm_slot_cache_gb300 as hsc

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    hsc.build()
    hbm_peak, hbm_src = _peaks()
    link_sm, link_ce = link_probe()
    link_peak = max(link_sm, link_ce)
    W = args.warmup
    if args.workload == "flash":
        cfg = workload.CONFIGS["flash"]
        L = args.layers or cfg.layers
        K = args.steps
        res = decode_bench(cfg, layers=L, slots=cfg.slots, K=K, W=W, prewarm=64, ev_rounds=16,
                           e2e_rounds=0, cold_rounds=0, world=1, rank=0)
        path = roofline_terms(cfg, res, hbm_peak, link_peak)
        kern, split = kernel_table(cfg, res, hbm_peak, link_peak)
        ls = K * L
        line = {"metric": "Flash-shape MoE decode layer-steps/s (M=1, 16 layers, S=54)",
                "value": res["value"], "unit": UNIT, "n_gpus": 1, "steps": K, "warmup": W,
                "ms_per_round": res["ms_total"] / K, "higher_is_better": True,
                "dtype": "nvfp4 weights, fp32 accumulate", "data": "synthetic",
                "config": {"workload": f"flash stack: {L} layers, hidden 4096, inter 2048, 288 "
                                       "experts, top-8, S=54 per layer, Zipf(1.05) routing "
                                       "independent per layer, one host bank aliased by every "
                                       "layer",
                           "graph": "one CUDA graph per round of all layers, fed fresh inputs",
                           "timing": f"{res['runs']} runs of K fresh rounds after an untimed pre-run "
                                     f"of {res['prerun']} fresh rounds, median"},
                "tok_s_equivalent": res["value"] / 42, "layer_steps": ls,
                "path_roofline": path, "kernels": kern, "timing_split": split,
                "clocks": res["clocks"]}
    else:
        from harness import Banks
        cfg = workload.CONFIGS["prefill"]
        L = args.layers or cfg.layers
        K = args.steps
        per_s = []
        clocks = []
        banks = Banks(cfg)
        for S in workload.SWEEP_SLOTS:
            res = decode_bench(cfg, layers=L, slots=S, K=K, W=W, prewarm=300, ev_rounds=8,
                               e2e_rounds=0, cold_rounds=300, world=1, rank=0, banks=banks)
            path = roofline_terms(cfg, res, hbm_peak, link_peak)
            per_s.append({"S": S, "layer_steps_per_s": res["value"],
                          "ms_per_layer_step": res["ms_total"] / (K * L),
                          "hit_rate": res["hit_rate"], "misses_per_step": res["misses_per_step"],
                          "path_roofline_frac": path["frac"],
                          "overlapped_bound_frac": path["overlapped_bound"]["frac"],
                          "cold": res["cold"]})
            clocks.append(res["clocks"])
        line = {"metric": "GLM-shape MoE decode layer-steps/s and hit rate per slot count "
                          "(M=1, 8 layers)",
                "value": per_s[[p["S"] for p in per_s].index(128)]["layer_steps_per_s"],
                "unit": UNIT, "n_gpus": 1, "steps": K, "warmup": W, "higher_is_better": True,
                "dtype": "nvfp4 weights, fp32 accumulate", "data": "synthetic",
                "config": {"workload": f"slot sweep: {L} layers, GLM shape, Zipf(1.1) routing "
                                       "independent per layer, S in "
                                       f"{list(workload.SWEEP_SLOTS)}; value = S=128",
                           "timing": f"300-round pre-warm and an untimed pre-run of ~{PRERUN_S} s "
                                     f"of fresh rounds, then {n_runs(K, L)} runs of K fresh rounds, "
                                     "median; cold = 300 rounds from empty"},
                "per_slots": per_s, "link_peak_gbs": link_peak, "hbm_peak_gbs": hbm_peak,
                "clocks": clocks}
        banks.close()
    print(json.dumps(line), flush=True)


# ------------------------------------------------- multi-row / prefill rounds

def run_rows(args) -> None:
    """Multi-row rounds (M = 16, cached, tcgen05) or prefill (M = 512, bypass):
    one JSON line for that workload.  Not the headline line; the default run
    measures the one-row decode step."""
    import torch

    import workload
    from harness import Banks, make_cache
    import hbm_slot_cache_gb300 as hsc

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    hsc.build()
    cfg = workload.CONFIGS[args.workload]
    E, H, I, k, M = cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, cfg.rows
    L = args.layers or cfg.layers
    W, K = args.warmup, args.steps
    prefill = args.workload == "prefill"
    # untimed fresh rounds right before the timed ones (see PRERUN_S)
    pre = max(2, int(PRERUN_S / (L * (26e-3 if prefill else 1.3e-3))) + 1)
    T = W + pre + K
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, layers=L, trace_capacity=0 if prefill else T,
                       max_rows=max(M, 16))
    Bexp = banks.Bw + banks.Bs
    # inputs: per (round, layer) logits; activations per round, shared by the layers
    if prefill:
        lgs = np.stack([np.stack([workload.prefill_logits(cfg, l, M) for l in range(L)])] * T)
    else:
        rts = [workload.Routing(cfg, layer=l) for l in range(L)]
        lgs = np.stack([np.stack([rts[l].step() for l in range(L)]) for _ in range(T)])
    xs = workload.activations(cfg.seed, 0, T, M, H)
    # every round reads fresh inputs: a one-round graph whose first node copies the
    # next trace entry into the fixed buffers (moe_feed_inputs), replayed
    fd = Feeder(lgs.astype(np.float32), xs)                  # lg [L, M, E], x [M, H]
    out_d = torch.empty((M, H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def one_round():
        fd.feed(stream)
        for l in range(L):
            cache.step(l, fd.lg[l], fd.x, out_d, stream)

    with torch.cuda.stream(stream):
        for _ in range(W):                         # eager warm-up (fills the rings)
            one_round()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        one_round()
    sampler = ClockSampler(None)
    with torch.cuda.stream(stream):
        for _ in range(pre):                       # uploads the graph, then the pre-run
            g.replay()
    s0 = cache.stats(-1)                           # (synchronizes)
    assert fd.position() == W + pre, fd.position()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(K):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    s1 = cache.stats(-1)
    layer_steps = K * L
    misses = s1["misses"] - s0["misses"]
    # experts each layer-step reads: the union of its rows' picks
    if prefill:
        ids = np.argsort(-lgs[0], axis=-1, kind="stable")[..., :k]        # [L, M, k]
        union = float(np.mean([len(np.unique(ids[l])) for l in range(L)]))
    else:
        unions = []
        for l in range(L):
            recs = cache.trace(l)[-K:]
            unions += [r.n_union for r in recs]
        union = float(np.mean(unions))
    hbm_peak, hbm_src = _peaks()
    link_peak = None
    hb = hsc.HostBank(1 << 30)
    try:
        dst = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
        link_peak = max(hsc.moe_probe_host_link(hb.ptr, dst.data_ptr(), 1 << 30, m, 5)
                        for m in (0, 1))
    finally:
        hb.close()
    s_layer = ms * 1e-3 / layer_steps
    useful_flop = 2.0 * M * k * 3 * H * I                  # per layer-step
    fp4_peak = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"] * 6.0 \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else 1900.0 * 6.0
    if prefill:
        link_bytes = union * Bexp                          # every expert read over the link
        t_roof = link_bytes / (link_peak * 1e9)
        roof = {"bound": "host-link", "bytes_per_layer_step": link_bytes,
                "t_roofline_ms": t_roof * 1e3, "frac": t_roof / s_layer, "peak_gbs": link_peak}
        metric = "GLM-shape MoE prefill bypass rows/s (M=512, 8 layers, experts read from host)"
    else:
        hbm_bytes = union * Bexp
        link_bytes = misses / layer_steps * Bexp
        t_roof = hbm_bytes / (hbm_peak * 1e9) + link_bytes / (link_peak * 1e9)
        # the hit groups run while the misses copy: bound by the larger of the
        # miss bytes over the link and the hit groups' HBM bytes, plus the
        # miss groups' HBM bytes after the copy
        hit_bytes = max(hbm_bytes - link_bytes, 0.0)
        t_ovl = max(hit_bytes / (hbm_peak * 1e9), link_bytes / (link_peak * 1e9)) \
            + link_bytes / (hbm_peak * 1e9)
        roof = {"bound": "hbm+host-link", "hbm_bytes_per_layer_step": hbm_bytes,
                "link_bytes_per_layer_step": link_bytes, "t_roofline_ms": t_roof * 1e3,
                "frac": t_roof / s_layer, "hbm_peak_gbs": hbm_peak, "hbm_peak_source": hbm_src,
                "link_peak_gbs": link_peak,
                "overlapped_bound": {"t_ms": t_ovl * 1e3, "frac": t_ovl / s_layer,
                                     "note": "max(hit groups' HBM bytes, miss bytes over the "
                                             "link) + the miss groups' HBM bytes"}}
        metric = "GLM-shape MoE multi-row round rows/s (M=16, 16 layers, S=128, tcgen05)"
    line = {"metric": metric, "value": M * layer_steps / (ms * 1e-3), "unit": "rows/s",
            "n_gpus": 1, "steps": K, "warmup": W, "ms_per_layer_step": s_layer * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "nvfp4 weights x residual nvfp4 activations, fp32 accumulate",
            "data": "synthetic",
            "config": {"workload": f"{args.workload}: hidden {H}, inter {I}, {E} experts, top-{k}, "
                                   f"M={M} rows, {L} layers, S={cfg.slots}",
                       "graph": "a one-round graph (all layers) replayed K times, its first node "
                                "feeding each round fresh inputs from a device trace",
                       "timing": f"{W} eager warm-up rounds, an untimed pre-run of {pre} fresh "
                                 "rounds, then K fresh rounds timed"},
            "layer_steps_per_s": layer_steps / (ms * 1e-3),
            "experts_read_per_layer_step": union, "misses_per_layer_step": misses / layer_steps,
            "roofline": roof,
            "tensor": {"useful_tflops": useful_flop / s_layer / 1e12,
                       "fp4_peak_tflops": fp4_peak,
                       "note": "useful = 2*M*k*3*H*I per layer-step; the MMA issues 6 "
                               "activation levels in N=32 columns per 5 rows"},
            "clocks": clocks}
    print(json.dumps(line), flush=True)
    cache.close()
    banks.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="glm",
                    choices=["glm", "flash", "sweep", "multirow", "prefill"],
                    help="glm: the one-row decode step (the headline line); flash: the "
                         "16-layer Flash stack; sweep: GLM decode per slot count; multirow / "
                         "prefill: M=16 rounds or M=512 bypass; each its own line")
    ap.add_argument("--layers", type=int, default=0, help="non-glm workloads: layers (0: config)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in ("flash", "sweep"):
        run_flash_or_sweep(args)
    elif args.workload != "glm":
        run_rows(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
