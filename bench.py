"""Benchmark: GLM-shape slot-cache MoE decode layer-steps/s (M=1, S=128).

One step = one layer-step of the whole hot path (route + remap/LRU, miss copy
over the host link, NVFP4 gate/up + SwiGLU, down + combine) on one row, GLM
shape (hidden 6144, inter 2048, 256 experts, top-8, 128 slots), seeded
synthetic routing (Zipf(1.1) popularity, ~0.27 step-to-step overlap) and
weights.  The cache is warmed to steady state first; each timed step routes a
fresh row, so misses are real and counted.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Our arm: inputs resident in HBM, the K steps captured as CUDA graphs and
replayed; per-kernel times come from event-record nodes in the last graph of
the timed region.  N > 1 (torchrun): independent replicas, one per GPU
("replicas only": the layer has no exchange step), value = all ranks' steps /
max time.  The reference arm (--impl reference) times the CPU oracle as it
stands on a bounded sample of the same workload.
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
    return {"route": m[1], "read_through": m[3] - m[2], "missed_down": m[4] - m[3],
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
    # size the per-step sample so warmup + steps take about a minute
    budget_s = 60.0
    full_step_s = 7.0
    frac = min(1.0, max(1.0 / 2048, budget_s / (full_step_s * (args.steps + args.warmup))))
    xs = workload.activations(cfg.seed, 0, 1, 1, cfg.hidden)
    for _ in range(args.warmup):
        oracle_sampled_step(cfg, banks, sim, rt, xs[0], frac)
    t = [oracle_sampled_step(cfg, banks, sim, rt, xs[0], frac) for _ in range(args.steps)]
    sec = float(np.sum(t))
    value = args.steps / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "glm-layer M=1 S=128 (hidden 6144, inter 2048, 256 experts, top-8)",
                       "global_batch": 1, "parallelism": "cpu oracle, 1 thread"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"per step: route + LRU in full, expert FFN on {frac:.5f} "
                                       "of each matrix's rows, time scaled to a full layer-step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    banks.close()


# ---------------------------------------------------------------- our arm

def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    import workload
    from harness import Banks, make_cache
    import hbm_slot_cache_gb300 as hsc

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    hsc.build()

    cfg = workload.CONFIGS["glm"]
    E, H, k = cfg.experts, cfg.hidden, cfg.top_k
    banks = Banks(cfg)
    cache = make_cache(cfg, banks, layers=1, trace_capacity=200)
    prewarm = 64
    W, K = args.warmup, args.steps
    G = min(K, 200)  # steps in the final (event-instrumented) graph
    total = prewarm + W + K
    rt = workload.Routing(cfg)
    lgs = np.stack([rt.step() for _ in range(total)])                 # [T, 1, E]
    xs = workload.activations(cfg.seed, 0, total, 1, H)               # [T, 1, H] bf16 bits
    lg_d = torch.from_numpy(lgs).cuda()
    x_d = torch.from_numpy(xs.view(np.int16)).cuda().view(torch.bfloat16)
    out_d = torch.empty((1, H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def steps_on(t0, t1):
        for t in range(t0, t1):
            cache.step(0, lg_d[t], x_d[t], out_d)

    with torch.cuda.stream(stream):
        steps_on(0, prewarm)                      # fill the ring to steady state (eager)
    stream.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(G)]
    for row in evs:
        for e in row:
            e.record(stream)                      # materialise the event handles
    stream.synchronize()

    def capture(t0, t1, with_events=False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for t in range(t0, t1):
                if with_events:
                    hsc.moe_cache_set_timing_events(cache.h, [e.cuda_event for e in evs[t - t0]])
                cache.step(0, lg_d[t], x_d[t], out_d)
            hsc.moe_cache_set_timing_events(cache.h, None)
        return g

    t_w = prewarm + W
    g_warm = capture(prewarm, t_w)
    g_main = capture(t_w, t_w + K - G) if K > G else None
    g_ev = capture(t_w + K - G, t_w + K, with_events=True)

    # Warm-up: the W-step graph, then one untimed pass of each timed graph (a
    # graph's first launch uploads it; the timed replays are the second).
    with torch.cuda.stream(stream):
        g_warm.replay()
        if g_main is not None:
            g_main.replay()
        g_ev.replay()
    stream.synchronize()
    s0 = cache.stats(0)

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(uuid)
    time.sleep(0.15)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    mid = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        if g_main is not None:
            g_main.replay()
        mid.record(stream)
        g_ev.replay()
        end.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    value, ms_total_max = job_rate(start.elapsed_time(end), K, world, "cuda")
    s1 = cache.stats(0)
    misses = s1["misses"] - s0["misses"]
    hits = s1["hits"] - s0["hits"]
    picks = s1["picks"] - s0["picks"]
    assert s1["error_flags"] == 0, s1

    # per-kernel times over the instrumented graph (last G steps of the timed
    # region); per-step hit/miss counts from the cache's trace ring
    recs = cache.trace(0)[-G:]
    n_miss = np.array([r.n_miss for r in recs], np.float64)
    n_hit = k - n_miss
    ev_ms = np.array([[row[0].elapsed_time(row[i]) for i in range(8)] for row in evs])
    t_route = ev_ms[:, 1]
    t_rt = ev_ms[:, 3] - ev_ms[:, 2]        # missed picks: read-through pass (link + gate/up)
    t_dn_miss = ev_ms[:, 4] - ev_ms[:, 3]   # missed picks: down from their slots
    t_gu_hit = ev_ms[:, 5] - ev_ms[:, 1]    # resident picks: gate/up from HBM slots
    t_dn_hit = ev_ms[:, 6] - ev_ms[:, 5]    # resident picks: down (+ combine if last)
    gap_ms = sum(evs[t][7].elapsed_time(evs[t + 1][0]) for t in range(G - 1)) / max(G - 1, 1)
    timing_split = {"ms_per_step_plain_graph": start.elapsed_time(mid) / (K - G) if K > G else None,
                    "ms_per_step_event_graph": mid.elapsed_time(end) / G,
                    "ms_between_steps": gap_ms,
                    "ms_miss_path": float(np.mean(ev_ms[:, 4] - ev_ms[:, 1])),
                    "ms_hit_path": float(np.mean(ev_ms[:, 6] - ev_ms[:, 1])),
                    "ms_route": float(np.mean(t_route)),
                    "ms_step_with_miss": float(np.mean(ev_ms[n_miss > 0, 7])) if (n_miss > 0).any() else None,
                    "ms_step_no_miss": float(np.mean(ev_ms[n_miss == 0, 7])) if (n_miss == 0).any() else None,
                    "frac_steps_with_miss": float(np.mean(n_miss > 0)),
                    "no_miss_breakdown_ms": _breakdown(ev_ms[n_miss == 0]),
                    "with_miss_breakdown_ms": _breakdown(ev_ms[n_miss > 0])}

    # host-link bandwidth probed in the same session
    from hbm_slot_cache_gb300 import HostBank, moe_probe_host_link
    nb = 1 << 30
    hb = HostBank(nb)
    hb.array[::4096] = 1
    dst = torch.empty(nb, dtype=torch.uint8, device="cuda")
    link_sm = moe_probe_host_link(hb.ptr, dst.data_ptr(), nb, 0, 5)
    link_ce = moe_probe_host_link(hb.ptr, dst.data_ptr(), nb, 1, 5)
    del dst
    hb.close()
    link_peak = max(link_sm, link_ce)
    hbm_peak, hbm_src = _peaks()

    Bexp = banks.Bw + banks.Bs
    ms_step = ms_total_max / K
    miss_per_step = misses / K
    hbm_bytes = k * Bexp                       # expert bytes the kernels read per step
    link_bytes = miss_per_step * Bexp           # miss bytes over the host link per step
    t_roof_s = hbm_bytes / (hbm_peak * 1e9) + link_bytes / (link_peak * 1e9)
    path_frac = t_roof_s / (ms_step * 1e-3)
    # with the miss path overlapped and read through, a step is bound by the
    # larger of its hit bytes over HBM and its miss bytes over the host link
    t_max_s = float(np.mean(np.maximum(n_hit * Bexp / (hbm_peak * 1e9),
                                       n_miss * Bexp / (link_peak * 1e9))))

    # kernel rooflines: algorithmic bytes of the launch / its measured time,
    # summed over the instrumented steps
    gu_pick = 2 * cfg.inter * (H // 2 + H // 16)   # gate/up bytes of one pick
    dn_pick = H * (cfg.inter // 2 + cfg.inter // 16)
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
        "gemv_down[missed picks]": entry(float((n_miss * dn_pick).sum()), float(t_dn_miss[hm].sum()),
                                         hbm_peak, "hbm", nm),
        "route_remap": {"ms_per_launch": float(t_route.mean())},
    }
    for n in kern:
        if "resident" in n:
            kern[n]["traffic"] = _traffic(n.split("[")[0], float(n_hit.mean()))
        elif "missed" in n:
            kern[n]["traffic"] = _traffic(n.split("[")[0] + ("_missed" if "down" in n else ""),
                                          float(n_miss[hm].mean()) if hm.any() else 0.0)
            kern[n]["note"] = "steps with at least one miss"
    kern["gemv_readthrough[missed picks]"]["note"] += (
        "; whole missed experts over the host link, gate/up computed on the way in, "
        "written to their slots")
    kern["gemv_down[missed picks]"]["note"] += "; W2 rows read back from the slots just written"

    share = {n: v["ms_per_launch"] * (nm if "missed" in n else G) for n, v in kern.items()}
    dom = max(share, key=share.get)
    roofline = dict(kern[dom])
    roofline["kernel"] = dom
    roofline["peak_source"] = (hbm_src if roofline.get("bound") == "hbm"
                               else "moe_probe_host_link, same session (best of SM copy / cudaMemcpyAsync)")

    # end to end through the public API: moe_cache_step_host with pinned host
    # buffers (H2D of the step's logits and x, the step, D2H of its output,
    # every step inside the timed region)
    Ke = min(K, 1000)
    lg_h = torch.from_numpy(lgs[prewarm:prewarm + Ke].copy()).pin_memory()
    x_h = torch.from_numpy(xs[prewarm:prewarm + Ke].view(np.int16).copy()).pin_memory().view(torch.bfloat16)
    out_h = torch.empty((Ke, 1, H), dtype=torch.float32).pin_memory()
    with torch.cuda.stream(stream):  # untimed: the layer's eager step, then its graph capture
        for t in range(2):
            cache.step_host(0, lg_h[t], x_h[t], out_h[t], stream)
    stream.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the step's buffers exist before its call, as a caller's would
    bufs = [(lg_h[t], x_h[t], out_h[t]) for t in range(Ke)]
    se0 = cache.stats(0)
    with torch.cuda.stream(stream):
        e0.record(stream)
        h0 = time.perf_counter()
        for lg_t, x_t, out_t in bufs:
            cache.step_host(0, lg_t, x_t, out_t, stream)
        h1 = time.perf_counter()
        e1.record(stream)
    stream.synchronize()
    e2e_host_us = 1e6 * (h1 - h0) / Ke  # host time a call spends enqueueing (copies + step)
    e2e_miss = (cache.stats(0)["misses"] - se0["misses"]) / Ke
    e2e_value, _ = job_rate(e0.elapsed_time(e1), Ke, world, "cuda")

    # cold: the first steps from an empty ring (the same routing stream), one
    # graph, after the steady-state measurement
    n_cold = min(300, prewarm + W + K)
    cache.reset()
    g_cold = capture(0, n_cold)
    cache.reset()  # capture does not execute; start from empty
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        c0.record(stream)
        g_cold.replay()
        c1.record(stream)
    stream.synchronize()
    sc = cache.stats(0)
    cold = {"value": n_cold / (c0.elapsed_time(c1) * 1e-3), "unit": UNIT, "steps": n_cold,
            "misses_per_step": sc["misses"] / n_cold,
            "note": "steps 0..n from an empty ring, one CUDA graph (the value above is steady "
                    "state after a 64-step pre-warm)"}
    del g_cold

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_layer_steps(cfg, banks, seconds=12.0, max_steps=8)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "nvfp4 weights, fp32 accumulate", "data": "synthetic",
            "config": {"workload": "glm-layer M=1 S=128: hidden 6144, inter 2048, 256 experts, "
                                   "top-8, 128 HBM slots, Zipf(1.1) routing, steady state",
                       "global_batch": world, "seq_len": 1,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2: 170 MB of expert bytes per step > 126 MB L2; "
                             "2.7 GB slot ring", "graph": "CUDA graphs, eager prewarm of 64 steps"},
            "tok_s_equivalent": value / GLM_MOE_LAYERS,
            "path_roofline": {"frac": path_frac, "t_roofline_us": t_roof_s * 1e6,
                              "t_measured_us": ms_step * 1e3, "hbm_bytes_per_step": hbm_bytes,
                              "link_bytes_per_step": link_bytes, "hbm_peak_gbs": hbm_peak,
                              "hbm_peak_source": hbm_src, "link_peak_gbs": link_peak,
                              "link_probe_sm_gbs": link_sm, "link_probe_memcpy_gbs": link_ce,
                              "misses_per_step": miss_per_step,
                              "overlapped_bound": {
                                  "t_us": t_max_s * 1e6, "frac": t_max_s / (ms_step * 1e-3),
                                  "note": "mean over the traced steps of max(hit bytes / HBM "
                                          "peak, miss bytes / link peak)"},
                              "hit_rate": hits / picks if picks else None},
            "roofline": roofline, "kernels": kern, "timing_split": timing_split, "cold": cold,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "host_us_per_call": e2e_host_us,
                    "misses_per_step": e2e_miss,
                    "h2d_bytes_per_step": E * 4 + H * 2,
                    "d2h_bytes_per_step": H * 4, "steps": Ke},
            "gpu_launches": K * 5, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    cache.close()
    banks.close()
    if world > 1:
        dist.destroy_process_group()


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
    if K * L > 4096:
        raise SystemExit("--workload multirow/prefill: steps x layers must be <= 4096 (one graph)")
    T = W + K
    banks = Banks(cfg)
    prefill = args.workload == "prefill"
    cache = make_cache(cfg, banks, layers=L, trace_capacity=0 if prefill else T,
                       max_rows=max(M, 16))
    Bexp = banks.Bw + banks.Bs
    # inputs: per (step, layer) logits; activations per step, shared by the layers
    if prefill:
        lgs = np.stack([np.stack([workload.prefill_logits(cfg, l, M) for l in range(L)])] * T)
    else:
        rts = [workload.Routing(cfg, layer=l) for l in range(L)]
        lgs = np.stack([np.stack([rts[l].step() for l in range(L)]) for _ in range(T)])
    xs = workload.activations(cfg.seed, 0, T, M, H)
    lg_d = torch.from_numpy(lgs.astype(np.float32)).cuda()               # [T, L, M, E]
    x_d = torch.from_numpy(xs.view(np.int16)).cuda().view(torch.bfloat16)  # [T, M, H]
    out_d = torch.empty((M, H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def run(t0, t1):
        for t in range(t0, t1):
            for l in range(L):
                cache.step(l, lg_d[t, l], x_d[t], out_d)

    with torch.cuda.stream(stream):
        run(0, W)                                  # eager warm-up (fills the rings)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run(W, T)
    with torch.cuda.stream(stream):
        g.replay()                                 # upload; the rings move on, steady state
    stream.synchronize()
    s0 = cache.stats(-1)
    sampler = ClockSampler(None)
    time.sleep(0.15)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
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
                       "graph": "one CUDA graph over the timed steps"},
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
    ap.add_argument("--workload", default="glm", choices=["glm", "multirow", "prefill"],
                    help="glm: the one-row decode step (the headline line); multirow / "
                         "prefill: M=16 rounds or M=512 bypass, their own line")
    ap.add_argument("--layers", type=int, default=0, help="multirow/prefill: layers (0: config)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "glm":
        run_rows(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
