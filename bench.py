"""Benchmark of the sink + short-window KV-cache hot path on one or more GPUs.

One step = one pass over every operation of the path for one layer of the
LongLive-1.3B-shaped workload (12 heads x 128, 4680-token chunks of 3 frames,
sink + 3-slot window = 18720 cached tokens):
    recache   [K|V] = Hid(18720x1536) @ W_kv(1536x3072), RMSNorm + 3D RoPE -> cache
    bf16      evict oldest chunk, append the new chunk, attention of its 4680 queries
    fp4       evict, append (FP4 encode), attention with fused dequantisation
Steps rotate over 8 independent layer caches, so every step touches > 126 MB
(larger than L2) that the previous step did not.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
With N > 1 launch under torchrun: every rank runs its own replica (weak scaling).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sink+window chunk-attn TFLOP/s & latent frames/s/layer; % of B300 bf16 peak"
H, D, TPF, CF, W = 12, 128, 1560, 3, 3
GRID_H, GRID_W = 30, 52
TC = TPF * CF            # 4680 query rows per chunk
LK = (1 + W) * TC        # 18720 visible keys at steady state
HD = H * D
ATTN_FLOP = 4.0 * H * TC * LK * D          # QK^T + PV, 538.27 GFLOP
RECACHE_FLOP = 2.0 * LK * HD * (2 * HD)    # 176.66 GFLOP
STEP_FLOP = 2 * ATTN_FLOP + RECACHE_FLOP
NLAYERS = 8
# algorithmic bytes per launch (read + write of the data the operation must touch)
APPEND_BF16_BYTES = 2 * 2 * TC * HD * 2                         # read K,V chunk + write cache
APPEND_FP4_BYTES = 2 * (TC * HD * 2 + TC * HD // 2 + TC * HD // 16)  # read bf16, write codes+scales
ATTN_BF16_BYTES = 2 * TC * HD * 2 + 2 * LK * HD * 2              # Q + O + K + V
ATTN_FP4_BYTES = 2 * TC * HD * 2 + 2 * LK * (HD // 2 + HD // 16)
RECACHE_BYTES = LK * HD * 2 + HD * 2 * HD * 2 + 2 * LK * HD * 2
WORKLOAD = ("LongLive-1.3B layer chunk step: 12 heads x 128, 4680 queries/chunk, "
            "18720 cached keys (1 sink chunk + 3 window slots), bf16 and FP4 caches, "
            "recache 18720x1536x3072")
# ncu dram bytes per launch of the dominant kernel, with the hash of the source
# they were taken on (null once the kernel changed)
TRAFFIC = {
    # ncu --set full on the LongLive-1.3B layer workload (one launch each);
    # summary in profiles/sinkwin_attn_layer1p3b_18720keys.md
    "sinkwin_attn_kernel<128,false>": {"bytes": 309258240 + 26184960, "src_sha": "e2953c2cbf9151d6"},
    "sinkwin_attn_kernel<128,true>": {"bytes": 48115200 + 4129024, "src_sha": "e2953c2cbf9151d6"},
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return (float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                float(d["hbm_gbs"]), "measured")
    except Exception:
        return 1800.0, 1400.0, 6400.0, "fallback"


def _src_sha(name):
    p = os.path.join(ROOT, "sink_short_window_sinkwin_b300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi every 10 ms with a timestamp; stop() keeps the samples that
    fall inside the timed window (all samples if none does, flagged)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.dev = dev_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "10", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self, t0: float | None = None, t1: float | None = None):
        """t0, t1: the timed window in time.time() seconds."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        from datetime import datetime
        rows = []
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 is not None and t0 <= r[0] <= t1]
        use = inside if inside else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = {n for r in use for n, v in zip(names, r[3]) if v.lower().startswith("active")}
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None, "reasons": sorted(reasons),
                "samples": len(use), "in_timed_window": bool(inside)}


# ---------------------------------------------------------------------------
# CPU baseline: the float64 oracle on a bounded sample of the same step
# ---------------------------------------------------------------------------
def cpu_sample(frac_rows: int, seed: int = 0):
    """Run the oracle on `frac_rows` query rows of both attentions, the same
    share of the recache rows and of the FP4 encode; returns (seconds, flop)."""
    import numpy as np
    from oracle import attention as oatt
    from oracle import fp4 as ofp4
    from oracle import recache as orc
    rng = np.random.default_rng(seed)
    f32 = np.float32
    k = (rng.standard_normal((LK, H, D), dtype=f32) / math.sqrt(D)).astype(np.float64)
    v = rng.standard_normal((LK, H, D), dtype=f32).astype(np.float64)
    q = (rng.standard_normal((frac_rows, H, D), dtype=f32) / math.sqrt(D)).astype(np.float64)
    hid = rng.standard_normal((4 * frac_rows, HD), dtype=f32).astype(np.float64)
    wkv = (rng.standard_normal((HD, 2 * HD), dtype=f32) * 0.02).astype(np.float64)
    kq = rng.standard_normal((frac_rows, H, D), dtype=f32)
    rows = np.arange(frac_rows)
    t0 = time.perf_counter()
    oatt.attention_rows(q, k, v, 1 / math.sqrt(D), rows)                     # bf16 row
    ofp4.quantize(kq), ofp4.quantize(kq)                                       # FP4 encode share
    oatt.attention_rows(q, k, v, 1 / math.sqrt(D), rows)                     # FP4 row (dequantised)
    kk, vv = orc.project(hid, wkv)                                            # recache share
    kk = orc.rmsnorm(kk, None, 1e-6).reshape(-1, H, D)
    t = np.arange(kk.shape[0]) % TC
    orc.rope3d(kk, t // TPF, (t % TPF) // GRID_W, t % GRID_W)
    dt = time.perf_counter() - t0
    frac = frac_rows / TC
    return dt, STEP_FLOP * frac


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return 1


def _cores():
    """Threads the oracle runs on: its matmuls use the BLAS pool, the einsum
    and elementwise parts one thread."""
    return min(len(os.sched_getaffinity(0)), _blas_threads())


def cpu_baseline(target_s: float = 12.0):
    dt, _ = cpu_sample(8)
    rows = int(max(8, min(TC, 8 * target_s / max(dt, 1e-3))))
    dt, flop = cpu_sample(rows, seed=1)
    return {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
            "host_cpus": len(os.sched_getaffinity(0)), "blas_threads": _blas_threads(),
            "sample": f"{rows} of 4680 query rows of both attentions (18720 keys, 12 heads), "
                      f"{4 * rows} of 18720 recache rows, FP4 encode of {rows} rows; "
                      f"{dt:.1f} s float64 numpy"}


def run_reference(args):
    """--impl reference: the oracle, as it stands, timed on the host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    dt, _ = cpu_sample(8)
    rows = int(max(8, min(TC, 8 * 4.0 / max(dt, 1e-3))))  # ~4 s per step
    for i in range(args.warmup):
        cpu_sample(rows, seed=100 + i)
    times, flop = [], 0.0
    for i in range(args.steps):
        dt, flop = cpu_sample(rows, seed=1000 + i)
        times.append(dt)
    mean = sum(times) / len(times)
    value = flop / mean / 1e12
    cores = _cores()
    sample = (f"{rows} of 4680 query rows of both attentions, {4 * rows} recache rows, "
              f"FP4 encode of {rows} rows per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# HBM-bound kernels, timed back to back
# ---------------------------------------------------------------------------
def hbm_kernels(swl, dev, layers, randn, per_graph: int = 8, replays: int = 6):
    """Per-launch time of the bandwidth kernels.  Each sequence is captured in
    a CUDA graph and replayed, CUDA events around the replays, so no host gap
    falls between launches; sources rotate over the layer inputs (> L2 in
    total).  bf16 append (copy) and FP4 append (encode): `per_graph`
    re-appends of the newest chunk.  Evict scrub: a graph of `per_graph`
    evicts with scrub, one per filled cache (> L2 in total)."""
    import torch
    srcs = [(L["k"], L["v"]) for L in layers]
    srcs4 = [(L["k4"], L["v4"]) for L in layers]
    while len(srcs) < 8:  # keep the rotating sources larger than L2
        srcs.append((randn((TC, H, D)), randn((TC, H, D))))
        srcs4.append((randn((TC, H, D), outliers=True), randn((TC, H, D), outliers=True)))
    stream = torch.cuda.Stream(device=dev)

    def timed(build):
        """us per replay of the graph `build` records"""
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            build()
        for _ in range(2):
            g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record()
            for _ in range(replays):
                g.replay()
            b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / replays

    def filled(dt, scrub=False):
        cache = swl.KVCache(H, D, TPF, CF, W, dtype=dt, device=dev, scrub_on_evict=scrub)
        src = srcs if dt == "bf16" else srcs4
        for c in range(1 + W):
            cache.append(*src[c % len(src)], c)
        torch.cuda.synchronize()
        return cache, src

    out = {}
    for name, dt, nbytes in (("append_bf16", "bf16", APPEND_BF16_BYTES),
                             ("append_fp4", "fp4", APPEND_FP4_BYTES)):
        cache, src = filled(dt)
        us = timed(lambda: [cache.append(*src[i % len(src)], W) for i in range(per_graph)])
        us /= per_graph
        out[name] = {"us": us, "bytes": nbytes, "gbs": nbytes / (us * 1e-6) / 1e9}

    for name, dt, nbytes in (("evict_scrub_bf16", "bf16", 2 * TC * HD * 2),
                             ("evict_scrub_fp4", "fp4", 2 * (TC * HD // 2 + TC * HD // 16))):
        # one filled cache per evict, so every captured evict is a legal call
        # (the oldest window chunk of its own cache) and launches one fill
        caches = [filled(dt, scrub=True)[0] for _ in range(per_graph)]
        us = timed(lambda: [c.evict(1) for c in caches]) / per_graph
        out[name] = {"us": us, "bytes": nbytes, "gbs": nbytes / (us * 1e-6) / 1e9}
        del caches
    return out


# ---------------------------------------------------------------------------
# Multi-rank bookkeeping (replicas: every rank runs the same step on its GPU)
# ---------------------------------------------------------------------------
def max_over_ranks(ms: float, dist, device) -> float:
    """The job's time for a weak-scaled step: the slowest rank's."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    return flop_per_rank_step * world / (ms_per_step * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=24)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=NLAYERS,
                    help="independent layer caches the steps rotate over (fewer: smaller "
                         "device footprint, e.g. for profiler captures)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import sink_short_window_sinkwin_b300 as swl

    dev = torch.device("cuda", local)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)

    def randn(shape, std=1.0, outliers=False):
        x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * std
        if outliers:
            m = torch.rand(shape, generator=gen, device=dev) < 0.01
            x = torch.where(m, x * 8.0, x)
        return x.to(torch.bfloat16)

    wkv = randn((HD, 2 * HD), 0.02)
    gamma = torch.ones(HD, dtype=torch.float32, device=dev)
    layers = []
    nlayers = max(1, args.layers)
    for li in range(nlayers):
        L = {
            "bf": swl.KVCache(H, D, TPF, CF, W, dtype="bf16", device=dev),
            "f4": swl.KVCache(H, D, TPF, CF, W, dtype="fp4", device=dev),
            "q": randn((TC, H, D), 1 / math.sqrt(D)),
            "k": randn((TC, H, D), 1 / math.sqrt(D)),
            "v": randn((TC, H, D)),
            "k4": randn((TC, H, D), outliers=True),
            "v4": randn((TC, H, D), outliers=True),
            "hid": randn((LK, HD)),
            "c": 0,
        }
        L["o"] = torch.empty_like(L["q"])
        L["o4"] = torch.empty_like(L["q"])
        for c in range(1 + W):  # sink + full window
            L["bf"].append(L["k"], L["v"], c)
            L["f4"].append(L["k4"], L["v4"], c)
        L["c"] = W
        layers.append(L)
    scale = 1.0 / math.sqrt(D)
    ROWS = ["recache", "evict_bf16", "append_bf16", "attn_bf16", "evict_fp4", "append_fp4", "attn_fp4"]

    def step(L, evs=None, wkv_t=None):
        c = L["c"] + 1
        present = [0] + list(range(c - W, c))
        w = wkv if wkv_t is None else wkv_t
        rec = (lambda: L["bf"].recache(L["hid"], w, gamma, present, GRID_H, GRID_W))
        ops = [rec,
               lambda: L["bf"].evict(c - W),
               lambda: L["bf"].append(L["k"], L["v"], c),
               lambda: L["bf"].attn(L["q"], scale, out=L["o"]),
               lambda: L["f4"].evict(c - W),
               lambda: L["f4"].append(L["k4"], L["v4"], c),
               lambda: L["f4"].attn(L["q"], scale, out=L["o4"])]
        if evs is not None:
            evs[0].record()
        for i, op in enumerate(ops):
            op()
            if evs is not None:
                evs[i + 1].record()
        L["c"] = c

    # recache (K GEMM, norm+RoPE, V GEMM), bf16 append copy, bf16 attention,
    # FP4 append (amax, encode), FP4 attention; evict without scrub launches nothing
    launches_per_step = 3 + 1 + 1 + 2 + 1

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ROWS) + 1)]
          for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else local)
    sampler.start()
    # Pre-warm for 0.3 s of wall time (the sampler's first readings fall in it):
    # the same step, so the host's launch path and the GPU are both in steady
    # state before the W warm-up steps.  A fresh process measured without it
    # showed host-side gaps (a launch-free evict taking 24 us instead of 2).
    prewarm, t_pw = 0, time.perf_counter()
    while time.perf_counter() - t_pw < 0.3:
        step(layers[prewarm % nlayers])
        prewarm += 1
        if prewarm % 8 == 0:
            torch.cuda.synchronize()  # keep the host within a few steps of the GPU
    torch.cuda.synchronize()
    # warm-up right before the timed steps: no idle gap in between
    for i in range(args.warmup):
        step(layers[(prewarm + i) % nlayers])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_epoch0 = time.time()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        step(layers[(prewarm + args.warmup + s) % nlayers], ev[s])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    t_epoch1 = time.time()
    if dist:
        dist.barrier()
    clocks = sampler.stop(t_epoch0, t_epoch1)

    row_ms = {r: 0.0 for r in ROWS}
    total_ms = 0.0
    for s in range(args.steps):
        total_ms += ev[s][0].elapsed_time(ev[s][-1])
        for i, r in enumerate(ROWS):
            row_ms[r] += ev[s][i].elapsed_time(ev[s][i + 1])
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    value = job_tflops(STEP_FLOP, world, ms_per_step)

    # ---- end to end through the public API with host buffers.  Every step's
    # inputs come from pinned host memory and its two attention outputs go back
    # to it, all inside the timed region; the copies run on their own streams so
    # that step s+1's inputs stream in (and step s-1's outputs stream out)
    # while step s computes, and the host reads step s-1's result meanwhile.
    host = {n: layers[0][n].cpu().pin_memory() for n in ("q", "k", "v", "k4", "v4", "hid")}
    host["wkv"] = wkv.cpu().pin_memory()
    out_h = [[torch.empty((TC, H, D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
             for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_h[0])
    n_e2e = max(3, min(args.steps, 10))
    for L in layers:  # per-layer weight buffer: a copy never races a recache reading it
        L["wkv"] = torch.empty_like(wkv)
    comp = torch.cuda.current_stream()
    cs, ds = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(n_e2e)]
    done = [torch.cuda.Event() for _ in range(n_e2e)]
    fetched = [torch.cuda.Event() for _ in range(n_e2e)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def enqueue_inputs(s):
        L = layers[s % nlayers]
        with torch.cuda.stream(cs):
            if s >= nlayers:  # the layer's buffers are free once step s - nlayers is done
                cs.wait_event(done[s - nlayers])
            for n in ("q", "k", "v", "k4", "v4", "hid", "wkv"):
                L[n].copy_(host[n], non_blocking=True)
            copied[s].record(cs)

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e_start.record(comp)
    cs.wait_event(e_start)
    enqueue_inputs(0)
    for s in range(n_e2e):
        L = layers[s % nlayers]
        if s + 1 < n_e2e:
            enqueue_inputs(s + 1)
        comp.wait_event(copied[s])
        if s >= nlayers:  # the layer's outputs of step s - nlayers have been read back
            comp.wait_event(fetched[s - nlayers])
        step(L, wkv_t=L["wkv"])
        done[s].record(comp)
        with torch.cuda.stream(ds):
            ds.wait_event(done[s])
            out_h[s % 2][0].copy_(L["o"], non_blocking=True)
            out_h[s % 2][1].copy_(L["o4"], non_blocking=True)
            fetched[s].record(ds)
        if s >= 1:
            fetched[s - 1].synchronize()  # the host reads step s-1's result
    fetched[n_e2e - 1].synchronize()
    comp.wait_event(fetched[n_e2e - 1])
    e_end.record(comp)
    torch.cuda.synchronize()
    e2e_ms = e_start.elapsed_time(e_end) / n_e2e
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = job_tflops(STEP_FLOP, world, e2e_ms)

    hbm = hbm_kernels(swl, dev, layers, randn)

    for L in layers:
        for cache in (L["bf"], L["f4"]):
            st = cache.last_device_error()
            if st != swl.KVC_OK:
                raise RuntimeError(f"device error after the bench: {swl.status_string(st)}")

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peak, peak_sus, hbm_peak, peak_src = _peaks()
    for r in hbm.values():
        r["frac_hbm_peak"] = r["gbs"] / hbm_peak
    steps = args.steps
    per = {r: row_ms[r] / steps for r in ROWS}
    flops = {"recache": RECACHE_FLOP, "attn_bf16": ATTN_FLOP, "attn_fp4": ATTN_FLOP}
    bytes_ = {"append_bf16": APPEND_BF16_BYTES, "append_fp4": APPEND_FP4_BYTES,
              "attn_bf16": ATTN_BF16_BYTES, "attn_fp4": ATTN_FP4_BYTES, "recache": RECACHE_BYTES}
    rows = {}
    for r in ROWS:
        d = {"ms": per[r], "share": per[r] / ms_per_step}
        if r in flops and per[r] > 0:
            d["tflops"] = flops[r] / (per[r] * 1e-3) / 1e12
            d["frac_bf16_peak"] = d["tflops"] / peak
        if r in bytes_ and per[r] > 0:
            d["gbs"] = bytes_[r] / (per[r] * 1e-3) / 1e9
            if r.startswith("append"):
                d["frac_hbm_peak"] = d["gbs"] / hbm_peak
        if r.startswith("attn") and per[r] > 0:
            d["latent_frames_per_s_per_layer"] = CF / (per[r] * 1e-3)
        rows[r] = d
    dom = max(("attn_bf16", "attn_fp4", "recache"), key=lambda r: per[r])
    kname = {"attn_bf16": "sinkwin_attn_kernel<128,false>", "attn_fp4": "sinkwin_attn_kernel<128,true>",
             "recache": "recache_gemm_kernel<256,*> x2 + recache_norm_rope_kernel"}[dom]
    src = {"attn_bf16": "kernels_attn.cu", "attn_fp4": "kernels_attn.cu",
           "recache": "kernels_recache.cu"}[dom]
    tr = TRAFFIC.get(kname)
    traffic = tr["bytes"] if tr and tr["src_sha"] == _src_sha(src) else None
    achieved = flops[dom] / (per[dom] * 1e-3) / 1e12
    chunk_step_ms = per["evict_bf16"] + per["append_bf16"] + per["attn_bf16"]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "step": "recache + (evict, append, attention) on a bf16 "
                   "cache + (evict, FP4 append, attention) on an FP4 cache",
                   "step_gflop": STEP_FLOP / 1e9, "layers_rotated": nlayers,
                   "l2": f"inputs larger than L2: {nlayers} rotating layer caches, each step "
                         "touches > 200 MB (the L2 holds 126 MB)",
                   "prewarm_steps": prewarm,
                   "parallelism": f"replicas x{world}"},
        "latent_frames_per_s_per_layer": CF / (chunk_step_ms * 1e-3),
        "rows": rows,
        "roofline": {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak,
                     "frac_sustained": achieved / peak_sus,
                     "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)",
                     "traffic": traffic},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "hbm_kernels": hbm,
        "gpu_launches": launches_per_step * steps,
        "clocks": clocks,
        "wall_s_timed": t_wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
