"""Benchmark of the sink + short-window KV-cache hot path on one or more GPUs.

The metric is the chunk attention of the LongLive-1.3B-shaped layer (12 heads
x 128, a 4680-query chunk of 3 frames against 18720 cached keys: 1 sink chunk +
3 window slots): TFLOP/s, latent frames/s per layer and % of the bf16 dense
peak.  It is measured inside one step of the whole path:
    recache   [K|V] = Hid(18720x1536) @ W_kv(1536x3072), RMSNorm + 3D RoPE -> cache
    bf16      evict oldest chunk, project the new chunk ([Q|K|V] = Hid(4680x1536) @
              W(1536x4608), Q/K RMSNorm + 3D RoPE, K/V straight into the ring slot),
              attention of its 4680 queries
    fp4       evict, append (FP4 encode), attention with fused dequantisation
Steps rotate over 8 independent layer caches, so every step touches > 126 MB
(larger than L2) that the previous step did not.  A second leg streams 30
layer caches x 320 chunks (evict + append + attention per layer and chunk) and
reports the steady-state latent frames/s per layer.

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
PROJECT_FLOP = 2.0 * TC * HD * (3 * HD)    # 66.25 GFLOP: one chunk's [Q|K|V] projection
STEP_FLOP = 2 * ATTN_FLOP + RECACHE_FLOP + PROJECT_FLOP
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
    # ncu dram__bytes_read.sum + dram__bytes_write.sum on the LongLive-1.3B
    # layer workload (one launch each); summary in
    # profiles/sinkwin_attn_layer1p3b_18720keys.md
    "sinkwin_attn_kernel<128,false>": {"bytes": 307172352 + 26303488, "src_sha": "c76cdafbd9a1ff12"},
    # the FP4 attention with a staging buffer, one call: the decode pass and
    # the kernel (the bench times the call)
    "fp4_to_f16_kernel + sinkwin_attn_kernel<128,true,true>": {
        "bytes": (32358656 + 52979712) + (312098560 + 26046720), "src_sha": "3ec9106f5bcd859f"},
    # the fused recache: the cluster launch and the cluster-free launch beside
    # it (captured one after the other); summary in profiles/recache_gemm_layer1p3b.md
    "recache_fused_kernel": {"bytes": (67131392 + 60844800) + (16364544 + 10752), "src_sha": "a496e9122d019fca"},
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


def _src_sha(names):
    """Hash of the kernel sources (one file name, or several joined by '+')."""
    h = hashlib.sha256()
    for name in names.split("+"):
        with open(os.path.join(ROOT, "sink_short_window_sinkwin_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


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
# CPU baseline: the float64 oracle on all host cores, on a sample of the
# metric's own workload (query rows of the LongLive-1.3B layer attention)
# ---------------------------------------------------------------------------
def cpu_attention_sample(rows: int, seed: int = 0):
    """The oracle's attention (oracle.pool: attention_rows on a spawn pool over
    every host core) for `rows` query rows x 12 heads against 18720 keys.
    Returns (seconds, flop, worker processes); the seconds include the pool's
    start-up (about a second)."""
    import numpy as np
    from oracle.pool import attention_rows_parallel, host_cores
    rng = np.random.default_rng(seed)
    f32 = np.float32
    k = (rng.standard_normal((LK, H, D), dtype=f32) / math.sqrt(D)).astype(np.float64)
    v = rng.standard_normal((LK, H, D), dtype=f32).astype(np.float64)
    q = (rng.standard_normal((rows, H, D), dtype=f32) / math.sqrt(D)).astype(np.float64)
    cores = host_cores()
    # one unit per (head, block of at most 1170 rows), at least as many units as cores
    per = max(1, min(rows, 1170, -(-rows * H // cores)))
    t0 = time.perf_counter()
    attention_rows_parallel(q, k, v, 1 / math.sqrt(D), rows_per_unit=per)
    dt = time.perf_counter() - t0
    return dt, 4.0 * H * rows * LK * D, min(cores, H * -(-rows // per))


def _sample_rows(target_s: float) -> int:
    dt, _, _ = cpu_attention_sample(120)
    return int(max(120, min(TC, 120 * target_s / max(dt, 1e-3))))


def cpu_baseline(target_s: float = 15.0):
    rows = _sample_rows(target_s / 2)
    dt, flop, cores = cpu_attention_sample(rows, seed=1)
    return {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "host_cpus": len(os.sched_getaffinity(0)), "blas_threads_per_worker": 1,
            "sample": f"{rows} of the 4680 query rows x 12 heads of the bf16 chunk attention "
                      f"against 18720 keys ({rows / TC:.1%} of one call), float64 numpy on "
                      f"{cores} spawned processes, {dt:.1f} s"}


def run_reference(args):
    """--impl reference: the oracle, as it stands, timed on the host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    rows = _sample_rows(6.0)  # ~6 s per step
    for i in range(args.warmup):
        cpu_attention_sample(rows, seed=100 + i)
    times, flop, cores = [], 0.0, 1
    for i in range(args.steps):
        dt, flop, cores = cpu_attention_sample(rows, seed=1000 + i)
        times.append(dt)
    mean = sum(times) / len(times)
    value = flop / mean / 1e12
    sample = (f"{rows} of the 4680 query rows x 12 heads of the bf16 chunk attention against "
              f"18720 keys per step, float64 numpy on {cores} spawned processes")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "latent_frames_per_s_per_layer": CF * (rows / TC) / mean,
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
# Further rows of the path, timed on their own (CUDA events, median of runs)
# ---------------------------------------------------------------------------
def extra_rows(swl, dev, randn, wkv, wqkv, gamma, runs: int = 12):
    """Split-KV attention of short query chunks (with and without the merge
    workspace), the recache into an FP4 cache, and the chunk projection into an
    FP4 cache.  Work rotates over two caches (> L2 together)."""
    import torch
    scale = 1.0 / math.sqrt(D)

    def med(fn):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(runs)]
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(evs):
            a.record()
            fn(i)
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    def filled(dt, **kw):
        c = swl.KVCache(H, D, TPF, CF, W, dtype=dt, device=dev, **kw)
        for ch in range(1 + W):
            c.append(randn((TC, H, D), 1 / math.sqrt(D)), randn((TC, H, D)), ch)
        return c

    out = {}
    caches = [filled("bf16") for _ in range(2)]
    whole = [filled("bf16", attn_workspace=False) for _ in range(2)]
    for tq in (128, 1560):
        q = randn((tq, H, D), 1 / math.sqrt(D))
        o = torch.empty_like(q)
        flop = 4.0 * H * tq * LK * D
        ms = med(lambda i: caches[i % 2].attn(q, scale, out=o))
        ms_whole = med(lambda i: whole[i % 2].attn(q, scale, out=o))
        out[f"split_kv_tq{tq}"] = {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12,
                                   "ms_whole_items": ms_whole, "speedup": ms_whole / ms,
                                   "what": f"bf16 attention, {tq} queries x 18720 keys x 12 heads; "
                                           "items spread over all SMs vs whole items per CTA"}
    del caches, whole
    # the FP4 attention without a staging buffer (K/V decoded inside the
    # kernel's tile load) next to the decode-once path the step uses
    q = randn((TC, H, D), 1 / math.sqrt(D))
    o = torch.empty_like(q)
    flop = 4.0 * H * TC * LK * D
    for name, st in (("attn_fp4_in_kernel_decode", False), ("attn_fp4_decode_once", True)):
        cs = [filled("fp4", stage=st) for _ in range(2)]
        ms = med(lambda i: cs[i % 2].attn(q, scale, out=o))
        out[name] = {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12,
                     "what": "FP4-KV attention, 4680 queries x 18720 keys x 12 heads, "
                             + ("K/V decoded in the kernel's tile load (no staging buffer)" if not st
                                else "visible K/V decoded once into the staging buffer, then "
                                     "f16 tiles by TMA")}
        for c in cs:
            if c.last_device_error() != swl.KVC_OK:
                raise RuntimeError("device error in the FP4 attention rows")
        del cs
    f4 = [filled("fp4", stage=True) for _ in range(2)]
    hid = randn((LK, HD))
    present = [0, 1, 2, 3]
    ms = med(lambda i: f4[i % 2].recache(hid, wkv, gamma, present, GRID_H, GRID_W))
    out["recache_fp4"] = {"ms": ms, "tflops": RECACHE_FLOP / (ms * 1e-3) / 1e12,
                          "what": "recache of 18720 rows into an FP4 cache: the fused projection "
                                  "launches into the staging buffer, then one FP4 encode of the "
                                  "four regions' K and V (8 tensors, two launches)"}
    hc = randn((TC, HD))
    qo = torch.empty((TC, H, D), dtype=torch.bfloat16, device=dev)
    ms = med(lambda i: f4[i % 2].project_append(hc, wqkv, None, gamma, W, GRID_H, GRID_W, q_out=qo))
    out["project_append_fp4"] = {"ms": ms, "tflops": PROJECT_FLOP / (ms * 1e-3) / 1e12,
                                 "what": "chunk [Q|K|V] projection with Q/K norm + RoPE, K/V "
                                         "FP4-encoded into the ring slot (re-append of the "
                                         "newest chunk)"}
    for c in f4:
        if c.last_device_error() != swl.KVC_OK:
            raise RuntimeError("device error in the extra rows")
    del f4
    # W4A4: the same chunk projection with FP4 activations and an FP4 weight
    # (one row per output feature), bf16 out; operands encoded once, outside
    # the timed region.  Each timed run is 8 calls back to back (the host's
    # tensor-map encoding per call then overlaps the GPU's work, as it does in
    # a stream of layers).
    a4 = swl.quant_fp4(hc.reshape(-1))
    b4 = swl.quant_fp4(wqkv.t().contiguous().reshape(-1))
    yo = torch.empty((TC, 3 * HD), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(swl.gemm_fp4_ws_bytes(TC, 3 * HD, HD), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    reps = 8
    for name, w4 in (("gemm_fp4_w4a4_fused", None), ("gemm_fp4_w4a4_two_phase", ws)):
        ms = med(lambda i: [swl.gemm_fp4(a4, b4, TC, 3 * HD, HD, out=yo, ws=w4, dev_err=err)
                            for _ in range(reps)]) / reps
        out[name] = {"ms": ms, "tflops": PROJECT_FLOP / (ms * 1e-3) / 1e12,
                     "what": "chunk [Q|K|V] projection in W4A4 (4680 x 1536 FP4 activations, "
                             "4608 x 1536 FP4 weight, bf16 out): "
                             + ("FP4 decoded to f16 tile by tile inside one tcgen05 GEMM"
                                if w4 is None else
                                "A and B decoded once to f16 in a workspace, then an f16 "
                                "tcgen05 GEMM")}
    if int(err.item()) != 0:
        raise RuntimeError("device error in the W4A4 projection")
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
    ap.add_argument("--no-rolling", action="store_true",
                    help="skip the 30-layer x 320-chunk rolling-stream leg")
    ap.add_argument("--prewarm-s", type=float, default=0.3,
                    help="seconds of pre-warm steps before the warm-up (0: none, e.g. for a "
                         "profiler's launch list)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the rows timed outside the step (split-KV, FP4 recache/projection)")
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
    wqkv = randn((HD, 3 * HD), 0.02)
    gamma = torch.ones(HD, dtype=torch.float32, device=dev)
    layers = []
    nlayers = max(1, args.layers)
    # one staging buffer shared by the layers' FP4 caches (their calls are
    # stream-ordered): the FP4 attention decodes the visible K/V into it
    stage4 = torch.empty(4 * TC * HD * 4, dtype=torch.uint8, device=dev)
    for li in range(nlayers):
        L = {
            "bf": swl.KVCache(H, D, TPF, CF, W, dtype="bf16", device=dev,
                              stage=2 * TC * HD * 4),  # the chunk projection's fp32 Q|K rows
            "f4": swl.KVCache(H, D, TPF, CF, W, dtype="fp4", device=dev, stage=stage4),
            "q": randn((TC, H, D), 1 / math.sqrt(D)),
            "k": randn((TC, H, D), 1 / math.sqrt(D)),
            "v": randn((TC, H, D)),
            "k4": randn((TC, H, D), outliers=True),
            "v4": randn((TC, H, D), outliers=True),
            "hid": randn((LK, HD)),
            "hc": randn((TC, HD)),  # hidden states of the new chunk
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
    ROWS = ["recache", "evict_bf16", "project_append_bf16", "attn_bf16", "evict_fp4", "append_fp4",
            "attn_fp4"]

    def step(L, evs=None, wkv_t=None):
        c = L["c"] + 1
        present = [0] + list(range(c - W, c))
        w = wkv if wkv_t is None else wkv_t
        rec = (lambda: L["bf"].recache(L["hid"], w, gamma, present, GRID_H, GRID_W))
        ops = [rec,
               lambda: L["bf"].evict(c - W),
               lambda: L["bf"].project_append(L["hc"], wqkv, None, gamma, c, GRID_H, GRID_W,
                                              q_out=L["q"]),
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

    # recache (the fused cluster launch and its cluster-free side launch),
    # chunk projection (GEMM, norm+RoPE), bf16 attention, FP4 append (amax,
    # encode), FP4 attention (K/V decode into the staging buffer, attention);
    # evict without scrub launches nothing
    launches_per_step = 2 + 2 + 1 + 2 + 2

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
    while time.perf_counter() - t_pw < args.prewarm_s:
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
    ms_per_step = max_over_ranks(total_ms / args.steps, dist, dev)
    # the metric: the bf16 chunk attention of the LongLive-1.3B layer, timed
    # inside each step (CUDA events on the launching stream around the call)
    attn_ms = max_over_ranks(row_ms["attn_bf16"] / args.steps, dist, dev)
    value = job_tflops(ATTN_FLOP, world, attn_ms)

    # ---- end to end through the public API with host buffers: the same chunk
    # attention, with every step's Q, K and V copied in from pinned host memory
    # (evict + append + attention on a bf16 cache) and its output copied back,
    # all inside the timed region.  The copies run on their own streams: step
    # s+1's inputs stream in and step s-1's output streams out while step s
    # computes, and the host reads step s-1's result meanwhile.  (The FP4
    # caches are not used after this point.)
    host = {n: layers[0][n].cpu().pin_memory() for n in ("q", "k", "v")}
    out_h = [torch.empty((TC, H, D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h[0].numel() * out_h[0].element_size()
    n_e2e = max(3, min(2 * args.steps, 24))
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
            for n in ("q", "k", "v"):
                L[n].copy_(host[n], non_blocking=True)
            copied[s].record(cs)

    def chunk_step(L):
        c = L["c"] + 1
        L["bf"].evict(c - W)
        L["bf"].append(L["k"], L["v"], c)
        L["bf"].attn(L["q"], scale, out=L["o"])
        L["c"] = c

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
        if s >= 2:  # the output buffer of step s - 2 has been read back
            comp.wait_event(fetched[s - 2])
        chunk_step(L)
        done[s].record(comp)
        with torch.cuda.stream(ds):
            ds.wait_event(done[s])
            out_h[s % 2].copy_(L["o"], non_blocking=True)
            fetched[s].record(ds)
        if s >= 1:
            fetched[s - 1].synchronize()  # the host reads step s-1's result
    fetched[n_e2e - 1].synchronize()
    comp.wait_event(fetched[n_e2e - 1])
    e_end.record(comp)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end) / n_e2e, dist, dev)
    e2e_value = job_tflops(ATTN_FLOP, world, e2e_ms)

    hbm = hbm_kernels(swl, dev, layers, randn)
    extra = None if args.no_extra else extra_rows(swl, dev, randn, wkv, wqkv, gamma)
    for L in layers:
        for cache in (L["bf"], L["f4"]):
            st = cache.last_device_error()
            if st != swl.KVC_OK:
                raise RuntimeError(f"device error after the bench: {swl.status_string(st)}")
    del layers, host
    torch.cuda.empty_cache()

    rolling = None if args.no_rolling else rolling_stream(swl, dev, rank, dist)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peak, peak_sus, hbm_peak, peak_src = _peaks()
    for r in hbm.values():
        r["frac_hbm_peak"] = r["gbs"] / hbm_peak
    steps = args.steps
    per = {r: row_ms[r] / steps for r in ROWS}
    flops = {"recache": RECACHE_FLOP, "attn_bf16": ATTN_FLOP, "attn_fp4": ATTN_FLOP,
             "project_append_bf16": PROJECT_FLOP}
    bytes_ = {"append_fp4": APPEND_FP4_BYTES,
              "attn_bf16": ATTN_BF16_BYTES, "attn_fp4": ATTN_FP4_BYTES, "recache": RECACHE_BYTES}
    rows = {}
    for r in ROWS:
        d = {"ms": per[r], "share": per[r] / (total_ms / steps)}
        if r in flops and per[r] > 0:
            d["tflops"] = flops[r] / (per[r] * 1e-3) / 1e12
            d["frac_bf16_peak"] = d["tflops"] / peak
            d["frac_bf16_peak_sustained"] = d["tflops"] / peak_sus
        if r in bytes_ and per[r] > 0:
            d["gbs"] = bytes_[r] / (per[r] * 1e-3) / 1e9
            if r.startswith("append"):
                d["frac_hbm_peak"] = d["gbs"] / hbm_peak
        if r.startswith("attn") and per[r] > 0:
            d["latent_frames_per_s_per_layer"] = CF / (per[r] * 1e-3)
        rows[r] = d
    dom = max(("attn_bf16", "attn_fp4", "recache"), key=lambda r: per[r])
    kname = {"attn_bf16": "sinkwin_attn_kernel<128,false>",
             "attn_fp4": "fp4_to_f16_kernel + sinkwin_attn_kernel<128,true,true>",
             "recache": "recache_fused_kernel"}[dom]
    src = {"attn_bf16": "kernels_attn.cu", "attn_fp4": "kernels_decode.cu+kernels_attn.cu",
           "recache": "kernels_recache.cu"}[dom]
    tr = TRAFFIC.get(kname)
    traffic = tr["bytes"] if tr and tr["src_sha"] == _src_sha(src) else None
    achieved = flops[dom] / (per[dom] * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "value": "bf16 chunk attention, 4680 queries x 18720 keys x 12 heads x 128 "
                            f"({ATTN_FLOP / 1e9:.2f} GFLOP per call), CUDA events around the call "
                            "inside each step, all ranks' calls over the slowest rank's time",
                   "step": "recache + (evict, [Q|K|V] projection appending K/V, attention) on a "
                           "bf16 cache + (evict, FP4 append, attention) on an FP4 cache",
                   "step_gflop": STEP_FLOP / 1e9, "layers_rotated": nlayers,
                   "l2": f"inputs larger than L2: {nlayers} rotating layer caches, each step "
                         "touches > 200 MB (the L2 holds 126 MB)",
                   "prewarm_steps": prewarm,
                   "parallelism": f"replicas x{world}"},
        "attn_ms": attn_ms,
        "attn_frac_bf16_peak": value / world / peak,
        "attn_frac_bf16_peak_sustained": value / world / peak_sus,
        "latent_frames_per_s_per_layer": CF / (attn_ms * 1e-3),
        "step_tflops": job_tflops(STEP_FLOP, world, ms_per_step),
        "rows": rows,
        "roofline": {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak,
                     "frac_sustained": achieved / peak_sus,
                     "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)",
                     "traffic": traffic},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": n_e2e,
                "what": "per step: Q, K, V of one chunk host->device, evict + append + "
                        "attention through the public API, O device->host"},
        "rolling": rolling,
        "hbm_kernels": hbm,
        "more_rows": extra,
        "gpu_launches": launches_per_step * steps,
        "clocks": clocks,
        "wall_s_timed": t_wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def rolling_stream(swl, dev, rank, dist, n_layers: int = 30, n_chunks: int = 320):
    """The rolling stream: n_layers independent bf16 layer caches, n_chunks
    chunks; for every chunk, every layer evicts its oldest window chunk (from
    chunk W + 1 on), appends the new chunk and runs its attention, the sink
    pinned.  Each chunk's Q/K/V for all layers are drawn on the device (seeded
    per chunk) before that chunk's timed region; CUDA events bracket the
    n_layers x (evict + append + attention) of a chunk.  Steady state: chunks
    >= 4 (the window full and evicting)."""
    import torch
    caches = [swl.KVCache(H, D, TPF, CF, W, dtype="bf16", device=dev) for _ in range(n_layers)]
    qkv = [[torch.empty((TC, H, D), dtype=torch.bfloat16, device=dev) for _ in range(3)]
           for _ in range(n_layers)]
    out = torch.empty((TC, H, D), dtype=torch.bfloat16, device=dev)
    g = torch.Generator(device=dev)
    scale = 1.0 / math.sqrt(D)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_chunks)]
    std = (1 / math.sqrt(D), 1 / math.sqrt(D), 1.0)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for c in range(n_chunks):
        g.manual_seed(100003 * (rank + 1) + c)
        for li in range(n_layers):
            for t, sd in zip(qkv[li], std):
                t.copy_(torch.randn((TC, H, D), generator=g, device=dev) * sd)
        evs[c][0].record()
        for li in range(n_layers):
            cache = caches[li]
            if c > W:
                cache.evict(c - W)
            cache.append(qkv[li][1], qkv[li][2], c)
            cache.attn(qkv[li][0], scale, out=out)
        evs[c][1].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    want = [0] + [-1] * W
    for x in range(max(1, n_chunks - W), n_chunks):  # the last W chunks, slot (x - 1) mod W
        want[1 + (x - 1) % W] = x
    for cache in caches:
        if cache.chunk_of_region != want:
            raise RuntimeError(f"rolling stream: slot map {cache.chunk_of_region}, want {want}")
        st = cache.last_device_error()
        if st != swl.KVC_OK:
            raise RuntimeError(f"device error in the rolling stream: {swl.status_string(st)}")
    steady = [a.elapsed_time(b) for a, b in evs[4:]]
    ms_chunk = max_over_ranks(sum(steady) / len(steady), dist, dev)
    ms_layer = ms_chunk / n_layers
    return {"layers": n_layers, "chunks": n_chunks, "steady_chunks": len(steady),
            "latent_frames": n_chunks * CF,
            "ms_per_layer_step": ms_layer,
            "latent_frames_per_s_per_layer": CF / (ms_layer * 1e-3),
            "latent_frames_per_s_all_layers": CF / (ms_chunk * 1e-3),
            "attn_tflops": ATTN_FLOP / (ms_layer * 1e-3) / 1e12,
            "wall_s": wall,
            "timing": "CUDA events around each chunk's 30 x (evict + append + attention), "
                      "chunks >= 4; wall_s includes drawing the inputs on the device"}


if __name__ == "__main__":
    main()
