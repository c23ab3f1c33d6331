#!/usr/bin/env python3
"""Benchmark of the Q4_K MoE layer hot path on GB300 (prints one JSON line).

A step is one pass of the whole layer over one batch: pair bucketing, fused gate|up +
SwiGLU (routed experts and the shared expert), down projections, combine. Each step
uses the weights and inputs of a different layer out of a rotation whose touched bytes
far exceed the 129 MB L2, so no step reads weights the previous steps left in L2. The
K timed steps are one CUDA graph, timed with CUDA events on the launching stream. For a
layer that runs as one kernel (the decode layers) that kernel is the roofline's kernel and
the step time is its launch duration; for a two-launch layer the roofline's kernel is the
fused gate|up launch, timed in a second graph of K back-to-back launches.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun each rank runs an independent replica on its own GPU (weak scaling);
rank 0 prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_quantized_moe_q4k_gb300 import inputs  # noqa: E402
from bit_quantized_moe_q4k_gb300.workloads import HEADLINE, MIXTRAL_M_SWEEP, PREFILL, WORKLOADS, Workload  # noqa: E402

METRIC = "Q4_K MoE id-GEMV: achieved HBM GB/s (% of peak) and (token,expert) pairs/sec"
# What the kernels compute in: weights Q4_K as stored; activations fp32 in HBM, staged on chip
# per 32-element sub-block as 16-bit fixed point (X = rint(x * 32767 / max|x|)) for the integer
# dp4a dot products, or as fp16 hi + lo parts for the tcgen05 path; fp32 accumulation.
DTYPE = ("q4k weights x activations staged as int16 per 32-element sub-block (dp4a, exact int sums) "
         "or fp16 hi+lo (tcgen05); fp32 accumulate")
UNIT = "pairs/s"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--m", type=int, default=0, help="override the token count of the workload")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ceiling", action="store_true", help="skip the loads-only ceiling of the step's bytes")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--layers", type=int, default=0, help="size of the layer rotation (default: > 3x L2 touched)")
    ap.add_argument("--separate-inputs", action="store_true",
                    help="one allocation per layer for its activations, ids and weights instead of stacked tensors")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads' records (per_config) after the headline")
    ap.add_argument("--per-config-steps", type=int, default=10)
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the router, routed-step and weight-format records after the headline")
    ap.add_argument("--next-rows-only", action="store_true",
                    help="run only the router, routed-step and weight-format records (a profiling aid)")
    ap.add_argument("--mem-cap-gb", type=float, default=24.0,
                    help="device memory the next-row records may fill with rotated weights")
    return ap.parse_args()


def workload(args) -> Workload:
    W = WORKLOADS[args.workload]
    return W.with_m(args.m) if args.m else W


def slab_bytes(n, k):
    return n * (k // 256) * 144


# ---------------------------------------------------------------------------------------------
# byte accounting (algorithmic: touched weights once, activations and outputs once)

def layer_bytes(W: Workload, ids: np.ndarray) -> dict:
    U = len(set(int(e) for e in ids.reshape(-1)))
    P, m = W.pairs, W.m
    gu_w = U * 2 * slab_bytes(W.inter, W.hidden) + (2 * slab_bytes(W.shared_inter, W.hidden) if W.shared_inter else 0)
    gu_io = m * W.hidden * 4 + P * W.inter * 4 + m * W.shared_inter * 4 + P * 4
    dn_w = U * slab_bytes(W.hidden, W.inter) + (slab_bytes(W.hidden, W.shared_inter) if W.shared_inter else 0)
    dn_io = P * W.inter * 4 + m * W.shared_inter * 4 + P * W.hidden * 4 + (m * W.hidden * 4 if W.shared_inter else 0)
    cb_io = m * W.hidden * 4 * 2 + P * W.hidden * 4 + P * 4 + (m * W.hidden * 4 + m * 4 if W.shared_inter else 0)
    return {"gate_up": gu_w + gu_io, "down": dn_w + dn_io, "combine": cb_io,
            "layer": gu_w + dn_w + m * W.hidden * 4 * 3 + P * 8 + (m * 4 if W.shared_inter else 0),
            "experts_touched": U}


# ---------------------------------------------------------------------------------------------
# clocks sampled during the timed region

CLOCK_SOAK_S = 0.8


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="q4k_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample of the workload

def oracle_sample_layers(W: Workload, n_layers: int, seed_base: int):
    import oracle
    out = []
    for li in range(n_layers):
        seed = seed_base + li
        ids = inputs.make_ids(seed, W.ids, W.m, W.top_k, W.num_experts)
        used = sorted(set(ids.tolist()))
        remap = {e: i for i, e in enumerate(used)}
        cids = np.array([remap[int(e)] for e in ids], np.int32)
        q = lambda proj, e, n, k: oracle.quantize_rows(inputs.expert_weights(seed, proj, e, n, k))
        wg = np.concatenate([q("gate", e, W.inter, W.hidden) for e in used])
        wu = np.concatenate([q("up", e, W.inter, W.hidden) for e in used])
        wd = np.concatenate([q("down", e, W.hidden, W.inter) for e in used])
        shared = None
        if W.shared_inter:
            shared = (q("sgate", 0, W.shared_inter, W.hidden), q("sup", 0, W.shared_inter, W.hidden),
                      q("sdown", 0, W.hidden, W.shared_inter))
        x = inputs.normal(seed, "h_post", (W.m, W.hidden))
        hm = inputs.normal(seed, "h_mid", (W.m, W.hidden))
        rw = inputs.routing_weights(seed, W.m, W.top_k)
        gl = inputs.normal(seed, "shared_gate", (W.m,))
        out.append((wg, wu, wd, len(used), shared, cids, x, hm, rw, gl))
    return out


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_oracle(W: Workload, target_s: float) -> dict:
    """Time the oracle's whole layer on host cores; returns pairs/s and the sample."""
    import oracle
    threads = oracle.set_threads(os.cpu_count() or 1)
    layers = oracle_sample_layers(W, 2, 0x0C0FFEE)
    done, pairs, t_total = 0, 0, 0.0
    while t_total < target_s and done < 10000:
        wg, wu, wd, E, shared, ids, x, hm, rw, gl = layers[done % len(layers)]
        t0 = time.perf_counter()
        oracle.moe_layer(wg, wu, wd, E, shared, W.shared_inter, W.shared_mode, x, hm, ids, rw, gl, W.m, W.top_k,
                         W.hidden, W.inter)
        t_total += time.perf_counter() - t0
        done += 1
        pairs += W.pairs
    # the same on one core, a shorter sample
    oracle.set_threads(1)
    done1, t1 = 0, 0.0
    while t1 < min(3.0, target_s / 4) and done1 < 1000:
        wg, wu, wd, E, shared, ids, x, hm, rw, gl = layers[done1 % len(layers)]
        t0 = time.perf_counter()
        oracle.moe_layer(wg, wu, wd, E, shared, W.shared_inter, W.shared_mode, x, hm, ids, rw, gl, W.m, W.top_k,
                         W.hidden, W.inter)
        t1 += time.perf_counter() - t0
        done1 += 1
    oracle.set_threads(threads)
    return {"value": pairs / t_total, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{done} layer forwards of {W.name} (2 distinct layers' weights, touched experts only), "
                      f"{t_total:.1f} s of oracle time, OpenMP over output rows",
            "single_thread": {"value": done1 * W.pairs / t1, "unit": UNIT, "cores": 1,
                              "sample": f"{done1} layer forwards of the same layers, {t1:.1f} s on one thread"}}


# ---------------------------------------------------------------------------------------------
# GPU arm

def run_ours(args, W: Workload, rank: int, world: int, local_rank: int):
    import torch
    import bit_quantized_moe_q4k_gb300 as q4k

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    q4k.load()
    H, I, E, T, m, Is = W.hidden, W.inter, W.num_experts, W.top_k, W.m, W.shared_inter
    P = W.pairs
    # rotation of distinct layers: enough that the bytes touched between two uses of a
    # layer exceed 3x the L2, and at least 4 layers
    ids0 = inputs.make_ids(W.seed, W.ids, m, T, E)
    per_layer_touched = layer_bytes(W, ids0)["layer"]
    n_layers = int(min(64, max(4, -(-3 * L2_BYTES // per_layer_touched))))
    if args.layers:
        n_layers = args.layers
    slab_total = E * (2 * slab_bytes(I, H) + slab_bytes(H, I))
    while n_layers > 2 and n_layers * slab_total > 120e9:
        n_layers -= 1

    gen = torch.Generator(device=dev)
    chunk_rows = max(1, (64 << 20) // (4 * max(H, I)))

    def make_slab(seed, n_exp, n, k):
        out = torch.empty(n_exp * n * (k // 256) * 144, dtype=torch.uint8, device=dev)
        rows_total = n_exp * n
        r0 = 0
        gen.manual_seed(seed)
        while r0 < rows_total:
            r1 = min(rows_total, r0 + chunk_rows)
            x = torch.randn(r1 - r0, k, generator=gen, device=dev, dtype=torch.float32) * 0.02
            q4k.q4k_quantize_rows(x, r1 - r0, k, out[r0 * (k // 256) * 144:])
            r0 = r1
        return out

    layers = []
    for li in range(n_layers):
        seed = W.seed * 1000 + li + 7919 * rank
        L = {
            "wg": make_slab(seed * 8 + 1, E, I, H), "wu": make_slab(seed * 8 + 2, E, I, H),
            "wd": make_slab(seed * 8 + 3, E, H, I),
        }
        if Is:
            L["sg"] = make_slab(seed * 8 + 4, 1, Is, H)
            L["su"] = make_slab(seed * 8 + 5, 1, Is, H)
            L["sd"] = make_slab(seed * 8 + 6, 1, H, Is)
        else:
            L["sg"] = L["su"] = L["sd"] = None
        L["np"] = {"ids": inputs.make_ids(seed, W.ids, m, T, E), "x": inputs.normal(seed, "h_post", (m, H)),
                   "hm": inputs.normal(seed, "h_mid", (m, H)), "rw": inputs.routing_weights(seed, m, T),
                   "gl": inputs.normal(seed, "shared_gate", (m,))}
        L["ids_np"] = L["np"]["ids"]
        layers.append(L)
    # Per-layer activations, ids and routing weights: one stacked tensor per kind (as an
    # inference engine keeps them in a few reused buffers), each layer reading its own slice;
    # only the weights rotate through HBM. --separate-inputs gives each its own allocation.
    for key in layers[0]["np"]:
        if args.separate_inputs:
            for L in layers:
                L[key] = torch.from_numpy(L["np"][key]).to(dev)
        else:
            stacked = torch.from_numpy(np.stack([L["np"][key] for L in layers])).to(dev)
            for li, L in enumerate(layers):
                L[key] = stacked[li]
    torch.cuda.synchronize()

    act = torch.empty(P * I, dtype=torch.float32, device=dev)
    act_s = torch.empty(max(1, m * Is), dtype=torch.float32, device=dev)
    eout = torch.empty(P * H, dtype=torch.float32, device=dev)
    sout = torch.empty(m * H, dtype=torch.float32, device=dev)
    # Layers are chained as in a model: step i reads h_post from xy[i % 2] and writes its output
    # y to xy[(i + 1) % 2], which the next step reads (--separate-inputs: each layer's own x).
    xy = [layers[0]["x"].clone().reshape(-1), torch.empty(m * H, dtype=torch.float32, device=dev)]
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    ws_gu_bytes = q4k.q4k_moe_layer_half_workspace_size(m, T, H, Is, H)
    ws_dn_bytes = q4k.q4k_moe_layer_half_workspace_size(m, T, I, Is, Is)
    ws_gu = torch.empty(max(256, ws_gu_bytes), dtype=torch.uint8, device=dev)
    ws_dn = torch.empty(max(256, ws_dn_bytes), dtype=torch.uint8, device=dev)

    def x_of(L, i):
        return L["x"] if args.separate_inputs else xy[i % 2]

    def gate_up(L, i):
        q4k.q4k_moe_layer_gate_up(L["wg"], L["wu"], E, L["sg"], L["su"], Is, x_of(L, i), L["ids"], m, T, H, I, act,
                                  act_s if Is else None, ws_gu, ws_gu_bytes, flag, stream)

    layer_ws_bytes = q4k.q4k_moe_layer_workspace_size(m, T, E, H, I, Is)
    layer_ws = torch.empty(layer_ws_bytes, dtype=torch.uint8, device=dev)

    def step(L, i):
        # the public layer call: gate|up + SwiGLU (routed and shared) then down with the combine fused
        y = xy[(i + 1) % 2]
        q4k.q4k_moe_layer_forward(L["wg"], L["wu"], L["wd"], E, L["sg"], L["su"], L["sd"], Is, W.shared_mode,
                                  x_of(L, i), L["hm"], L["ids"], L["rw"], L["gl"], m, T, H, I, y, layer_ws,
                                  layer_ws_bytes, flag,
                                  stream)

    # eager warm-up (first launches set kernel attributes), then capture
    with torch.cuda.stream(stream):
        for i in range(max(1, min(args.warmup, n_layers))):
            step(layers[i % n_layers], i)
    stream.synchronize()
    assert int(flag.item()) == 0, f"device error flag raised: {int(flag.item())}"

    K, Wm = args.steps, args.warmup

    # the timed graph: K whole-layer steps; the kernel graph (two-launch layers): the dominant
    # kernel (fused gate|up, launched as in the step) over the same K layers back to back.
    # A single-launch layer's one kernel is the step: its duration comes from the timed graph.
    single = q4k.q4k_moe_layer_launch_count(m, T, E, H, I, Is) == 1
    path = q4k.q4k_moe_layer_path(m, T, E, H, I, Is)
    g_warm, g_timed, g_kernel = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_warm, stream=stream, capture_error_mode="thread_local"):
            for i in range(Wm):
                step(layers[i % n_layers], i)
        with torch.cuda.graph(g_timed, stream=stream, capture_error_mode="thread_local"):
            for i in range(K):
                step(layers[(Wm + i) % n_layers], Wm + i)
        if not single:
            with torch.cuda.graph(g_kernel, stream=stream, capture_error_mode="thread_local"):
                for i in range(K):
                    gate_up(layers[(Wm + i) % n_layers], Wm + i)
    stream.synchronize()

    dist = None
    if world > 1:
        import torch.distributed as dist
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g_warm.replay()
    stream.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    # The timed region lasts milliseconds, less than the sampler's 100 ms period, so the same
    # graph is replayed (untimed) for CLOCK_SOAK_S seconds right before it: the clock samples
    # are taken under this load, and the sampler keeps running through the timed region.
    soak, t_soak = 0, time.perf_counter()
    with torch.cuda.stream(stream):
        while time.perf_counter() - t_soak < CLOCK_SOAK_S and soak < 100000:
            g_timed.replay()
            stream.synchronize()
            soak += 1
    soak_s = time.perf_counter() - t_soak
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    with torch.cuda.stream(stream):
        g_timed.replay()
    ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    clk["window"] = (f"nvidia-smi every 100 ms over {soak} untimed replays of the timed graph "
                     f"({soak_s:.2f} s) and then the timed region")
    total_ms = ev0.elapsed_time(ev1)
    # dominant kernel alone, same layers, right after the timed region
    gu_ms = [total_ms / K]
    if not single:
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g_kernel.replay()  # warm
        k0.record(stream)
        with torch.cuda.stream(stream):
            g_kernel.replay()
        k1.record(stream)
        k1.synchronize()
        gu_ms = [k0.elapsed_time(k1) / K]
    assert int(flag.item()) == 0, f"device error flag raised: {int(flag.item())}"

    # algorithmic bytes per step (touched experts differ per layer)
    per = [layer_bytes(W, layers[(Wm + i) % n_layers]["ids_np"]) for i in range(K)]
    gu_bytes = float(np.mean([p["gate_up"] for p in per]))
    layer_b = float(np.mean([p["layer"] for p in per]))

    if dist:
        total_ms = max_over_ranks(total_ms, dev)

    # the loads-only ceiling of the same burst: the layer's algorithmic bytes streamed by a
    # kernel that only loads them (q4k_stream_ceiling), from windows of a buffer larger than
    # L2 taken in turn so every launch reads from HBM; K launches in a graph
    ceiling = None
    if not args.no_ceiling:
        burst = int(layer_b) // 4096 * 4096
        # (a burst of twice the L2 or more streams from HBM on its own)
        n_win = 1 if burst >= 2 * L2_BYTES else max(4, -(-3 * L2_BYTES // burst))
        big = torch.empty(burst * n_win, dtype=torch.uint8, device=dev)
        big.fill_(1)
        sink = torch.empty(q4k.q4k_stream_ceiling_sink_words(), dtype=torch.int32, device=dev)
        g_ceil = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(3):
                q4k.q4k_stream_ceiling(big[(i % n_win) * burst:], burst, sink, stream)
            with torch.cuda.graph(g_ceil, stream=stream, capture_error_mode="thread_local"):
                for i in range(K):
                    q4k.q4k_stream_ceiling(big[(i % n_win) * burst:], burst, sink, stream)
            g_ceil.replay()
        stream.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        with torch.cuda.stream(stream):
            g_ceil.replay()
        c1.record(stream)
        c1.synchronize()
        ceil_us = c0.elapsed_time(c1) / K * 1e3
        ceiling = {"kernel": "stream_ceiling_kernel (loads only, same bytes as one layer step)",
                   "bytes_per_launch": burst, "avg_launch_us": ceil_us,
                   "gbs": burst / (ceil_us * 1e-6) / 1e9}
        del big

    # end to end through the host-buffer C-ABI call: per step H2D inputs, the layer, D2H output
    e2e = None
    if not args.no_e2e:
        ws_bytes = (q4k.q4k_moe_layer_workspace_size(m, T, E, H, I, Is) + q4k.q4k_moe_layer_host_staging_size(m, T, H))
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        pinned = [{k: torch.from_numpy(v).pin_memory() for k, v in L["np"].items()} for L in layers]
        hy = torch.empty(m * H, dtype=torch.float32).pin_memory()

        def host_step(i):
            L, h = layers[i % n_layers], pinned[i % n_layers]
            q4k.q4k_moe_layer_forward_host(L["wg"], L["wu"], L["wd"], E, L["sg"], L["su"], L["sd"], Is, W.shared_mode,
                                           h["x"], h["hm"], h["ids"], h["rw"], h["gl"], m, T, H, I, hy, ws, ws_bytes,
                                           flag, stream)

        for i in range(max(3, min(Wm, 20))):
            host_step(i)
        stream.synchronize()

        def timed(run):
            if dist:
                dist.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            t0 = time.perf_counter()
            run()
            e1.record(stream)
            e1.synchronize()
            ms = max(e0.elapsed_time(e1), (time.perf_counter() - t0) * 1e3)
            return max_over_ranks(ms, dev) if dist else ms

        # the K calls as a decode loop with fixed buffers runs them: captured once in a CUDA
        # graph (every step still copies its inputs in and its output out), then replayed
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g_e2e, stream=stream, capture_error_mode="thread_local"):
                for i in range(K):
                    host_step(Wm + i)
        stream.synchronize()
        with torch.cuda.stream(stream):
            g_e2e.replay()  # warm
        stream.synchronize()

        def replay():
            with torch.cuda.stream(stream):
                g_e2e.replay()

        e2e_ms = timed(replay)
        eager_ms = timed(lambda: [host_step(Wm + i) for i in range(K)])
        e2e = {"value": P * K * world / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(m * H * 4 * 2 + P * 4 * 2 + m * 4),
               "d2h_bytes_per_step": int(m * H * 4),
               "ms_per_step": e2e_ms / K, "eager_ms_per_step": eager_ms / K,
               "api": "q4k_moe_layer_forward_host (host buffers, pinned): per step one launch gathers the inputs "
                      "from host memory into the workspace, the layer's launches run, the fused combine stores y "
                      "into host memory; K calls captured in one CUDA graph (eager_ms_per_step: the same K calls "
                      "issued one by one)"}

    # kernels per step: gate|up and down (+ prep and GEMM of the tensor-core path when a half uses it)
    launches_per_step = q4k.q4k_moe_layer_launch_count(m, T, E, H, I, Is)
    return {"ceiling": ceiling, "single": single, "path": path, "launches_per_step": launches_per_step, "total_ms": total_ms, "gu_ms": gu_ms, "gu_bytes": gu_bytes, "layer_bytes": layer_b, "clocks": clk,
            "n_layers": n_layers, "e2e": e2e, "per_layer_touched": per_layer_touched,
            "experts_touched": float(np.mean([p["experts_touched"] for p in per]))}


# The other workloads of the layer, measured after the headline in the same run (one record each).
PER_CONFIG = [("qwen3moe_h2048_i768_e128_t8_m16_zipf", 0), ("deepseekv3_h7168_i2048_e256_t8_m64", 0)] + \
    [("mixtral_h4096_i14336_e8_t2", m) for m in MIXTRAL_M_SWEEP] + list(PREFILL)


FLAG_NAMES = {6: "expert id out of range", 9: "size limit", 10: "a bounded wait gave up (timeout)"}


def flag_error(flag):
    """None, or what the device error flag of a secondary measurement says. A raised flag there
    is reported in that record (the other records and the headline line still print)."""
    v = int(flag.item())
    return None if v == 0 else f"device error flag {v}: {FLAG_NAMES.get(v, 'see q4kmoe.h')}"


def per_config_records(args, rank, world, local_rank, peak):
    import argparse
    import torch
    tensor_peak = measured_tensor_peak()
    global CLOCK_SOAK_S
    out = []
    soak = CLOCK_SOAK_S
    CLOCK_SOAK_S = 0.3
    try:
        for name, m in PER_CONFIG:
            W = WORKLOADS[name].with_m(m) if m else WORKLOADS[name]
            sub = argparse.Namespace(**vars(args))
            sub.steps, sub.warmup, sub.no_e2e, sub.no_ceiling, sub.layers = args.per_config_steps, 3, True, True, 0
            try:
                r = run_ours(sub, W, rank, world, local_rank)
            except AssertionError as e:  # this workload's device error flag: reported, not timed
                out.append({"workload": name if not m else f"{name.removesuffix('_m1')}_m{m}", "m": W.m,
                            "error": str(e)})
                torch.cuda.empty_cache()
                continue
            K = sub.steps
            step_ms = r["total_ms"] / K
            gu_ms = float(np.mean(r["gu_ms"]))
            kbytes = r["layer_bytes"] if r["single"] else r["gu_bytes"]
            flops = 2.0 * 3 * W.hidden * (W.pairs * W.inter + W.m * W.shared_inter)  # the layer's multiply-adds x 2
            out.append({
                "workload": name if not m else f"{name.removesuffix('_m1')}_m{m}", "m": W.m, "pairs": W.pairs,
                "layer_tflops": flops / (step_ms * 1e-3) / 1e12,
                "layer_tensor_frac": flops / (step_ms * 1e-3) / 1e12 / tensor_peak,
                "ms_per_step": step_ms, "pairs_per_s": W.pairs * K * max(1, world) / (r["total_ms"] / 1e3),
                "layer_bytes": r["layer_bytes"], "layer_hbm_gbs": r["layer_bytes"] / (step_ms * 1e-3) / 1e9,
                "layer_hbm_frac": r["layer_bytes"] / (step_ms * 1e-3) / 1e9 / peak,
                "experts_touched_per_step": r["experts_touched"], "launches_per_step": r["launches_per_step"],
                "roofline": {"kernel": "layer_wide_kernel / layer_kernel (one persistent launch)" if r["single"] else
                             "idgemv_kernel<fused gate|up+SwiGLU> (routed + shared)",
                             "bound": "hbm", "bytes_per_launch": kbytes, "avg_launch_us": gu_ms * 1e3,
                             "achieved": kbytes / (gu_ms * 1e-3) / 1e9, "peak": peak,
                             "frac": kbytes / (gu_ms * 1e-3) / 1e9 / peak, "unit": "GB/s"},
                "clocks": r["clocks"], "l2": f"rotating {r['n_layers']} layers ({r['per_layer_touched'] / 1e6:.0f} MB "
                                             f"touched per step)"})
            del r
            torch.cuda.empty_cache()
    finally:
        CLOCK_SOAK_S = soak
    return out


# ---------------------------------------------------------------------------------------------
# The rows after the layer: router, the routed decode step, other 4-bit weight formats

def time_graph(step, K, Wm, stream, local_rank, soak_s=0.3):
    """Eager warm-up, W steps then K steps captured in CUDA graphs; clocks sampled over an
    untimed soak of the K-step graph and the timed replay. Returns (ms per step, clocks)."""
    import torch
    for i in range(3):
        with torch.cuda.stream(stream):
            step(i)
    stream.synchronize()
    g_warm, g = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_warm, stream=stream, capture_error_mode="thread_local"):
            for i in range(Wm):
                step(i)
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(K):
                step(Wm + i)
    stream.synchronize()
    with torch.cuda.stream(stream):
        g_warm.replay()
    stream.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        while time.perf_counter() - t0 < soak_s:
            g.replay()
            stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        g.replay()
    e1.record(stream)
    e1.synchronize()
    clk = clocks.stop()
    return e0.elapsed_time(e1) / K, clk


def rotation(bytes_per_step, cap, bytes_per_copy):
    """Copies to rotate through so the bytes touched between two uses of one exceed 3x L2
    (at most `cap` bytes of copies)."""
    n = max(4, -(-3 * L2_BYTES // max(1, bytes_per_step)))
    return int(max(2, min(n, cap // max(1, bytes_per_copy))))


ROUTER_CONFIGS = [
    # (name, num_experts, hidden, top_k, scoring, n_group, topk_group, scale, m)
    ("qwen3moe_router_e128_h2048_t8_softmax", 128, 2048, 8, 0, 1, 1, 1.0, 1),
    ("qwen3moe_router_e128_h2048_t8_softmax", 128, 2048, 8, 0, 1, 1, 1.0, 16),
    ("deepseekv3_router_e256_h7168_t8_noaux_g8k4", 256, 7168, 8, 1, 8, 4, 2.5, 1),
    ("deepseekv3_router_e256_h7168_t8_noaux_g8k4", 256, 7168, 8, 1, 8, 4, 2.5, 64),
]


def cap_bytes(args, default_gb):
    return int(min(default_gb, args.mem_cap_gb) * (1 << 30))


def router_records(args, local_rank, peak):
    import torch
    import bit_quantized_moe_q4k_gb300 as q4k
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.Stream(device=dev)
    out = []
    for name, E, H, k, scoring, ng, tg, scale, m in ROUTER_CONFIGS:
        wbytes = E * H * 2
        n = rotation(wbytes, cap_bytes(args, 4), wbytes)
        gen = torch.Generator(device=dev)
        gen.manual_seed(E * 131 + H)
        wr = (torch.randn(n, E, H, generator=gen, device=dev) / H ** 0.5).to(torch.bfloat16).view(torch.int16)
        bias = (torch.rand(E, generator=gen, device=dev) - 0.5) * 0.1
        xs = torch.randn(16, m, H, generator=gen, device=dev)
        ids = torch.empty(m, k, dtype=torch.int32, device=dev)
        wt = torch.empty(m, k, dtype=torch.float32, device=dev)
        lg = torch.empty(m, E, dtype=torch.float32, device=dev)

        def step(i):
            q4k.q4k_moe_router(xs[i % 16], wr[i % n], bias if scoring else None, None, m, E, H, k, scoring, True,
                               scale, ng, tg, ids, wt, lg, None, stream)

        K = max(10, args.per_config_steps * 4)
        ms, clk = time_graph(step, K, 3, stream, local_rank)
        b = wbytes + m * H * 4 + m * k * 8
        out.append({"workload": f"{name}_m{m}", "kernel": "router_logits_kernel + router_topk_kernel (two launches, "
                                                            "programmatic dependent)",
                    "bound": "hbm", "bytes_per_launch": b, "avg_launch_us": ms * 1e3,
                    "achieved": b / (ms * 1e-3) / 1e9, "peak": peak, "frac": b / (ms * 1e-3) / 1e9 / peak,
                    "unit": "GB/s", "clocks": clk, "l2": f"rotating {n} router weight copies"})
        del wr, xs
        torch.cuda.empty_cache()
    return out


def routed_step_record(args, W: Workload, local_rank, peak, fused=True):
    """One decode MoE block per step, chained as in a model: the router (softmax top-k, plus
    the shared expert's gate logit) on h_post, the layer with the router's ids / weights /
    gate, the next layer's input RMSNorm on the layer's output, which is the next step's
    h_post. fused: one q4k_moe_layer_forward_routed call per step; else the three calls."""
    import torch
    import bit_quantized_moe_q4k_gb300 as q4k
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.Stream(device=dev)
    H, I, E, T, m, Is = W.hidden, W.inter, W.num_experts, W.top_k, W.m, W.shared_inter
    ids0 = inputs.make_ids(W.seed, "uniform", m, T, E)
    lb = layer_bytes(W, ids0)
    per_layer = lb["layer"] + E * H * 2 + H * 2 * 2
    slab_total = E * (2 * slab_bytes(I, H) + slab_bytes(H, I)) + (3 * slab_bytes(Is, H) if Is else 0)
    n = rotation(per_layer, cap_bytes(args, 40), slab_total)
    gen = torch.Generator(device=dev)

    def slab(seed, n_exp, rows, k):
        buf = torch.empty(n_exp * rows * (k // 256) * 144, dtype=torch.uint8, device=dev)
        gen.manual_seed(seed)
        step_rows = max(1, (64 << 20) // (4 * k))
        for r0 in range(0, n_exp * rows, step_rows):
            r1 = min(n_exp * rows, r0 + step_rows)
            x = torch.randn(r1 - r0, k, generator=gen, device=dev) * 0.02
            q4k.q4k_quantize_rows(x, r1 - r0, k, buf[r0 * (k // 256) * 144:])
        return buf

    layers = []
    for li in range(n):
        s = 50000 + li * 8
        L = {"wg": slab(s + 1, E, I, H), "wu": slab(s + 2, E, I, H), "wd": slab(s + 3, E, H, I)}
        L.update({"sg": slab(s + 4, 1, Is, H), "su": slab(s + 5, 1, Is, H), "sd": slab(s + 6, 1, H, Is)} if Is else
                 {"sg": None, "su": None, "sd": None})
        gen.manual_seed(s + 7)
        L["wr"] = (torch.randn(E, H, generator=gen, device=dev) / H ** 0.5).to(torch.bfloat16).view(torch.int16)
        L["wsg"] = (torch.randn(H, generator=gen, device=dev) / H ** 0.5).to(torch.bfloat16).view(torch.int16)
        L["wn"] = (1 + 0.1 * torch.randn(H, generator=gen, device=dev)).to(torch.bfloat16).view(torch.int16)
        L["hm"] = torch.randn(m, H, generator=gen, device=dev)
        layers.append(L)
    ids = torch.empty(m, T, dtype=torch.int32, device=dev)
    wt = torch.empty(m, T, dtype=torch.float32, device=dev)
    sgl = torch.empty(m, dtype=torch.float32, device=dev)
    lgt = torch.empty(m, E, dtype=torch.float32, device=dev)
    y = torch.empty(m, H, dtype=torch.float32, device=dev)
    xy = [torch.randn(m, H, generator=gen, device=dev), torch.empty(m, H, dtype=torch.float32, device=dev)]
    ws_bytes = (q4k.q4k_moe_layer_routed_workspace_size if fused else q4k.q4k_moe_layer_workspace_size)(
        m, T, E, H, I, Is)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(i):
        L = layers[i % n]
        x, xn = xy[i % 2], xy[(i + 1) % 2]
        if fused:
            q4k.q4k_moe_layer_forward_routed(L["wg"], L["wu"], L["wd"], E, L["sg"], L["su"], L["sd"], Is,
                                             W.shared_mode, x, L["hm"], L["wr"], None, L["wsg"] if Is else None,
                                             q4k.ROUTE_SOFTMAX, True, 1.0, 1, 1, m, T, H, I, y, L["wn"], 1e-6, xn,
                                             None, None, ws, ws_bytes, flag, stream)
            return
        q4k.q4k_moe_router(x, L["wr"], None, L["wsg"] if Is else None, m, E, H, T, q4k.ROUTE_SOFTMAX, True, 1.0, 1, 1,
                           ids, wt, lgt, sgl if Is else None, stream)
        q4k.q4k_moe_layer_forward(L["wg"], L["wu"], L["wd"], E, L["sg"], L["su"], L["sd"], Is, W.shared_mode, x,
                                  L["hm"], ids, wt, sgl if Is else None, m, T, H, I, y, ws, ws_bytes, flag, stream)
        q4k.q4k_rms_norm(y, L["wn"], m, H, 1e-6, xn, stream)

    K = max(10, args.per_config_steps * 4)
    ms, clk = time_graph(step, K, 3, stream, local_rank)
    err = flag_error(flag)
    b = per_layer + m * H * 4 * 2
    rec = {"workload": f"{W.name} + router + rms_norm" + (" (one call)" if fused else " (three calls)"),
           "ms_per_step": ms,
           "launches_per_step": 3 + q4k.q4k_moe_layer_launch_count(m, T, E, H, I, Is),
           "bytes_per_step": b, "hbm_gbs": b / (ms * 1e-3) / 1e9, "hbm_frac": b / (ms * 1e-3) / 1e9 / peak,
           "chain": ("q4k_moe_layer_forward_routed: the router's two kernels, the layer, the norm kernel, "
                     "in one call" if fused else
                     "router -> layer -> rms_norm on one stream, each a programmatic dependent of the one before") +
                    "; the norm's output is the next step's h_post", "clocks": clk,
           "l2": f"rotating {n} layers"}
    if err:
        rec["error"] = err
    del layers
    torch.cuda.empty_cache()
    return rec


FORMAT_CASES = [  # (format, affine group size); the Q4_K row is the same projection through the layer half
    ("q4k", 0), ("mlx_affine4_gs64", 64), ("q4tp", 0)]


def format_records(args, local_rank, peak):
    """Fused gate|up + SwiGLU of the Qwen3-like routed experts (128 experts, hidden 2048, width 768,
    top-8) in each 4-bit format, m = 1 and m = 16: the same walk, bucketing and staging, different
    block decoders and bytes per weight."""
    import torch
    import bit_quantized_moe_q4k_gb300 as q4k
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.Stream(device=dev)
    E, H, I, T = 128, 2048, 768, 8
    out = []
    for fmt, gs in FORMAT_CASES:
        if fmt == "q4k":
            mat = slab_bytes(I, H)
            stride = mat
        elif fmt == "q4tp":
            mat = I * H // 2 + 4 * I + I * (H // 32) * 5 // 8
            stride = -(-mat // 16) * 16
        else:
            mat = I * H // 2 + 4 * I * (H // gs)
            stride = -(-mat // 16) * 16
        for m in (1, 16):
            ids_np = [inputs.ids_uniform_distinct(60000 + j, m, T, E) for j in range(8)]
            U = np.mean([len(set(a.tolist())) for a in ids_np])
            per_step = U * 2 * mat + m * H * 4 + m * T * I * 4
            n = rotation(int(per_step), cap_bytes(args, 24), 2 * E * stride)
            gen = torch.Generator(device=dev)
            gen.manual_seed(70000 + m)
            slabs = [torch.randint(0, 256, (2, E * stride), dtype=torch.uint8, device=dev, generator=gen)
                     for _ in range(n)]
            if fmt != "q4k":  # sane scales: affine bf16 scale/bias ~ 0.01, q4tp base -7, step 0.1
                for sl in slabs:
                    v = sl.view(2, E, stride)
                    if fmt == "q4tp":
                        prm = torch.tensor([-7.0, 0.1], dtype=torch.float16, device=dev).view(torch.uint8)
                        v[:, :, I * H // 2: I * H // 2 + 4 * I] = prm.repeat(I)
                    else:
                        sc = torch.full((I * (H // gs),), 0.01, dtype=torch.bfloat16, device=dev).view(torch.uint8)
                        v[:, :, I * H // 2: I * H // 2 + 2 * I * (H // gs)] = sc
                        v[:, :, I * H // 2 + 2 * I * (H // gs): mat] = sc
            else:
                for sl in slabs:  # real Q4_K blocks
                    for j in range(2):
                        x = torch.randn(E * I, H, generator=gen, device=dev) * 0.02
                        q4k.q4k_quantize_rows(x, E * I, H, sl[j])
            ids = [torch.from_numpy(a).to(dev) for a in ids_np]
            xs = torch.randn(8, m, H, generator=gen, device=dev)
            act = torch.empty(m * T, I, dtype=torch.float32, device=dev)
            flag = torch.zeros(1, dtype=torch.int32, device=dev)
            ws_bytes = q4k.q4k_moe_layer_half_workspace_size(m, T, H, 0, H)
            ws = torch.empty(max(256, ws_bytes), dtype=torch.uint8, device=dev)

            def step(i):
                sl = slabs[i % n]
                if fmt == "q4k":
                    q4k.q4k_moe_layer_gate_up(sl[0], sl[1], E, None, None, 0, xs[i % 8], ids[i % 8], m, T, H, I, act,
                                              None, ws, ws_bytes, flag, stream)
                else:
                    q4k.q4k_moe_id_gemv_fmt(q4k.FMT_Q4TP if fmt == "q4tp" else q4k.FMT_AFFINE4, sl[0], sl[1], 0,
                                            stride, I * H // 2, I * H // 2 + 2 * I * (H // max(gs, 1)), max(gs, 32),
                                            E, xs[i % 8], H, 0, ids[i % 8], m, T, I, H, act, flag, stream)

            K = max(10, args.per_config_steps * 4)
            ms, clk = time_graph(step, K, 3, stream, local_rank)
            err = flag_error(flag)
            out.append({"workload": f"qwen3moe_gate_up_{fmt}_m{m}", "format": fmt,
                        "bytes_per_weight": mat / (I * H), "kernel": "idgemv_kernel<fused>" if fmt == "q4k" else
                        "fmt4_kernel<fused>", "bound": "hbm", "bytes_per_launch": per_step,
                        "avg_launch_us": ms * 1e3, "achieved": per_step / (ms * 1e-3) / 1e9, "peak": peak,
                        "frac": per_step / (ms * 1e-3) / 1e9 / peak, "unit": "GB/s", "clocks": clk,
                        "l2": f"rotating {n} slab pairs", **({"error": err} if err else {})})
            del slabs
            torch.cuda.empty_cache()
    return out


def measured_tensor_peak():
    """Dense bf16 TFLOP/s (cuBLAS, sustained when measured; the fp16 MMA rate is the same)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d.get("bf16_tflops_sustained") or d["bf16_tflops"])
    except (OSError, KeyError, ValueError, TypeError):
        return 1700.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


KERNEL_SOURCES = {  # the files whose text a kernel's counters depend on
    "idgemv_kernel<true>": ("q4k_gemv.cu", "q4k_gemv_common.cuh"),
    "layer_kernel": ("q4k_layer.cu", "q4k_gemv_common.cuh", "q4k_sync.cuh"),
    "layer_wide_kernel": ("q4k_layer.cu", "q4k_gemv_common.cuh", "q4k_sync.cuh"),
}


def code_text(text: str) -> str:
    """The source without blank lines and whole-line comments (code lines, trailing comments
    included, are kept): an edit of comments alone does not invalidate a capture."""
    return "\n".join(ln for ln in text.splitlines() if ln.strip() and not ln.strip().startswith("//"))


def source_sha(kernel: str, read=None) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        path = os.path.join("bit_quantized_moe_q4k_gb300", "csrc", name)
        if read is None:
            with open(os.path.join(ROOT, path)) as f:
                text = f.read()
        else:
            text = read(path)
        h.update(code_text(text).encode())
    return h.hexdigest()[:16]


def kernel_traffic(kernel: str, workload_name: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entries = json.load(f)
    except (OSError, ValueError):
        return None
    sha = source_sha(kernel)
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload_name and e.get("source_sha") == sha:
            return e.get("traffic_bytes_per_launch")
    return None


def main():
    args = parse()
    W = workload(args)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    config = {"workload": W.name, "hidden": W.hidden, "inter": W.inter, "num_experts": W.num_experts,
              "top_k": W.top_k, "m": W.m, "ids": W.ids, "shared_inter": W.shared_inter,
              "shared": ["none", "sigmoid", "unscaled"][W.shared_mode], "weights": "Q4_K from N(0,0.02)",
              "global_batch": W.m * max(1, world), "parallelism": f"replicas x{max(1, world)}"}

    if args.impl == "reference":
        if rank != 0:
            return
        cb = time_oracle(W, min(args.cpu_seconds, 20.0))
        per_step_ms = W.pairs / cb["value"] * 1e3
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step_ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": dict(config, l2="n/a (CPU oracle)"), "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line), flush=True)
        return

    if args.next_rows_only:
        peak, _ = measured_peaks()
        if rank == 0:
            print(json.dumps({"next_rows": {"router": router_records(args, local_rank, peak),
                                            "routed_step": routed_step_record(args, W, local_rank, peak),
                                            "formats": format_records(args, local_rank, peak)}}), flush=True)
        return
    r = run_ours(args, W, rank, world, local_rank)
    K = args.steps
    step_ms = r["total_ms"] / K
    value = W.pairs * K * max(1, world) / (r["total_ms"] / 1e3)
    peak, peak_kind = measured_peaks()
    gu_ms = float(np.mean(r["gu_ms"]))
    if r["single"]:
        # one kernel per step: the whole layer's bytes over its launch duration
        # the 256-thread kernel where each CTA takes at most one item of each half from tiles in
        # shared memory (the decode layer), else the 128-thread one (Q4K_LAYER_WIDE=0 forces it)
        kernel = "layer_wide_kernel" if r["path"] == 2 else "layer_kernel"  # Q4K_PATH_PERSISTENT_WIDE
        kbytes = r["layer_bytes"]
        kdesc = (f"{kernel} (gate|up+SwiGLU, down, combine; routed + shared) in one persistent launch")
        ktiming = ("CUDA events around the timed graph: K back-to-back launches of this kernel, one per step, "
                   "on the launching stream")
    else:
        kernel, kbytes = "idgemv_kernel<true>", r["gu_bytes"]
        kdesc = "idgemv_kernel<fused gate|up+SwiGLU> (routed + shared)"
        ktiming = ("CUDA events around a graph of K back-to-back launches of this kernel over the same rotating "
                   "layers, right after the timed region")
    achieved = kbytes / (gu_ms * 1e-3) / 1e9
    layer_gbs = r["layer_bytes"] / (step_ms * 1e-3) / 1e9
    per_config = None
    if not args.no_per_config and not args.m and args.workload == HEADLINE:
        per_config = per_config_records(args, rank, world, local_rank, peak)
    next_rows = None
    if not args.no_next_rows and not args.m and args.workload == HEADLINE:
        next_rows = {"router": router_records(args, local_rank, peak),
                     "routed_step": routed_step_record(args, W, local_rank, peak),
                     "formats": format_records(args, local_rank, peak)}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = time_oracle(W, args.cpu_seconds)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": max(1, world), "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE, "data": "synthetic",
        "config": dict(config, l2=f"rotating {r['n_layers']} layers' weights, "
                                  f"{r['per_layer_touched'] / 1e6:.1f} MB touched per step (> L2 between reuses)",
                    inputs="separate allocations per layer" if args.separate_inputs else
                    "layers chained (each step's h_post is the previous step's output); per-layer "
                    "h_mid/ids/routing weights as slices of stacked tensors"),
        "layer_hbm_gbs": layer_gbs, "layer_hbm_frac": layer_gbs / peak,
        "experts_touched_per_step": r["experts_touched"],
        "ceiling": r["ceiling"],
        "roofline": {"kernel": kdesc, "bound": "hbm",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "bytes_per_launch": kbytes, "avg_launch_us": gu_ms * 1e3,
                     "timing": ktiming, "traffic": kernel_traffic(kernel, W.name)},
        "cpu_baseline": cpu,
        "e2e": r["e2e"],
        "clocks": r["clocks"],
        "gpu_launches": r["launches_per_step"] * K,
        "per_config": per_config,
        "next_rows": next_rows,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
