#!/usr/bin/env python
"""Benchmark of the Flint-shape W4A16 (NVFP4) MoE decode layer on one GB300.

Metric: microseconds per MoE decode layer at batch 1 (lower is better), with
the achieved HBM bandwidth over the unique weight bytes the layer touches.
A step is one decode of one layer (router, sigmoid top-6, gate/up + SiLU*up,
down + combine, shared expert) for one batch of synthetic tokens. Steps rotate
through a pool of distinct seeded layers (47 by default, the MoE layer count
of the Flint stack), launched back to back on one stream with programmatic
dependent launch and replayed from a CUDA graph: each layer's weights are
touched once per rotation, 631 MB per rotation at batch 1 against a 129 MB
L2, so inputs are larger than L2.

One JSON line is printed by rank 0. --impl reference times the CPU oracle on
the same workload instead (a bounded sample per step).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FLINT = dict(hidden=2048, num_experts=256, top_k=6, inter=512, n_shared=1)
WORKLOAD = ("Flint-shape NVFP4 W4A16 MoE decode layer: hidden 2048, 256 experts, sigmoid top-6 renormalised "
            "+ 1 shared expert, intermediate 512, SwiGLU, bf16 router and activations")
METRIC = "us per MoE decode layer (batch 1) and achieved HBM GB/s"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--batch", type=int, default=1)
    p.add_argument("--layers", type=int, default=47)
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--quick", action="store_true", help="skip the batch-8, isolated, e2e, stack and CPU legs")
    p.add_argument("--stack-only", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--dense-only", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--bf16-only", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--prefill-only", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--prefill-batches", default="", help=argparse.SUPPRESS)
    p.add_argument("--prefill-layers", type=int, default=8, help=argparse.SUPPRESS)
    p.add_argument("--oracle-leg", type=int, default=0, help=argparse.SUPPRESS)
    p.add_argument("--ncu-case", default="", help="small case for ncu captures: a batch size (2 Flint-shape layers, "
                   "4 decodes, L2 flushed between them) or 'gemv' (one 2048 x 8192 NVFP4 GEMV, 4 calls)")
    return p.parse_args()


# --------------------------------------------------------------------------- CPU oracle leg

def oracle_leg(n_steps: int, batch: int, seed: int, budget_s: float) -> dict:
    """Times the oracle's decode of one Flint-shape layer, n_steps times (or
    fewer if the time budget runs out). Weights of the experts the routing
    selects are generated and quantised before timing starts."""
    import numpy as np  # noqa: F401

    import synth
    from oracle import moe, nvfp4
    d = FLINT
    cfg = moe.Config(**d)
    x = moe.bf16_bits_to_f64(synth.x_bf16(seed, 0, batch, d["hidden"]))
    router = moe.bf16_bits_to_f64(synth.router_bf16(seed, 0, d["num_experts"], d["hidden"]))
    routing = moe.route(x, router, cfg)
    cache = {}
    for e in sorted(set(routing.idx.ravel().tolist()) | {d["num_experts"] + s for s in range(d["n_shared"])}):
        mats = synth.expert_f32(seed, 0, e, d["hidden"], d["inter"])
        cache[e] = tuple(moe.NVFP4Matrix(*nvfp4.quantize(m)) for m in mats)
    times = []
    t_start = time.perf_counter()
    for _ in range(max(1, n_steps)):
        t0 = time.perf_counter()
        moe.moe_layer(x, router, cache.__getitem__, cfg)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > budget_s:
            break
    return {"us_per_layer": 1e6 * statistics.mean(times), "steps_timed": len(times),
            "seconds": time.perf_counter() - t_start}


def run_oracle_subprocess(n_steps: int, batch: int, seed: int, budget_s: float) -> dict:
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.oracle_leg(%d, %d, %d, %f)))" % (ROOT, n_steps, batch, seed, budget_s))
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT)
    if res.returncode != 0:
        raise RuntimeError("oracle leg failed: " + res.stderr[-2000:])
    return json.loads(res.stdout.strip().splitlines()[-1])


def reference_arm(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    budget = 150.0
    warm = run_oracle_subprocess(min(args.warmup, 1), args.batch, args.seed, budget)
    res = run_oracle_subprocess(args.steps, args.batch, args.seed, budget)
    sample = (f"oracle decode of one Flint-shape layer at batch {args.batch} per step (float64 numpy, 1 thread), "
              f"{res['steps_timed']} of {args.steps} requested steps timed within a {budget:.0f} s budget; "
              f"expert weights generated and quantised before timing")
    v = res["us_per_layer"]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us/layer", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1000.0, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": args.batch},
            "cpu_baseline": {"value": v, "unit": "us/layer", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "us/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "warmup_us": warm["us_per_layer"]}
    print(json.dumps(line))


# --------------------------------------------------------------------------- GPU arm

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed work runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peak_gbs() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def measured_peak_tflops() -> tuple[float, str]:
    """Dense bf16 tensor-core peak (cuBLAS burst, measured on this part)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def recorded_traffic(batch: int):
    """DRAM bytes per decode from the committed ncu summary, if it was taken on
    the current sources of the decode kernels (common.cuh, decode.cu; the
    summary records their hash)."""
    import hashlib
    csrc = os.path.join(ROOT, "w4a16_moe_decode_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("common.cuh", "decode.cu"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    digest = h.hexdigest()[:16]
    path = os.path.join(ROOT, "profiles", "traffic_b%d.txt" % batch)
    try:
        with open(path) as f:
            kv = dict(line.strip().split("=", 1) for line in f if "=" in line and not line.startswith("#"))
        if kv.get("csrc_sha256_16") == digest:
            return float(kv["dram_bytes_per_layer"])
    except (OSError, ValueError, KeyError):
        pass
    return None


# --------------------------------------------------------------------------- replicas (N GPUs)
# The layer has no exchange step and runs at TP = 1, so N GPUs run N independent
# replicas: rank r draws its own layers and tokens, every rank times the same
# number of steps, and the job's time is the slowest rank's.

def replica_seed(seed: int, rank: int) -> int:
    """Generator seed of rank `rank`'s layers and tokens."""
    return seed + 1000 * rank


def max_over_ranks(v: float, world: int, device) -> float:
    """The largest value of v over the ranks of the default process group."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_layer(ms_slowest: float, steps: int, world: int) -> float:
    """Whole-job time per decoded layer: world * steps layers in the slowest
    rank's time."""
    return ms_slowest * 1000.0 / steps / world


STACK_BIAS_FILE = os.path.join(ROOT, "tests", "golden", "flint_stack_bias.txt")


def stack_bias() -> tuple[float, int]:
    """(beta, number of biased experts) of the stack workload, as recorded by
    tests/golden/make_stack_bias.py."""
    import struct
    kv = {}
    with open(STACK_BIAS_FILE) as f:
        for line in f:
            if not line.startswith("#") and line.strip():
                k, v = line.split(None, 1)
                kv[k] = v.strip()
    beta = struct.unpack(">f", bytes.fromhex(kv["beta_f32_hex"]))[0]
    return beta, int(kv["biased_experts"])


def gpu_arm(args) -> None:
    import torch
    import torch.distributed as dist

    import synth  # noqa: F401  (the CPU generator is the definition the device one follows)
    from w4a16_moe_decode_gb300 import binding as fb
    from w4a16_moe_decode_gb300 import layers
    from w4a16_moe_decode_gb300.build import build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
    fb.lib()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def slowest(v: float) -> float:
        return max_over_ranks(v, world, dev)

    cfg = fb.make_config(**FLINT)
    P = args.layers

    def build_pool(B):
        pool = [layers.synth_layer(cfg, replica_seed(args.seed, rank), L, dev) for L in range(P)]
        xs = [layers.synth_x(B, cfg.hidden, replica_seed(args.seed, rank), L, dev) for L in range(P)]
        outs = [torch.empty_like(x) for x in xs]
        ws = layers.workspace(cfg, B, dev)
        return pool, xs, outs, ws

    def distinct_per_layer(pool, xs, outs, ws, B):
        idx = torch.empty(B, cfg.top_k, dtype=torch.int32, device=dev)
        w = torch.empty(B, cfg.top_k, dtype=torch.float32, device=dev)
        ds = []
        for L in range(P):
            fb.flint_moe_decode(pool[L].handle, xs[L], B, outs[L], ws)
            fb.flint_moe_debug_routing(cfg, ws, B, idx, w)
            ds.append(len(set(idx.cpu().numpy().ravel().tolist())))
        st, bits = fb.flint_moe_read_status(ws)
        if st != fb.OK or bits:
            raise RuntimeError(f"device status {bits} during setup")
        return ds

    def unique_bytes(D, B):
        per_matrix = cfg.inter * cfg.hidden // 2 + cfg.inter * cfg.hidden // 16 + 4
        return cfg.num_experts * cfg.hidden * 2 + (D + cfg.n_shared) * 3 * per_matrix + 2 * B * cfg.hidden * 2

    def timed_graph(pool, xs, outs, ws, B, steps, warmup, sample_clocks=False, min_ms=100.0):
        """Times regions of exactly `steps` decodes, each region bracketed by
        its own CUDA events on the launching stream, back to back until at
        least `min_ms` of regions (and at least 3) are timed; returns the
        slowest rank's median region time (ms), the number of regions and the
        clocks. A region is steps // P replays of the rotation graph (P layers)
        and one replay of a graph of the remaining steps. One untimed rotation
        is queued before the first region, so the device is busy while the host
        enqueues the regions: no event measures host launch latency."""
        stream = torch.cuda.Stream(device=dev)
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            for s in range(warmup):
                L = s % P
                fb.flint_moe_decode(pool[L].handle, xs[L], B, outs[L], ws, stream)
            cycle = torch.cuda.CUDAGraph()
            with torch.cuda.graph(cycle, stream=stream):
                for L in range(P):
                    fb.flint_moe_decode(pool[L].handle, xs[L], B, outs[L], ws, stream)
            rem = steps % P
            tail = None
            if rem:
                tail = torch.cuda.CUDAGraph()
                with torch.cuda.graph(tail, stream=stream):
                    for L in range(rem):
                        fb.flint_moe_decode(pool[L].handle, xs[L], B, outs[L], ws, stream)

            def region():
                for _ in range(steps // P):
                    cycle.replay()
                if tail is not None:
                    tail.replay()

            cycle.replay()
            region()
            stream.synchronize()
            clocks = None
            if sample_clocks:
                sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                                       else 0)
                sampler.start()
                t_end = time.time() + 1.5  # sustained load so the sampler sees the clocks under this work
                while time.time() < t_end:
                    for _ in range(50):
                        cycle.replay()
                    stream.synchronize()
            # the number of regions: enough for min_ms, from one timed region
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            cycle.replay()
            e0.record(stream)
            region()
            e1.record(stream)
            stream.synchronize()
            n_regions = max(3, min(100000, int(min_ms / max(e0.elapsed_time(e1), 1e-3)) + 1))
            barrier()
            events = [torch.cuda.Event(enable_timing=True) for _ in range(n_regions + 1)]
            cycle.replay()  # run-ahead: the device works while the regions are enqueued
            events[0].record(stream)
            for i in range(n_regions):
                region()
                events[i + 1].record(stream)
            stream.synchronize()
            barrier()
            if sample_clocks:
                clocks = sampler.stop()
        times = [events[i].elapsed_time(events[i + 1]) for i in range(n_regions)]
        st, bits = fb.flint_moe_read_status(ws, stream)
        if st != fb.OK or bits:
            raise RuntimeError(f"device status {bits} after the timed region")
        return slowest(statistics.median(times)), n_regions, clocks

    def isolated(pool, xs, outs, ws, B, reps=40):
        """One layer at a time with L2 flushed before each (256 MB write)."""
        flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream()
        times = []
        for r in range(reps):
            L = r % P
            flush.fill_(float(r))
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fb.flint_moe_decode(pool[L].handle, xs[L], B, outs[L], ws, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1000.0)
        return statistics.median(times)

    def e2e(pool, B, steps, mapped, min_ms=100.0):
        """Through the C ABI with host buffers: every step's x comes from pinned
        host memory and its out goes back to pinned host memory. With mapped,
        flint_moe_decode is given the pinned host buffers themselves: a staging
        kernel reads x across NVLink-C2C into the workspace and the down kernel
        writes out across it (the same bytes cross the link, with no
        copy-engine operation and no break in the programmatic-launch chain
        between steps); otherwise each step is a
        cudaMemcpyAsync of x, the decode on device buffers and a cudaMemcpyAsync
        of out. The steps of one rotation are captured once into a CUDA graph
        and replayed, as a serving loop would, so the number is not the Python
        launch overhead. Regions of whole rotations are timed back to back (one
        untimed rotation queued ahead), at least min_ms in all; the median
        region gives the time per step."""
        xh = [layers.synth_x(B, cfg.hidden, args.seed, L, dev).cpu().pin_memory() for L in range(P)]
        oh = [torch.empty(B, cfg.hidden, dtype=torch.int16).pin_memory() for _ in range(P)]
        xd = torch.empty(B, cfg.hidden, dtype=torch.int16, device=dev)
        od = torch.empty_like(xd)
        ws = layers.workspace(cfg, B, dev)
        stream = torch.cuda.Stream(device=dev)
        stream.wait_stream(torch.cuda.current_stream())
        # plain cudaMemcpyAsync (one per copy) from the runtime the library uses
        cudart = ctypes.CDLL("libcudart.so.13")
        cudart.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                           ctypes.c_void_p]
        nbytes = B * cfg.hidden * 2

        def memcpy(dst, src, kind):  # kind 1: host to device, 2: device to host
            if cudart.cudaMemcpyAsync(dst.data_ptr(), src.data_ptr(), nbytes, kind, stream.cuda_stream) != 0:
                raise RuntimeError("cudaMemcpyAsync failed")

        with torch.cuda.stream(stream):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for L in range(P):
                    if mapped:
                        fb.flint_moe_decode(pool[L].handle, xh[L], B, oh[L], ws, stream)
                    else:
                        memcpy(xd, xh[L], 1)
                        fb.flint_moe_decode(pool[L].handle, xd, B, od, ws, stream)
                        memcpy(oh[L], od, 2)
            for _ in range(3):
                g.replay()
            stream.synchronize()
            per_region = max(1, steps // P)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            g.replay()
            e0.record(stream)
            for _ in range(per_region):
                g.replay()
            e1.record(stream)
            stream.synchronize()
            n_regions = max(3, int(min_ms / max(e0.elapsed_time(e1), 1e-3)) + 1)
            barrier()
            events = [torch.cuda.Event(enable_timing=True) for _ in range(n_regions + 1)]
            g.replay()  # run-ahead
            events[0].record(stream)
            for i in range(n_regions):
                for _ in range(per_region):
                    g.replay()
                events[i + 1].record(stream)
            stream.synchronize()
        barrier()
        st, bits = fb.flint_moe_read_status(ws)
        if st != fb.OK or bits:
            raise RuntimeError(f"device status {bits} in the end-to-end leg")
        med = statistics.median(events[i].elapsed_time(events[i + 1]) for i in range(n_regions))
        return job_us_per_layer(slowest(med), per_region * P, world)

    def replay_times(g, stream, n):
        """Milliseconds of n back-to-back replays of graph g, each between its
        own events; one untimed replay is queued first so that the device is
        busy while the host enqueues the rest (no event sees launch latency)."""
        events = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        g.replay()
        events[0].record(stream)
        for i in range(n):
            g.replay()
            events[i + 1].record(stream)
        stream.synchronize()
        return [events[i].elapsed_time(events[i + 1]) for i in range(n)]

    def stack_leg(batches=(1, 2, 4, 8, 16, 32), passes=20):
        """The 47-layer stack: distinct layers (generator seed 1000 + L) as
        pre-norm sublayers of one residual stream, r_{L+1} = r_L +
        layer_L(rmsnorm_L(r_L)), routing skewed by a selection bias on experts
        0..25; per batch, the median over `passes` replays of the whole stack
        (one CUDA graph, PDL between all kernels)."""
        beta, nb = stack_bias()
        bias = torch.zeros(cfg.num_experts, dtype=torch.float32, device=dev)
        bias[:nb] = beta
        stack = [layers.synth_layer(cfg, 1000 + L, L, dev, bias=bias, norm_eps=layers.NORM_EPS) for L in range(P)]
        ws_s = layers.workspace(cfg, max(batches), dev)
        res = {}
        for Bs in batches:
            bufs = [layers.synth_x(Bs, cfg.hidden, 1000, 0, dev)] + \
                   [torch.empty(Bs, cfg.hidden, dtype=torch.int16, device=dev) for _ in range(P)]
            idx = torch.empty(Bs, cfg.top_k, dtype=torch.int32, device=dev)
            w = torch.empty(Bs, cfg.top_k, dtype=torch.float32, device=dev)
            dl, picks, biased = [], 0, 0
            for L in range(P):  # one eager pass: distinct experts and skew per layer
                fb.flint_moe_decode_prenorm(stack[L].handle, bufs[L], Bs, bufs[L + 1], ws_s)
                fb.flint_moe_debug_routing(cfg, ws_s, Bs, idx, w)
                ii = idx.cpu().numpy().ravel()
                dl.append(len(set(ii.tolist())))
                picks += ii.size
                biased += int((ii < nb).sum())
            st, bits = fb.flint_moe_read_status(ws_s)
            if st != fb.OK or bits:
                raise RuntimeError(f"device status {bits} in the stack")
            stream = torch.cuda.Stream(device=dev)
            stream.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(stream):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for L in range(P):
                        fb.flint_moe_decode_prenorm(stack[L].handle, bufs[L], Bs, bufs[L + 1], ws_s, stream)
                for _ in range(3):
                    g.replay()
                stream.synchronize()
                times = replay_times(g, stream, passes)
            us_layer = statistics.median(times) * 1000.0 / P
            ub = statistics.mean(unique_bytes(D, Bs) for D in dl)
            res[str(Bs)] = {"us_per_layer": us_layer, "gbs": ub / (us_layer * 1e-6) / 1e9,
                            "frac": ub / (us_layer * 1e-6) / 1e9 / measured_peak_gbs()[0],
                            "mean_distinct_experts": statistics.mean(dl), "unique_bytes_per_layer": ub,
                            "biased_pick_fraction": biased / picks, "passes": passes}
            if Bs >= 16:  # the same stack on the expert-grouped tensor-core path
                ws_p = layers.prefill_workspace(cfg, Bs, dev)
                with torch.cuda.stream(stream):
                    gp = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gp, stream=stream):
                        for L in range(P):
                            fb.flint_moe_prefill_prenorm(stack[L].handle, bufs[L], Bs, bufs[L + 1], ws_p, None,
                                                         stream)
                    for _ in range(3):
                        gp.replay()
                    stream.synchronize()
                    times = replay_times(gp, stream, passes)
                st, bits = fb.flint_moe_read_status(ws_p)
                if st != fb.OK or bits:
                    raise RuntimeError(f"device status {bits} in the stack (tensor-core path)")
                res[str(Bs)]["prefill_path_us_per_layer"] = statistics.median(times) * 1000.0 / P
                del gp, ws_p
            del bufs
        del stack, ws_s
        torch.cuda.empty_cache()
        return {"workload": f"{P} Flint-shape NVFP4 layers (generator seeds 1000 + L) chained as pre-norm sublayers "
                            f"of one residual stream (RMSNorm eps {layers.NORM_EPS:g} in the router and gate/up "
                            f"kernels, residual add in the down kernel), selection bias {beta:.6g} on experts "
                            f"0..{nb - 1}",
                "timing": f"median of {passes} replays of the whole stack (one CUDA graph), us per layer = "
                          f"stack time / {P}",
                "beta": beta, "per_batch": res}

    def dense_leg(shapes=((2048, 2048), (8192, 2048), (2048, 8192)), batches=(1, 8), steps=2000):
        """Small-batch dense GEMV y = x W^T on packed NVFP4 matrices, rotating
        through distinct seeded matrices (more bytes than L2 per rotation),
        launched back to back with programmatic dependent launch from a CUDA
        graph; GB/s over the matrix bytes."""
        res = {}
        peak = measured_peak_gbs()[0]
        for (N, K) in shapes:
            nbytes = fb.flint_gemv_packed_bytes(N, K, fb.NVFP4)
            nm = max(8, -(-384 * 1024 * 1024 // nbytes))  # at least 3x L2 per rotation
            mats = [layers.synth_dense(N, K, 2000 + i, 0, fb.NVFP4, dev)[0] for i in range(nm)]
            for Bd in batches:
                x = layers.synth_x(Bd, K, 2000, 0, dev)
                y = torch.empty(Bd, N, dtype=torch.int16, device=dev)
                stream = torch.cuda.Stream(device=dev)
                stream.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(stream):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        for m in mats:
                            fb.flint_gemv(m, N, K, fb.NVFP4, x, Bd, y, None, 0.0, None, stream)
                    for _ in range(3):
                        g.replay()
                    reps = max(1, steps // nm)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(reps):
                        g.replay()
                    e1.record(stream)
                    stream.synchronize()
                us = e0.elapsed_time(e1) * 1000.0 / (reps * nm)
                gbs = nbytes / (us * 1e-6) / 1e9
                res[f"{N}x{K}_b{Bd}"] = {"us": us, "gbs": gbs, "frac": gbs / peak, "matrix_bytes": nbytes,
                                         "matrices_in_rotation": nm}
            del mats
            torch.cuda.empty_cache()
        return {"workload": "y[B][N] = x[B][K] W^T, W NVFP4 [N][K] packed, bf16 x and y, FP32 accumulation",
                "per_shape": res}

    def bf16_leg(batches=(1, 8), n_layers=16, steps=2000):
        """The same layer with BF16 expert weights (no quantisation): a rotation
        of distinct seeded BF16 layers (45 MB touched per layer at batch 1, so
        each rotation is far larger than L2), CUDA graph, PDL."""
        cfg_b = fb.make_config(**FLINT, weight_fmt=fb.BF16)
        pool_b = [layers.synth_layer(cfg_b, args.seed, L, dev) for L in range(n_layers)]
        res = {}
        peak = measured_peak_gbs()[0]
        per_matrix = cfg_b.inter * cfg_b.hidden * 2
        for Bb in batches:
            xs_b = [layers.synth_x(Bb, cfg_b.hidden, args.seed, L, dev) for L in range(n_layers)]
            outs_b = [torch.empty_like(x) for x in xs_b]
            ws_b = layers.workspace(cfg_b, Bb, dev)
            idx = torch.empty(Bb, cfg_b.top_k, dtype=torch.int32, device=dev)
            w = torch.empty(Bb, cfg_b.top_k, dtype=torch.float32, device=dev)
            dl = []
            for L in range(n_layers):
                fb.flint_moe_decode(pool_b[L].handle, xs_b[L], Bb, outs_b[L], ws_b)
                fb.flint_moe_debug_routing(cfg_b, ws_b, Bb, idx, w)
                dl.append(len(set(idx.cpu().numpy().ravel().tolist())))
            stream = torch.cuda.Stream(device=dev)
            stream.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(stream):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for L in range(n_layers):
                        fb.flint_moe_decode(pool_b[L].handle, xs_b[L], Bb, outs_b[L], ws_b, stream)
                for _ in range(3):
                    g.replay()
                reps = max(1, steps // n_layers)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
                stream.synchronize()
            st, bits = fb.flint_moe_read_status(ws_b)
            if st != fb.OK or bits:
                raise RuntimeError(f"device status {bits} in the BF16 leg")
            us = e0.elapsed_time(e1) * 1000.0 / (reps * n_layers)
            ub = statistics.mean(cfg_b.num_experts * cfg_b.hidden * 2 + (D + cfg_b.n_shared) * 3 * per_matrix +
                                 2 * Bb * cfg_b.hidden * 2 for D in dl)
            res[str(Bb)] = {"us_per_layer": us, "gbs": ub / (us * 1e-6) / 1e9, "frac": ub / (us * 1e-6) / 1e9 / peak,
                            "mean_distinct_experts": statistics.mean(dl), "unique_bytes_per_layer": ub}
            del xs_b, outs_b, ws_b
        del pool_b
        torch.cuda.empty_cache()
        return {"workload": f"Flint-shape layer with BF16 expert weights, {n_layers} distinct layers rotated",
                "per_batch": res}

    def prefill_leg(batches=(16, 32, 64, 128, 256, 512, 1024, 4096), n_layers=8, max_calls=400):
        """The expert-grouped tensor-core path (flint_moe_prefill) on a rotation of
        distinct seeded Flint-shape layers (every layer's touched experts are
        read from HBM: 8 layers hold 3.6 GB), one CUDA graph per batch size;
        the decode path on the same layers beside it up to 32 tokens."""
        pool_p = [layers.synth_layer(cfg, args.seed, L, dev) for L in range(n_layers)]
        peak_tf, peak_tf_kind = measured_peak_tflops()
        peak = measured_peak_gbs()[0]
        res = {}
        for Bp in batches:
            xs_p = [layers.synth_x(Bp, cfg.hidden, args.seed, L, dev) for L in range(n_layers)]
            outs_p = [torch.empty_like(x) for x in xs_p]
            ws_p = layers.prefill_workspace(cfg, Bp, dev)
            idx = torch.empty(Bp, cfg.top_k, dtype=torch.int32, device=dev)
            w = torch.empty(Bp, cfg.top_k, dtype=torch.float32, device=dev)
            dl = []
            for L in range(n_layers):
                fb.flint_moe_prefill(pool_p[L].handle, xs_p[L], Bp, outs_p[L], ws_p)
                fb.flint_moe_prefill_debug_routing(cfg, ws_p, Bp, idx, w)
                dl.append(len(set(idx.cpu().numpy().ravel().tolist())))

            def time_graph(call):
                stream = torch.cuda.Stream(device=dev)
                stream.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(stream):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        for L in range(n_layers):
                            call(L, stream)
                    for _ in range(3):
                        g.replay()
                    reps = max(3, max_calls // n_layers if Bp <= 1024 else 64 // n_layers)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(reps):
                        g.replay()
                    e1.record(stream)
                    stream.synchronize()
                return e0.elapsed_time(e1) * 1000.0 / (reps * n_layers)

            us = time_graph(lambda L, st: fb.flint_moe_prefill(pool_p[L].handle, xs_p[L], Bp, outs_p[L], ws_p,
                                                               None, st))
            stt, bits = fb.flint_moe_read_status(ws_p)
            if stt != fb.OK or bits:
                raise RuntimeError(f"device status {bits} in the prefill leg")
            flops = 2.0 * Bp * cfg.num_experts * cfg.hidden + 6.0 * Bp * (cfg.top_k + cfg.n_shared) * cfg.hidden * \
                cfg.inter
            ub = statistics.mean(unique_bytes(D, Bp) for D in dl)
            tf = flops / (us * 1e-6) / 1e12
            r = {"us_per_layer": us, "tokens_per_s": Bp / (us * 1e-6), "tflops": tf, "tflops_frac": tf / peak_tf,
                 "gbs": ub / (us * 1e-6) / 1e9, "gbs_frac": ub / (us * 1e-6) / 1e9 / peak,
                 "mean_distinct_experts": statistics.mean(dl), "unique_bytes_per_layer": ub,
                 "flops_per_layer": flops}
            if Bp <= 32:
                ws_d = layers.workspace(cfg, Bp, dev)
                r["decode_path_us_per_layer"] = time_graph(
                    lambda L, st: fb.flint_moe_decode(pool_p[L].handle, xs_p[L], Bp, outs_p[L], ws_d, st))
                del ws_d
            res[str(Bp)] = r
            del xs_p, outs_p, ws_p
            torch.cuda.empty_cache()
        del pool_p
        torch.cuda.empty_cache()
        return {"workload": f"Flint-shape NVFP4 layer, {n_layers} distinct layers rotated, B tokens per call",
                "tflops_peak": peak_tf, "tflops_peak_kind": peak_tf_kind,
                "flops": "2 B E H (router) + 6 B (k + S) H I (gate, up, down)", "per_batch": res}

    if args.prefill_only:
        if rank == 0:
            kw = {"n_layers": args.prefill_layers}
            if args.prefill_batches:
                kw["batches"] = tuple(int(b) for b in args.prefill_batches.split(","))
            print(json.dumps({"prefill": prefill_leg(**kw)}))
        return
    if args.stack_only:
        if rank == 0:
            print(json.dumps({"stack": stack_leg()}))
        return
    if args.bf16_only:
        if rank == 0:
            print(json.dumps({"bf16_experts": bf16_leg()}))
        return
    if args.dense_only:
        if rank == 0:
            print(json.dumps({"dense_gemv": dense_leg()}))
        return

    K, W, B = args.steps, max(args.warmup, 3), args.batch
    pool, xs, outs, ws = build_pool(B)
    ds = distinct_per_layer(pool, xs, outs, ws, B)
    bytes_per_step = statistics.mean(unique_bytes(D, B) for D in ds)
    ms, n_regions, clocks = timed_graph(pool, xs, outs, ws, B, K, W, sample_clocks=True)
    us = job_us_per_layer(ms, K, world)
    us_rank = ms * 1000.0 / K
    gbs = bytes_per_step / (us_rank * 1e-6) / 1e9
    peak, peak_kind = measured_peak_gbs()
    legs, tail_legs = {}, {}
    if not args.quick:
        legs["isolated_l2_flushed_us"] = isolated(pool, xs, outs, ws, B)
        e2e_us = e2e(pool, B, min(K, 4000), mapped=True)
        legs["e2e_copy_engine_us"] = e2e(pool, B, min(K, 4000), mapped=False)
    else:
        e2e_us = None
    del pool, xs, outs, ws
    torch.cuda.empty_cache()
    if not args.quick and B == 1:
        pool8, xs8, outs8, ws8 = build_pool(8)
        ds8 = distinct_per_layer(pool8, xs8, outs8, ws8, 8)
        b8 = statistics.mean(unique_bytes(D, 8) for D in ds8)
        ms8, n8, _ = timed_graph(pool8, xs8, outs8, ws8, 8, K, W)
        us8 = ms8 * 1000.0 / K
        tail_legs["batch8"] = {"us_per_layer": us8, "gbs": b8 / (us8 * 1e-6) / 1e9,
                               "frac": b8 / (us8 * 1e-6) / 1e9 / peak, "mean_distinct_experts": statistics.mean(ds8),
                               "unique_bytes_per_layer": b8, "regions": n8,
                               "isolated_l2_flushed_us": isolated(pool8, xs8, outs8, ws8, 8)}
        del pool8, xs8, outs8, ws8
        torch.cuda.empty_cache()
    if not args.quick and B == 1 and world == 1:
        legs["prefill"] = prefill_leg()
        legs["dense_gemv"] = dense_leg()
        legs["bf16_experts"] = bf16_leg()
        legs["stack"] = stack_leg()
        tail_legs["stack_us_per_layer"] = {b: v["us_per_layer"] for b, v in legs["stack"]["per_batch"].items()}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.quick and world == 1:
        try:
            r = run_oracle_subprocess(30, B, args.seed, 25.0)
            cpu = {"value": r["us_per_layer"], "unit": "us/layer", "cores": 1, "kind": "oracle",
                   "sample": f"{r['steps_timed']} oracle decodes of one Flint-shape layer at batch {B} "
                             f"(float64 numpy, 1 thread, {r['seconds']:.1f} s); weights of the selected experts "
                             f"generated before timing"}
        except Exception as exc:  # the GPU number stands without the CPU leg
            cpu = {"value": None, "unit": "us/layer", "cores": 1, "kind": "oracle", "sample": f"failed: {exc}"}
    line = {
        "metric": METRIC, "value": us, "unit": "us/layer", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": us_rank / 1000.0, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4 x bf16 -> f16 tensor-core products, f32 accumulate", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": B, "layers_in_rotation": P,
                   "l2": f"inputs larger than L2: {P} distinct layers rotated, "
                         f"{P * bytes_per_step / 1e6:.0f} MB touched per rotation",
                   "launch": "3 kernels per layer, programmatic dependent launch, CUDA graph replay",
                   "timing": f"median over {n_regions} back-to-back regions of exactly {K} steps, each between "
                             f"its own CUDA events (at least 100 ms timed in all)"},
        "gbs": gbs,
        "unique_bytes_per_layer": bytes_per_step,
        "mean_distinct_experts": statistics.mean(ds),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_kind": peak_kind, "kernel": "flint_moe_decode (k_router + k_gateup + k_down)",
                     "traffic": recorded_traffic(B)},
        "clocks": clocks,
        "e2e": None if e2e_us is None else {"value": e2e_us, "unit": "us/layer",
                                            "h2d_bytes_per_step": B * cfg.hidden * 2,
                                            "d2h_bytes_per_step": B * cfg.hidden * 2,
                                            "transfer": "x and out in pinned host memory: x read once over "
                                                        "NVLink-C2C into the workspace by a staging kernel, out "
                                                        "written over the link by the down kernel (no copy-engine "
                                                        "operation); the copy-engine variant is e2e_copy_engine_us"},
        "gpu_launches": 3 * K * n_regions,
        "cpu_baseline": cpu,
    }
    line.update(legs)
    line.update(tail_legs)  # last, so that a reader of the line's tail sees batch 8 and the stack
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def ncu_case(args) -> None:
    """A few launches on a small device footprint (about 1 GB), for --set full
    ncu captures of one kernel: 2 Flint-shape layers decoded alternately at
    batch B, or one 2048 x 8192 NVFP4 GEMV at batch 1; a 256 MB write flushes
    L2 before every call."""
    import torch
    from w4a16_moe_decode_gb300 import binding as fb
    from w4a16_moe_decode_gb300 import layers
    from w4a16_moe_decode_gb300.build import build
    build()
    dev = torch.device("cuda", 0)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    if args.ncu_case == "gemv":
        N, K = 2048, 8192
        packed, _ = layers.synth_dense(N, K, 2000, 0, fb.NVFP4, dev)
        x = layers.synth_x(1, K, 2000, 0, dev)
        y = torch.empty(1, N, dtype=torch.int16, device=dev)
        for i in range(4):
            flush.fill_(float(i))
            fb.flint_gemv(packed, N, K, fb.NVFP4, x, 1, y)
        torch.cuda.synchronize()
        return
    B = int(args.ncu_case)
    cfg = fb.make_config(**FLINT)
    pool = [layers.synth_layer(cfg, args.seed, L, dev) for L in range(2)]
    xs = [layers.synth_x(B, cfg.hidden, args.seed, L, dev) for L in range(2)]
    outs = [torch.empty_like(x) for x in xs]
    ws = layers.workspace(cfg, B, dev)
    for i in range(4):
        flush.fill_(float(i))
        fb.flint_moe_decode(pool[i % 2].handle, xs[i % 2], B, outs[i % 2], ws)
    torch.cuda.synchronize()
    st, bits = fb.flint_moe_read_status(ws)
    if st != fb.OK or bits:
        raise RuntimeError(f"device status {bits}")


def main():
    args = parse_args()
    if args.ncu_case:
        ncu_case(args)
        return
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
