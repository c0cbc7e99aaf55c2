#!/usr/bin/env python3
"""Benchmark of the latent routed-expert MXFP4 MoE layer on GB300.

One step = one k3moe_forward over one batch of synthetic tokens (router,
permutation, expert FFNs, combine).  Default workload: the K3 decode shape
(T = 1 token, 896 experts, top-16, latent 3584, expert hidden 3072, 15.7 GB
of MXFP4 expert weights resident in HBM).

Cold caches: every step uses a different token batch from a pool, so each
step routes to a fresh set of experts (the 15.7 GB weight set is far larger
than L2), and a 256 MB buffer is written between steps (outside the timed
kernels) to flush L2 of the previous step's router and activation bytes.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(the float64 NumPy statement of the layer) on the same workload instead.
Multi-GPU (torchrun): every rank runs an independent replica with its own
weights (the layer is data-parallel over tokens; no collective on the path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s; HBM GB/s at T=1/8, tensor TFLOPS at T=512/8192"
EXPERT_MATRIX_BYTES = None  # filled per config


# DRAM bytes (read + write) per launch of a kernel from an ncu capture of the
# current kernel version, by (workload, kernel); absent: not captured.  The
# decode capture (profiles/mx_stream_kernel_decode_e128.md) ran a 128-expert
# copy of the layer: one token touches 16 experts either way, so a launch moves
# the same bytes as in the 896-expert layer.
TRAFFIC = {
    ("decode_t1", "decode_up"): 187_269_376 + 3_475_968,
    ("decode_t1", "decode_down"): 94_227_200 + 2_305_024,
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="decode_t1", choices=synth.CONFIG_ORDER)
    ap.add_argument("--pool", type=int, default=64, help="distinct token batches rotated over steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=0)
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 decode, 2 grouped")
    ap.add_argument("--E", type=int, default=0,
                    help="fewer resident experts (small profiling captures only; not a bench line)")
    ap.add_argument("--T", type=int, default=0,
                    help="other token count (small profiling captures only; not a bench line)")
    ap.add_argument("--format", choices=["split", "ggml"], default="split",
                    help="expert weight format: compressed-tensors codes + scales, or llama.cpp "
                         "17-byte MXFP4 blocks read directly by the streaming kernels")
    ap.add_argument("--prepared", action="store_true",
                    help="hand the kernels the scales in the prepared atom layout instead of the "
                         "checkpoint's canonical E8M0 rows")
    ap.add_argument("--cache-slots", type=int, default=0,
                    help="host-resident experts behind a device cache of this many experts "
                         "(k3moe_forward_cached); 0 = experts resident in HBM")
    return ap.parse_args()


def bench_config(args):
    cfg = synth.CONFIGS[args.config]
    if args.E:
        cfg = synth.custom(cfg.name, E=args.E)
    if args.T:
        cfg = synth.custom(cfg.name, E=cfg.E, T=args.T)
    return cfg


# ---------------------------------------------------------------------------
# workload facts
# ---------------------------------------------------------------------------
def matrix_bytes(cfg):
    rows, cols = cfg.matrix_shape(synth.W1)
    return rows * cols // 2 + rows * cols // 32


def workload_config(cfg, pool):
    c = {"workload": cfg.name, "tokens_per_step": cfg.T, "experts": cfg.E, "top_k": cfg.k,
         "latent_d": cfg.d, "expert_hidden_f": cfg.f,
         "expert_bytes_resident": 3 * cfg.E * matrix_bytes(cfg),
         "l2": f"{pool} rotating token batches (fresh experts per step) + 256 MB L2 flush "
               "between steps, outside the timed kernels",
         "parallelism": "replicas only"}
    if cfg.block:
        c["model_width_D"] = cfg.D
    return c


def token_pool(cfg, pool):
    """[pool, T, width] bf16 bits: distinct seeded token batches of the config's distribution."""
    big = synth.custom(cfg.name, T=cfg.T * pool, seed_index=cfg.seed_index + 100)
    h = synth.hidden(big)
    return h.reshape(pool, cfg.T, -1)


# ---------------------------------------------------------------------------
# clocks sampler
# ---------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_step_setup(cfg, dense, tokens_bits):
    """Pre-fetch the expert bytes a batch touches (input generation, not timed)."""
    import oracle

    x = oracle.bf16_to_f64(tokens_bits)
    wr = oracle.bf16_to_f64(dense["router_w"])
    if cfg.block:
        hn = oracle.round_bf16(oracle.rmsnorm(x, oracle.bf16_to_f64(dense["norm_gamma"]),
                                              dense["eps"]))
        xr = hn
    else:
        xr = x
    sel = oracle.select_experts(oracle.router_logits(xr, wr), dense["router_b"], cfg.k)["idx"]
    cache = {}
    for e in np.unique(sel):
        for m in range(3):
            cache[(m, int(e))] = synth.expert_matrix_np(cfg, m, int(e))
    return cache


def oracle_step(cfg, dense, tokens_bits, cache):
    import oracle

    x = oracle.bf16_to_f64(tokens_bits)
    wr = oracle.bf16_to_f64(dense["router_w"])
    expert = lambda m, e: cache[(m, e)]
    if cfg.block:
        return oracle.block_forward(x, oracle.bf16_to_f64(dense["norm_gamma"]), dense["eps"],
                                    oracle.bf16_to_f64(dense["w_down"]),
                                    oracle.bf16_to_f64(dense["w_up"]), wr, dense["router_b"],
                                    cfg.k, expert)["out"]
    return oracle.moe_forward(x, wr, dense["router_b"], cfg.k, x, expert)["out"]


def oracle_tokens_per_step(cfg):
    """Tokens the oracle processes per timed step (bounded CPU work)."""
    return min(cfg.T, {"tiny": 4, "decode_t1": 1, "verify_t8": 2, "chunk_t512": 1,
                       "block_t8192": 1}[cfg.name])


def time_oracle(cfg, pool_bits, steps, warmup, dense):
    nt = oracle_tokens_per_step(cfg)
    times = []
    for i in range(warmup + steps):
        toks = pool_bits[i % len(pool_bits)][:nt]
        cache = oracle_step_setup(cfg, dense, toks)
        t0 = time.perf_counter()
        oracle_step(cfg, dense, toks, cache)
        dt = time.perf_counter() - t0
        if i >= warmup:
            times.append(dt)
    return nt, times


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device="cpu") -> float:
    """The largest value over all ranks (the job takes as long as its slowest rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_step: int, steps: int, world: int, max_total_ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_step * steps * world / (max_total_ms / 1e3)


def reference_arm(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    cfg = bench_config(args)
    dense = synth.dense_inputs(cfg)
    pool = token_pool(cfg, max(args.steps + args.warmup, 1))
    nt, times = time_oracle(cfg, pool, args.steps, args.warmup, dense)
    total = sum(times)
    value = nt * len(times) / total
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg, args.steps + args.warmup),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{nt} token(s) of the workload per step, expert bytes "
                                   "prefetched outside the timed region"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def ours_arm(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_setup()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__

    __graft_entry__.build()
    import mxfp4_routed_expert_sigmoid_gb300 as k3

    cfg = bench_config(args)
    dense = synth.dense_inputs(cfg)
    ex = synth.experts_torch(cfg, dev)

    def dv(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    kw = dict(router_w=dv(dense["router_w"]), router_b=dv(dense["router_b"]), k=cfg.k,
              path=args.path, prepared=args.prepared, **ex)
    if cfg.block:
        kw.update(norm_gamma=dv(dense["norm_gamma"]), w_down=dv(dense["w_down"]),
                  w_up=dv(dense["w_up"]), eps=dense["eps"])
    layer = k3.MoELayer(**kw)
    del kw, ex
    if args.format == "ggml":
        layer = k3.ggml_layer(layer)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    pool_np = token_pool(cfg, args.pool)
    pool = [dv(pool_np[i]) for i in range(args.pool)]
    ws = k3.workspace(k3.k3moe_workspace_size(layer, cfg.T) + k3.k3moe_host_staging_size(layer, cfg.T), dev)
    ws_fwd = ws.numel() - k3.k3moe_host_staging_size(layer, cfg.T)
    out = torch.empty_like(pool[0])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    ws_f = ws[:ws_fwd]

    def step(i):
        k3.k3moe_forward(layer, pool[i % args.pool], out=out, ws=ws_f)

    # routing of every pool entry: experts touched per step (algorithmic bytes)
    uniq = []
    for i in range(args.pool):
        step(i)
        idx, _, _ = k3.k3moe_forward_routing(layer, ws, cfg.T, with_logits=False)
        uniq.append(len(torch.unique(idx)))
    check_status(k3, ws)

    # one CUDA graph per token batch: the forward's launches replay back to
    # back on the device, without host launch overhead between them
    def capture(traced):
        # one library-made CUDA graph of k3moe_forward per token batch
        k3.k3moe_trace(traced)
        graphs = [k3.ForwardGraph(layer, pool[i], out, ws_f) for i in range(args.pool)]
        torch.cuda.synchronize()
        k3.k3moe_trace(False)
        return graphs

    graphs = capture(False)
    for i in range(max(args.warmup, 3)):
        graphs[i % args.pool].launch(stream)
    torch.cuda.synchronize()

    # ---- timed region: K steps, per-step events on the launching stream ----
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            graphs[(args.warmup + i) % args.pool].launch(stream)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = job_tokens_per_s(cfg.T, args.steps, world, total_ms)

    # ---- per-kernel durations (traced pass over the same steps) ----
    tgraphs = capture(True)
    per_kernel = {}
    launches_per_step = 0
    trace_source = "graph replay"
    for i in range(args.steps):
        flush.zero_()
        tgraphs[(args.warmup + i) % args.pool].launch(stream)
        tr = k3.k3moe_trace_read()
        launches_per_step = max(launches_per_step, len(tr))
        for name, ms in tr:
            per_kernel.setdefault(name, []).append(ms)
    if not per_kernel:  # events of the graph not readable: trace direct launches
        trace_source = "direct launches (host launch gaps included)"
        k3.k3moe_trace(True)
        for i in range(args.steps):
            flush.zero_()
            step(args.warmup + i)
            tr = k3.k3moe_trace_read()
            launches_per_step = max(launches_per_step, len(tr))
            for name, ms in tr:
                per_kernel.setdefault(name, []).append(ms)
        k3.k3moe_trace(False)
    torch.cuda.synchronize()
    kern_mean = {n: sum(v) / len(v) for n, v in per_kernel.items()}
    del graphs, tgraphs

    # ---- end to end through the host-buffer entry point ----
    width = layer.width
    h2d = cfg.T * width * 2
    pool_host = [torch.from_numpy(pool_np[i].view(np.int16)).view(torch.bfloat16).pin_memory()
                 for i in range(args.pool)]
    out_host = torch.empty_like(pool_host[0]).pin_memory()
    for i in range(args.warmup):
        k3.k3moe_forward_host(layer, pool_host[i % args.pool], out_host=out_host, ws=ws)
    torch.cuda.synchronize()
    e2e_s = 0.0
    for i in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        k3.k3moe_forward_host(layer, pool_host[(args.warmup + i) % args.pool], out_host=out_host,
                              ws=ws)
        e2e_s += time.perf_counter() - t0
    e2e_value = cfg.T * args.steps / e2e_s

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # ---- roofline of the dominant kernel ----
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            peaks = json.load(fh)
    except OSError:
        pass
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    mb = matrix_bytes(cfg)
    u_mean = sum(uniq) / len(uniq)
    # algorithmic bytes per launch of the streaming kernels: every distinct
    # selected expert's matrices once (units of the same expert re-read them)
    algo = {
        "decode_up": u_mean * 2 * mb,
        "decode_down": u_mean * mb,
        "units_up": u_mean * 2 * mb,
        "units_down": u_mean * mb,
        "route_small": cfg.E * cfg.d_router * 2 + cfg.T * cfg.d_router * 2 + cfg.T * cfg.E * 4,
    }
    # algorithmic flops of the grouped GEMMs: 2 f d per (token, expert) and matrix
    flops = {
        "expert_up": cfg.T * cfg.k * 2 * 2.0 * cfg.f * cfg.d,
        "expert_down": cfg.T * cfg.k * 2.0 * cfg.f * cfg.d,
    }
    dom = max(kern_mean, key=kern_mean.get)
    roof = None
    if dom in algo:
        achieved = algo[dom] / (kern_mean[dom] * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                "peak_source": peak_src, "unit": "GB/s", "frac": achieved / hbm_peak,
                "traffic": TRAFFIC.get((cfg.name, dom)) if args.format == "split" else None,
                "algorithmic_bytes_per_launch": algo[dom],
                "avg_launch_ms": kern_mean[dom]}
    elif dom in flops:
        # f16 operands: the measured bf16 rate (same tensor-core rate); the kernel
        # runs inside a step of several ms, so the sustained figure
        tf_peak = peaks.get("bf16_tflops_sustained", 1700.0)
        achieved = flops[dom] / (kern_mean[dom] * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": tf_peak,
                "peak_source": ("measured bf16, sustained" if "bf16_tflops_sustained" in peaks else "fallback"),
                "unit": "TFLOP/s", "frac": achieved / tf_peak, "traffic": TRAFFIC.get((cfg.name, dom)),
                "algorithmic_flops_per_launch": flops[dom], "avg_launch_ms": kern_mean[dom]}
    step_bytes = u_mean * 3 * mb + algo["route_small"]
    mean_ms = total_ms / args.steps
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_of(cfg.T, args.path),
        "data": "synthetic (seeded; random-init weights of the K3 layer shapes)",
        "config": dict(workload_config(cfg, args.pool),
                       weight_format=("ggml 17-byte MXFP4 blocks" if args.format == "ggml" else
                                      "codes + E8M0 scales, " +
                                      ("prepared atoms" if args.prepared else "canonical rows"))),
        "hbm_gbs_step": step_bytes / (mean_ms * 1e-3) / 1e9,
        "experts_touched_per_step": u_mean,
        "kernels_ms": kern_mean,
        "kernels_ms_source": trace_source,
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": h2d},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and world == 1:
        k_steps = 2 if cfg.name != "tiny" else 5
        nt, times = time_oracle(cfg, pool_np, k_steps, 0, dense)
        line["cpu_baseline"] = {"value": nt * len(times) / sum(times), "unit": "tokens/s",
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{k_steps} steps of {nt} token(s) of the workload "
                                          "(NumPy fp64 oracle, expert bytes prefetched)"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def cached_arm(args):
    """The layer with its experts in pinned host memory behind a device cache
    of ``--cache-slots`` experts (k3moe_forward_cached): every step routes,
    fetches the missing experts over the host link (NVLink-C2C on GB300) and
    runs the expert kernels on the cache slots."""
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import __graft_entry__

    __graft_entry__.build()
    import mxfp4_routed_expert_sigmoid_gb300 as k3

    cfg = bench_config(args)
    dense = synth.dense_inputs(cfg)

    def dv(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    layer = k3.MoELayer(router_w=dv(dense["router_w"]), router_b=dv(dense["router_b"]), k=cfg.k,
                        path=args.path, prepared=args.prepared, **synth.experts_torch(cfg, dev))
    hlayer = k3.host_resident(layer)
    del layer
    torch.cuda.empty_cache()
    S = args.cache_slots
    cache = k3.ExpertCache(hlayer, S)
    pool_np = token_pool(cfg, args.pool)
    pool = [dv(pool_np[i]) for i in range(args.pool)]
    ws = k3.workspace(k3.k3moe_workspace_size(hlayer, cfg.T), dev)
    out = torch.empty_like(pool[0])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # link bandwidth for the roofline: copy-engine transfers of 2 GiB from the
    # pinned expert buffer (host -> device), best of 3
    nb = min(2 << 30, hlayer.host_buffer.numel())
    dst = torch.empty(nb, dtype=torch.uint8, device=dev)
    h2d = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst.copy_(hlayer.host_buffer[:nb], non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        h2d.append(nb / (a.elapsed_time(b) * 1e-3) / 1e9)
    link_gbs = max(h2d)
    del dst

    # one pass over the pool fills the cache; graphs per batch (each
    # set-up forward is a call of the cache too)
    for i in range(args.pool):
        k3.k3moe_forward_cached(hlayer, cache, pool[i], out=out, ws=ws)
    torch.cuda.synchronize()
    graphs = [k3.ForwardGraph(hlayer, pool[i], out, ws, cache=cache) for i in range(args.pool)]
    for i in range(max(args.warmup, 3)):
        graphs[i % args.pool].launch(stream)
    check_status(k3, ws)
    before = cache.stats()

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    with Clocks(0) as clk:
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            graphs[(args.warmup + i) % args.pool].launch(stream)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    after = cache.stats()
    total_ms = sum(a.elapsed_time(b) for a, b in evs)
    value = job_tokens_per_s(cfg.T, args.steps, 1, total_ms)
    calls = after["calls"] - before["calls"]
    hits, misses = after["hits"] - before["hits"], after["misses"] - before["misses"]
    fetched = (after["bytes"] - before["bytes"]) / max(calls, 1)

    # per-kernel durations: traced direct launches over the same batches
    k3.k3moe_trace(True)
    per_kernel, launches = {}, 0
    for i in range(args.steps):
        flush.zero_()
        k3.k3moe_forward_cached(hlayer, cache, pool[(args.warmup + i) % args.pool], out=out, ws=ws)
        tr = k3.k3moe_trace_read()
        launches = max(launches, len(tr))
        for name, ms in tr:
            per_kernel.setdefault(name, []).append(ms)
    k3.k3moe_trace(False)
    kern_mean = {n: sum(v) / len(v) for n, v in per_kernel.items()}
    traced = cache.stats()
    fill_bytes = (traced["bytes"] - after["bytes"]) / max(traced["calls"] - after["calls"], 1)

    # end to end: pinned host input -> device, cached forward, result -> host
    pool_host = [torch.from_numpy(pool_np[i].view(np.int16)).view(torch.bfloat16).pin_memory()
                 for i in range(args.pool)]
    out_host = torch.empty_like(pool_host[0]).pin_memory()
    x_dev = torch.empty_like(pool[0])
    e2e_s = 0.0
    for i in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        x_dev.copy_(pool_host[(args.warmup + i) % args.pool], non_blocking=True)
        k3.k3moe_forward_cached(hlayer, cache, x_dev, out=out, ws=ws)
        out_host.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        e2e_s += time.perf_counter() - t0

    fill_ms = kern_mean.get("cache_fill", 0.0)
    fill_gbs = fill_bytes / (fill_ms * 1e-3) / 1e9 if fill_ms > 0 else None
    mb = matrix_bytes(cfg)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_of(cfg.T, args.path),
        "data": "synthetic (seeded; random-init weights of the K3 layer shapes)",
        "config": dict(workload_config(cfg, args.pool), workload=cfg.name + "_host_experts",
                       expert_bytes_resident=0, expert_bytes_host=3 * cfg.E * mb,
                       cache_slots=S, cache_bytes=3 * S * mb),
        "cache": {"hit_rate": hits / max(hits + misses, 1), "hits_per_step": hits / max(calls, 1),
                  "misses_per_step": misses / max(calls, 1), "fetched_bytes_per_step": fetched},
        "kernels_ms": kern_mean,
        "kernels_ms_source": "direct launches (host launch gaps included)",
        "roofline": {"kernel": "cache_fill", "bound": "c2c", "achieved": fill_gbs,
                     "peak": link_gbs, "unit": "GB/s",
                     "peak_source": "measured in this run: pinned host -> device copy-engine "
                                    "transfer of 2 GiB",
                     "frac": (fill_gbs / link_gbs) if fill_gbs else None, "traffic": None,
                     "algorithmic_bytes_per_launch": fill_bytes, "avg_launch_ms": fill_ms},
        "e2e": {"value": cfg.T * args.steps / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": cfg.T * cfg.d * 2, "d2h_bytes_per_step": cfg.T * cfg.d * 2},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def check_status(k3, ws):
    """Raise with the device status word and the place it was set, if any."""
    import torch

    torch.cuda.synchronize()
    code, info = ws[:8].view(torch.int32).cpu().tolist()
    if k3.k3moe_get_status(ws) != 0:
        raise RuntimeError(f"device status {k3.STATUS.get(code, code)} (where: {info}) during setup")


def dtype_of(T: int, path: int) -> str:
    """Arithmetic of the expert path the layer takes for T tokens."""
    decode = path == 1 or (path == 0 and T <= 1024)
    if decode:
        terms = 4 if T > 8 else 5
        return (f"e2m1 x e2m1 block-scaled tensor-core MMA (activations as {terms} E2M1 terms), "
                "fp32 accumulation")
    return "f16 x f16 tensor-core MMA (E2M1 weights dequantised exactly), fp32 accumulation"


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
    elif args.cache_slots > 0:
        cached_arm(args)
    else:
        ours_arm(args)


if __name__ == "__main__":
    main()
