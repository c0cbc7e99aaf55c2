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
# current kernel version, by (workload, weight format, scales, kernel); absent:
# not captured since the kernel last changed.  Source: the launch lists of
# these four workloads at full size (dram__bytes_read.sum +
# dram__bytes_write.sum, one pass, mean over the captured launches of the
# kernel; profiles/launches_<workload>.md give the command).
TRAFFIC = {
    ("decode_t1", "split", "prepared", "decode_up"): 187.6e6,
    ("verify_t8", "split", "prepared", "decode_up"): 379.1e6,
    ("chunk_t512", "split", "prepared", "units_up"): 9122.0e6,
    ("block_t8192", "split", "prepared", "expert_up"): 8467.6e6,
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
    ap.add_argument("--scales", choices=["prepared", "canonical"], default="prepared",
                    help="hand the kernels the E8M0 scales in the prepared atom layout (written once "
                         "at load by k3moe_prepare_scales) or as the checkpoint's canonical rows")
    ap.add_argument("--all-configs", type=int, default=1,
                    help="the default decode_t1 run also measures verify_t8, chunk_t512 and "
                         "block_t8192 (key 'configs'); 0 = the headline workload only")
    ap.add_argument("--oracle-timing", action="store_true", help=argparse.SUPPRESS)
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


def workload_config(cfg):
    """The workload and its L2 handling; how many distinct token batches a run
    rotates through is reported beside it (``token_batches``), so that both
    arms name the same workload with the same dictionary."""
    c = {"workload": cfg.name, "tokens_per_step": cfg.T, "experts": cfg.E, "top_k": cfg.k,
         "latent_d": cfg.d, "expert_hidden_f": cfg.f,
         "expert_bytes_resident": 3 * cfg.E * matrix_bytes(cfg),
         "l2": "rotating token batches (fresh experts per step) + 256 MB L2 flush "
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
        "config": workload_config(cfg),
        "token_batches": args.steps + args.warmup,
        "weight_format": "codes + E8M0 scales as the checkpoint's canonical rows",
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{nt} token(s) of the workload per step, expert bytes "
                                   "prefetched outside the timed region"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def dev_tensor(a, dev):
    import torch

    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def build_layer(k3, cfg, args, dev):
    """The config's layer on the device: seeded expert bytes generated in place
    (15.7 GB at the K3 shape), the scales canonical or also prepared."""
    dense = synth.dense_inputs(cfg)
    kw = dict(router_w=dev_tensor(dense["router_w"], dev), router_b=dev_tensor(dense["router_b"], dev),
              k=cfg.k, path=args.path, prepared=args.scales == "prepared", **synth.experts_torch(cfg, dev))
    if cfg.block:
        kw.update(norm_gamma=dev_tensor(dense["norm_gamma"], dev), w_down=dev_tensor(dense["w_down"], dev),
                  w_up=dev_tensor(dense["w_up"], dev), eps=dense["eps"])
    layer = k3.MoELayer(**kw)
    if args.format == "ggml":
        import torch

        layer = k3.ggml_layer(layer)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return layer, dense


def pool_size(cfg, requested):
    # token batches rotated over the steps: enough distinct batches for the
    # small-T workloads (every step routes to fresh experts); the large ones
    # are far larger than L2 each
    return requested if cfg.T <= 8 else max(4, min(requested, 8))


def stamp_pass(k3, layer, pool, out, ws, order, flush, stream):
    """Device stamps of the forward replayed from graphs captured with stamps
    on (k3moe_trace mode 2): per kernel the mean of (last CTA end - first CTA
    start after its dependency wait), and the mean span of the whole forward."""
    import torch

    k3.k3moe_trace(2)
    graphs = {i: k3.ForwardGraph(layer, pool[i], out, ws) for i in sorted(set(order))}
    k3.k3moe_trace(0)
    per, spans, marks = {}, [], {}
    for i in order:
        flush.zero_()
        graphs[i].launch(stream)
        st = k3.k3moe_trace_read_stamps()
        seen = {}
        for n, a, b in st:
            if a < 0:
                continue
            c = seen.get(n, 0)
            seen[n] = c + 1
            key = n if c == 0 else f"{n}#{c}"
            per.setdefault(key, []).append((b - a) * 1e-3)
            marks.setdefault(key, []).append((a, b))
        spans.append(max(b for _, _, b in st) * 1e-3)
    torch.cuda.synchronize()
    del graphs
    mean = {n: sum(v) / len(v) for n, v in per.items()}
    # mean start / end (us after the forward's first kernel start) per kernel
    timeline = {n: [round(sum(a for a, _ in v) / len(v), 2), round(sum(b for _, b in v) / len(v), 2)]
                for n, v in marks.items()}
    return mean, sum(spans) / len(spans), timeline


def algorithmic_work(cfg, u_mean, mb):
    """Per launch: bytes of the streaming kernels (every distinct selected
    expert's matrices once; the router's weights), flops of the tensor-core
    GEMMs (2 m n k)."""
    T, k, d, f = cfg.T, cfg.k, cfg.d, cfg.f
    bytes_ = {
        "decode_up": u_mean * 2 * mb, "decode_down": u_mean * mb,
        "units_up": u_mean * 2 * mb, "units_down": u_mean * mb,
        "route_small": cfg.E * cfg.d_router * 2 + T * cfg.d_router * 2 + T * cfg.E * 4,
    }
    flops = {
        "expert_up": T * k * 2 * 2.0 * f * d, "expert_down": T * k * 2.0 * f * d,
        "latent_down": 2.0 * T * cfg.D * d, "latent_up": 2.0 * T * d * cfg.D,
        "router_logits": 2.0 * T * cfg.E * cfg.d_router,
    }
    return bytes_, flops


def roofline_of(name, ms, bytes_, flops, peaks, traffic):
    """The roofline entry of one kernel from its stamp duration."""
    if name in bytes_:
        peak = peaks.get("hbm_gbs", 6800.0)
        achieved = bytes_[name] / (ms * 1e-3) / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": achieved, "peak": peak,
                "peak_source": "measured" if "hbm_gbs" in peaks else "fallback",
                "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                "algorithmic_bytes_per_launch": bytes_[name], "avg_launch_ms": ms,
                "duration_source": "device stamps inside the graph replay (first CTA past its "
                                   "dependency wait to last CTA end)"}
    if name in flops:
        # f16 / bf16 operands, inside a step of several ms: the sustained bf16 figure
        peak = peaks.get("bf16_tflops_sustained", 1700.0)
        achieved = flops[name] / (ms * 1e-3) / 1e12
        return {"kernel": name, "bound": "tensor", "achieved": achieved, "peak": peak,
                "peak_source": "measured bf16, sustained" if "bf16_tflops_sustained" in peaks else "fallback",
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "algorithmic_flops_per_launch": flops[name], "avg_launch_ms": ms,
                "duration_source": "device stamps inside the graph replay"}
    return None


def measure(k3, cfg, args, dev, world, steps, warmup, peaks):
    """One workload: its layer, a pool of token batches, one CUDA graph of
    k3moe_forward per batch; K timed replays (events around each on the
    launching stream, L2 flushed between steps outside the events), a second
    pass with device stamps for the per-kernel times, and the end-to-end
    figure through k3moe_forward_host (pinned host input and output, copies
    inside the call).  Returns the measurement and the per-rank total ms."""
    import torch
    import torch.distributed as dist

    layer, dense = build_layer(k3, cfg, args, dev)
    npool = pool_size(cfg, args.pool)
    pool_np = token_pool(cfg, npool)
    pool = [dev_tensor(pool_np[i], dev) for i in range(npool)]
    stage = k3.k3moe_host_staging_size(layer, cfg.T)
    ws = k3.workspace(k3.k3moe_workspace_size(layer, cfg.T) + stage, dev)
    ws_f = ws[: ws.numel() - stage]
    out = torch.empty_like(pool[0])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # routing of every pool entry: experts touched per step (algorithmic bytes)
    uniq = []
    for i in range(npool):
        k3.k3moe_forward(layer, pool[i], out=out, ws=ws_f)
        idx, _, _ = k3.k3moe_forward_routing(layer, ws_f, cfg.T, with_logits=False)
        uniq.append(len(torch.unique(idx)))
    check_status(k3, ws_f)

    graphs = [k3.ForwardGraph(layer, pool[i], out, ws_f) for i in range(npool)]
    for i in range(max(warmup, 3)):
        flush.zero_()
        graphs[i % npool].launch(stream)
    torch.cuda.synchronize()
    order = [(warmup + i) % npool for i in range(steps)]

    # ---- timed region: K steps, per-step events on the launching stream ----
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(dev.index or 0) as clk:
        for i in range(steps):
            flush.zero_()
            evs[i][0].record(stream)
            graphs[order[i]].launch(stream)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    check_status(k3, ws_f)
    total_ms = sum(a.elapsed_time(b) for a, b in evs)
    del graphs

    kern, span, timeline = stamp_pass(k3, layer, pool, out, ws_f, order, flush, stream)

    # ---- end to end through the host-buffer entry point ----
    width = layer.width
    io = cfg.T * width * 2
    pool_host = [torch.from_numpy(pool_np[i].view(np.int16)).view(torch.bfloat16).pin_memory()
                 for i in range(npool)]
    out_host = torch.empty_like(pool_host[0]).pin_memory()
    for i in range(max(warmup, 1)):
        k3.k3moe_forward_host(layer, pool_host[i % npool], out_host=out_host, ws=ws)
    torch.cuda.synchronize()
    e2e_s = 0.0
    for i in range(steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        k3.k3moe_forward_host(layer, pool_host[order[i]], out_host=out_host, ws=ws)
        e2e_s += time.perf_counter() - t0
    check_status(k3, ws)

    mb = matrix_bytes(cfg)
    u_mean = sum(uniq) / len(uniq)
    bytes_, flops = algorithmic_work(cfg, u_mean, mb)
    dom = max(kern, key=kern.get)
    fmt = "split" if args.format == "split" else "ggml"
    roof = roofline_of(dom, kern[dom], bytes_, flops, peaks,
                       TRAFFIC.get((cfg.name, fmt, args.scales, dom)))
    mean_ms = total_ms / steps
    res = {
        "value": cfg.T * steps / (total_ms / 1e3), "unit": "tokens/s", "ms_per_step": mean_ms,
        "dtype": dtype_of(cfg.T, args.path),
        "config": workload_config(cfg),
        "token_batches": npool,
        "weight_format": ("ggml 17-byte MXFP4 blocks" if args.format == "ggml" else
                          "codes + E8M0 scales as " +
                          ("prepared atoms" if args.scales == "prepared" else
                           "the checkpoint's canonical rows")),
        "experts_touched_per_step": u_mean,
        "hbm_gbs_step": (u_mean * 3 * mb + bytes_["route_small"]) / (mean_ms * 1e-3) / 1e9,
        "kernels_ms": kern,
        "kernels_ms_source": "device stamps inside graph replays of the same steps",
        "forward_span_ms": span,
        "timeline_us": timeline,
        "roofline": roof,
        "e2e": {"value": cfg.T * steps / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": io,
                "d2h_bytes_per_step": io},
        "gpu_launches": len(kern) * steps,
        "clocks": clk.summary(),
    }
    if cfg.T >= 512:
        fl = sum(v for n, v in flops.items() if n.startswith("expert_") or cfg.block)
        res["tflops_step"] = fl / (mean_ms * 1e-3) / 1e12
    del layer, pool, ws, ws_f, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res, total_ms


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

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            peaks = json.load(fh)
    except OSError:
        pass

    cfg = bench_config(args)
    res, total_ms = measure(k3, cfg, args, dev, world, args.steps, args.warmup, peaks)
    total_ms = max_over_ranks(total_ms, world, dev)
    value = job_tokens_per_s(cfg.T, args.steps, world, total_ms)

    # the other workloads of the layer, measured in the same run (headline run only)
    others = {}
    if args.all_configs and not (args.E or args.T or args.config != "decode_t1"):
        for name in ("verify_t8", "chunk_t512", "block_t8192"):
            o, o_ms = measure(k3, synth.CONFIGS[name], args, dev, world, args.steps, args.warmup, peaks)
            o_ms = max_over_ranks(o_ms, world, dev)
            o["value"] = job_tokens_per_s(synth.CONFIGS[name].T, args.steps, world, o_ms)
            others[name] = o

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": res["dtype"],
        "data": "synthetic (seeded; random-init weights of the K3 layer shapes)",
    }
    line.update({k: v for k, v in res.items() if k not in ("value", "ms_per_step", "unit", "dtype")})
    line["gpu_launches"] = res["gpu_launches"]
    if others:
        line["configs"] = others
    if not args.no_cpu_baseline and world == 1:
        k_steps = 2 if cfg.name != "tiny" else 5
        dense = synth.dense_inputs(cfg)
        nt, times = time_oracle(cfg, token_pool(cfg, k_steps), k_steps, 0, dense)
        one = oracle_one_thread(cfg.name, k_steps)
        line["cpu_baseline"] = {"value": nt * len(times) / sum(times), "unit": "tokens/s",
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{k_steps} steps of {nt} token(s) of the workload "
                                          "(NumPy fp64 oracle, expert bytes prefetched; BLAS "
                                          "threads = cores)",
                                "one_thread": one}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def oracle_one_thread(config: str, steps: int):
    """The same oracle timing in a child process whose BLAS and OpenMP pools
    have one thread (value in tokens/s), or None if the child fails."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-timing", "--config", config,
                            "--steps", str(steps)], env=env, capture_output=True, text=True, timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])["value"]
    except Exception:
        return None


def oracle_timing_only(args):
    cfg = bench_config(args)
    dense = synth.dense_inputs(cfg)
    nt, times = time_oracle(cfg, token_pool(cfg, args.steps), args.steps, 0, dense)
    print(json.dumps({"value": nt * len(times) / sum(times), "unit": "tokens/s"}), flush=True)


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
                        path=args.path, prepared=args.scales == "prepared", **synth.experts_torch(cfg, dev))
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
        "token_batches": args.pool,
        "config": dict(workload_config(cfg), workload=cfg.name + "_host_experts",
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
    if args.oracle_timing:
        oracle_timing_only(args)
    elif args.impl == "reference":
        reference_arm(args)
    elif args.cache_slots > 0:
        cached_arm(args)
    else:
        ours_arm(args)


if __name__ == "__main__":
    main()
