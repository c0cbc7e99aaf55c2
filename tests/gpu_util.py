"""Device tensors for the seeded workloads (tests only)."""
from __future__ import annotations

import numpy as np

import oracle
import synth


def to_dev(arr: np.ndarray, dev):
    import torch

    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(dev)


def make_layer(cfg: synth.Config, dev="cuda", path=0, on_device_experts=None, prepared=False):
    """(layer, dense host inputs, expert accessor for the oracle, device expert dict).

    The layer gets the expert bytes exactly as generated: codes and canonical
    E8M0 scales (the checkpoint's weight_packed / weight_scale layout); with
    ``prepared`` it also carries the prepared scale atoms, which the kernels
    then read instead."""
    import mxfp4_routed_expert_sigmoid_gb300 as k3

    dense = synth.dense_inputs(cfg)
    big = cfg.E * cfg.f * cfg.d > 64 * 1024 * 1024 if on_device_experts is None else on_device_experts
    if big:
        ex_dev = synth.experts_torch(cfg, dev)
        expert = lambda m, e: synth.expert_matrix_np(cfg, m, e)
    else:
        ex = synth.experts_np(cfg)
        ex_dev = {k: to_dev(v, dev) for k, v in ex.items()}
        names = synth.MATRIX_NAMES
        expert = lambda m, e: (ex[names[m] + "_q"][e], ex[names[m] + "_s"][e])
    kw = dict(router_w=to_dev(dense["router_w"], dev), router_b=to_dev(dense["router_b"], dev),
              k=cfg.k, path=path, prepared=prepared, **ex_dev)
    if cfg.block:
        kw.update(norm_gamma=to_dev(dense["norm_gamma"], dev), w_down=to_dev(dense["w_down"], dev),
                  w_up=to_dev(dense["w_up"], dev), eps=dense["eps"])
    layer = k3.MoELayer(**kw)
    return layer, dense, expert, ex_dev


def oracle_forward(cfg, dense, expert, tokens=None, idx=None):
    """Oracle output (float64) for all tokens or a subset (rows of the input)."""
    h = dense["hidden"] if tokens is None else dense["hidden"][tokens]
    x = oracle.bf16_to_f64(h)
    wr = oracle.bf16_to_f64(dense["router_w"])
    if cfg.block:
        return oracle.block_forward(x, oracle.bf16_to_f64(dense["norm_gamma"]), dense["eps"],
                                    oracle.bf16_to_f64(dense["w_down"]),
                                    oracle.bf16_to_f64(dense["w_up"]), wr, dense["router_b"],
                                    cfg.k, expert, idx=idx)
    return oracle.moe_forward(x, wr, dense["router_b"], cfg.k, x, expert, idx=idx)


def rel_err_rows(got: np.ndarray, ref: np.ndarray, out_bf16: bool = True) -> np.ndarray:
    """Per row: max over elements of (|got - ref| - q * |ref|) / RMS(ref).

    The layer's output is bf16, and rounding a value to bf16 moves it by up to
    half a unit in the last place, i.e. up to 2^-8 of its magnitude: exact
    arithmetic followed by a correctly rounded bf16 output already reaches
    1.05e-2 x RMS on the tiny workload.  The layer's stated bound (1e-2 x RMS)
    therefore applies to the computed value, and the final bf16 conversion is
    allowed its half ulp on top (q = 2^-8; q = 0 for fp32 outputs).
    """
    q = 2.0 ** -8 if out_bf16 else 0.0
    rms = np.sqrt(np.mean(ref ** 2, axis=1))
    excess = np.abs(got - ref) - q * np.abs(ref)
    return np.max(excess, axis=1) / np.maximum(rms, 1e-300)


def bf16_tensor_to_np(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


# ---------------------------------------------------------------------------
# margins: every parity check records its worst err / RMS against its bound,
# and the session prints them (tests/conftest.py) so the headroom is visible
# ---------------------------------------------------------------------------
MARGINS = []


def record_margin(label: str, err, tol: float):
    import os

    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    MARGINS.append((test, label, float(np.max(err)), float(tol)))


# ---------------------------------------------------------------------------
# the oracle on many rows of a full-size workload, its expert sum split over
# processes: the output is the sum of per-expert terms, so each worker sums a
# subset of the used experts (oracle.moe_forward with `experts`) and the parts
# are added; block mode wraps that in oracle.block_head / block_tail
# ---------------------------------------------------------------------------
def _moe_part(args):
    cfg, x_router, router_w, bias, x_expert, idx, experts = args
    expert = lambda m, e: synth.expert_matrix_np(cfg, m, e)  # noqa: E731
    return oracle.moe_forward(x_router, router_w, bias, cfg.k, x_expert, expert, idx=idx,
                              experts=experts)["out"]


def oracle_rows_parallel(cfg, dense, tokens, idx=None, workers=None, moe_inputs=None):
    """oracle_forward(cfg, dense, expert, tokens, idx)["out"] with the expert
    bytes regenerated per worker (synth.expert_matrix_np) and the used experts
    split over a spawn pool.  Returns (out [n, width] float64, routing dict of
    the oracle on these rows: idx, margin).  With ``moe_inputs`` = (router
    input rows, expert input rows) the MoE layer alone is evaluated on them
    (block mode: its unrounded output, before the bf16 hand-off and W_up)."""
    import multiprocessing as mp
    import os

    wr = oracle.bf16_to_f64(dense["router_w"])
    if moe_inputs is not None:
        x_r, x_e = moe_inputs
    elif cfg.block:
        h = oracle.bf16_to_f64(dense["hidden"][tokens])
        x_r, x_e = oracle.block_head(h, oracle.bf16_to_f64(dense["norm_gamma"]), dense["eps"],
                                     oracle.bf16_to_f64(dense["w_down"]))
    else:
        x_r = x_e = oracle.bf16_to_f64(dense["hidden"][tokens])
    r = oracle.select_experts(oracle.router_logits(x_r, wr), dense["router_b"], cfg.k)
    used = np.unique(r["idx"] if idx is None else idx)
    n = workers or min(len(used), os.cpu_count() or 1)
    parts = [used[i::n] for i in range(n)]
    jobs = [(cfg, x_r, wr, dense["router_b"], x_e, idx, p) for p in parts]
    ctx = mp.get_context("spawn")
    with ctx.Pool(n) as pool:
        out = sum(pool.map(_moe_part, jobs))
    if cfg.block and moe_inputs is None:
        out = oracle.block_tail(out, oracle.bf16_to_f64(dense["w_up"]))[1]
    return out, {"idx": r["idx"], "margin": r["margin"]}


def sample_rows(T: int, idx_gpu: np.ndarray, n: int, seed: int, per_expert: int = 6):
    """n token rows of a large batch for a sampled parity check: the first and
    last tokens routed to each of the 8 most-loaded experts (the heaviest
    expert segments, their first and last tiles), the last tokens of the
    highest-numbered expert that has tokens (the end of the tile list), and
    seeded random rows for the rest."""
    loads = np.bincount(idx_gpu.reshape(-1), minlength=int(idx_gpu.max()) + 1)
    pick = []
    for e in np.argsort(-loads, kind="stable")[:8]:
        toks = np.nonzero((idx_gpu == e).any(axis=1))[0]
        pick += toks[: per_expert // 2].tolist() + toks[-(per_expert // 2):].tolist()
    last = int(np.nonzero(loads)[0][-1])
    pick += np.nonzero((idx_gpu == last).any(axis=1))[0][-per_expert:].tolist()
    chosen = list(dict.fromkeys(pick))[:n]
    rest = np.setdiff1d(np.arange(T), chosen)
    rng = np.random.default_rng(seed)
    chosen += rng.choice(rest, n - len(chosen), replace=False).tolist()
    return np.sort(np.asarray(chosen, dtype=np.int64))
