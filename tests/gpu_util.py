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


def make_layer(cfg: synth.Config, dev="cuda", path=0, on_device_experts=None):
    """(layer, dense host inputs, expert accessor for the oracle, device expert dict)."""
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
              k=cfg.k, path=path, **ex_dev)
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
