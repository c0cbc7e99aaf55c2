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


def rel_err_rows(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """max |got - ref| / RMS(ref) per row."""
    rms = np.sqrt(np.mean(ref ** 2, axis=1))
    return np.max(np.abs(got - ref), axis=1) / np.maximum(rms, 1e-300)


def bf16_tensor_to_np(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
