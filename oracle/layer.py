"""Expert FFN, the routed MoE layer and the full latent block.

Test infrastructure (see the package docstring); float64 throughout.

Sources:
  * llama.cpp PR #26185 "model: add Kimi-K3 text model", opening post
    (pwilkin): latent MoE - routed experts run at the latent width - and the
    "situ" activation replacing SwiGLU; review by GrEarl, section "Dry run":
    the ``ffn_routed_{down,up,norm}`` tensors and embedding length 7168; review
    by GrEarl, section "repack_mxfp4_blocks is bit-exact": the w1 tensor of an
    expert is logical [3072, 3584].
  * Lucebox PR #573, section "DSpark acceptance-contract correction": the
    checkpoint's RMS epsilon is 1e-5.

Readings (the pages do not print these):
  * expert e maps a latent row x (width d) to W2_e (act(W1_e x, W3_e x)) with
    W1_e, W3_e logical [f, d] and W2_e logical [d, f]; blocks of 32 run along
    the input dimension;
  * "situ" is not defined on the pages; the activation is a pluggable gated
    function exercised as act(g, u) = silu(g) * u, silu(g) = g / (1 + e^-g);
  * layer output out[t] = sum_j w[t, j] * expert_{idx[t, j]}(x[t]);
  * block mode: RMSNorm over the model width, x / sqrt(mean(x^2) + eps) * gamma;
    the router reads the normalised hidden; the experts read its latent
    down-projection; the combined latent row goes through the up-projection.
    The tensors between these steps are bf16 (the projections are bf16), so
    the normalised hidden, the latent input z and the combined latent row are
    rounded to bf16 (nearest, ties to even) where the block hands them on.
"""
from __future__ import annotations

import numpy as np

from .mxfp4 import decode_source
from .routing import router_logits, select_experts


def silu(g: np.ndarray) -> np.ndarray:
    """g / (1 + exp(-g))."""
    g = np.asarray(g, np.float64)
    return g / (1.0 + np.exp(-g))


ACTIVATIONS = {"silu_gated": lambda g, u: silu(g) * u}


def expert_ffn(x, w1, w3, w2, act: str = "silu_gated") -> np.ndarray:
    """One expert on rows x [n, d]: W2 (act(W1 x, W3 x)), float64 [n, d]."""
    x = np.asarray(x, np.float64)
    g = x @ np.asarray(w1, np.float64).T
    u = x @ np.asarray(w3, np.float64).T
    h = ACTIVATIONS[act](g, u)
    return h @ np.asarray(w2, np.float64).T


def moe_forward(x_router, router_w, router_b, k, x_expert, expert, idx=None,
                act: str = "silu_gated", experts=None):
    """The routed MoE layer on T token rows.

    x_router [T, d_r] float64   router input;
    router_w [E, d_r] float64; router_b [E] selection bias;
    x_expert [T, d] float64     expert input (the same rows as x_router in
                                latent mode);
    expert(m, e) -> (packed, scale) of matrix m (0 = w1, 1 = w3, 2 = w2) of
                                expert e, in the compressed-tensors layout;
    idx [T, k] optional         a selection to use instead of the top-k (used
                                only for tokens whose top-k is a near tie);
    experts optional            only these experts' terms enter the sum (the
                                layer output is the sum of such parts over a
                                partition of the experts).

    Returns a dict: out [T, d] float64 plus the routing (idx, w, s, beta,
    margin, logits).
    """
    x_router = np.asarray(x_router, np.float64)
    x_expert = np.asarray(x_expert, np.float64)
    T = x_router.shape[0]
    logits = router_logits(x_router, router_w)
    r = select_experts(logits, router_b, k)
    if idx is not None:
        idx = np.asarray(idx, dtype=np.int64)
        s_sel = np.take_along_axis(r["s"], idx, axis=1)
        r["idx"] = idx
        r["w"] = s_sel / s_sel.sum(axis=1, keepdims=True)
    r["logits"] = logits
    out = np.zeros((T, x_expert.shape[1]), dtype=np.float64)
    used = np.unique(r["idx"])
    if experts is not None:
        used = np.intersect1d(used, np.asarray(experts, dtype=np.int64))
    for e in used:
        tok, slot = np.nonzero(r["idx"] == e)
        w1 = decode_source(*expert(0, int(e)))
        w3 = decode_source(*expert(1, int(e)))
        w2 = decode_source(*expert(2, int(e)))
        y = expert_ffn(x_expert[tok], w1, w3, w2, act)
        out[tok] += r["w"][tok, slot][:, None] * y
    r["out"] = out
    return r


def rmsnorm(h, gamma, eps: float) -> np.ndarray:
    """h / sqrt(mean(h^2, over the row) + eps) * gamma."""
    h = np.asarray(h, np.float64)
    return h / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + eps) * np.asarray(gamma, np.float64)


_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_bf16(v) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits: a value in [2**(e-1), 2**e) is rounded to a
    multiple of 2**(e-8); below the normal range the step stays 2**-133.
    Values whose rounded magnitude exceeds the largest finite bf16 become inf.
    """
    v = np.asarray(v, np.float64)
    _, e = np.frexp(v)
    q = np.maximum(e.astype(np.int64) - 8, -133)
    r = np.ldexp(np.rint(np.ldexp(v, -q)), q)
    r = np.where(np.abs(r) > _BF16_MAX, np.copysign(np.inf, v), r)
    return np.where(v == 0, v, r)


def block_head(h, gamma, eps, w_down):
    """The block's steps before the MoE: hn = bf16(RMSNorm(h) * gamma) (the
    router input) and z = bf16(hn W_down^T) (the experts' latent input)."""
    hn = round_bf16(rmsnorm(h, gamma, eps))
    z = round_bf16(hn @ np.asarray(w_down, np.float64).T)
    return hn, z


def block_tail(moe_out, w_up):
    """The block's step after the MoE: the combined latent row, rounded to bf16
    where the block hands it on (m), through the up-projection."""
    m = round_bf16(moe_out)
    return m, m @ np.asarray(w_up, np.float64).T


def block_forward(h, gamma, eps, w_down, w_up, router_w, router_b, k, expert, idx=None,
                  act: str = "silu_gated"):
    """Full latent block: RMSNorm -> router + down-projection -> MoE -> up-projection.

    h [T, D], gamma [D], w_down [d, D], w_up [D, d], router_w [E, D] float64.
    Returns a dict with out [T, D] and the intermediates (hn, z, m) and routing.
    """
    hn, z = block_head(h, gamma, eps, w_down)
    r = moe_forward(hn, router_w, router_b, k, z, expert, idx=idx, act=act)
    m, out = block_tail(r["out"], w_up)
    r["hn"], r["z"], r["m"] = hn, z, m
    r["moe_out"] = r["out"]
    r["out"] = out
    return r
