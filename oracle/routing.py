"""Router and token-to-expert permutation of the layer.

Test infrastructure (see the package docstring); float64 throughout.

Sources: llama.cpp PR #26185 "model: add Kimi-K3 text model", review by
GrEarl, section "Dry run: prepare_tensors() completes, all 93 layers mapped,
file type = 38" (896 experts, 16 used, "expert score gating function
sigmoid", the ``exp_probs_b`` selection-bias tensor).

Readings (the pages name the parts but print no formula):
  * score s_e = sigmoid(l_e) of the router logit l_e = <x, W_r[e]>;
  * the bias only steers the choice: the k experts with the largest
    s_e + b_e are selected;
  * ties in s + b go to the lower expert index, and the selected experts are
    listed in that order (key: s + b descending, index ascending);
  * combine weights are the unbiased scores renormalised over the selected
    set, w_j = s_{S_j} / sum_j' s_{S_j'}; no extra routed scaling factor.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def router_logits(x: np.ndarray, w_r: np.ndarray) -> np.ndarray:
    """l[t, e] = sum_i x[t, i] * W_r[e, i] (float64 inputs)."""
    return np.asarray(x, np.float64) @ np.asarray(w_r, np.float64).T


def sigmoid(l: np.ndarray) -> np.ndarray:
    """1 / (1 + exp(-l))."""
    return 1.0 / (1.0 + np.exp(-np.asarray(l, np.float64)))


def select_experts(logits: np.ndarray, bias: np.ndarray, k: int):
    """Top-k selection on s + b with renormalised unbiased weights.

    Returns a dict with
      idx    [T, k] int64, slot order = (s + b) descending, index ascending;
      w      [T, k] float64 combine weights;
      s, beta [T, E] the scores and the selection keys;
      margin [T] beta of the k-th selected minus beta of the best unselected
             (inf when k == E).
    """
    logits = np.asarray(logits, np.float64)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    s = sigmoid(logits)
    beta = s + np.asarray(bias, np.float64)[None, :]
    # a stable sort on -beta keeps equal keys in ascending index order
    order = np.argsort(-beta, axis=1, kind="stable")
    idx = order[:, :k]
    s_sel = np.take_along_axis(s, idx, axis=1)
    w = s_sel / s_sel.sum(axis=1, keepdims=True)
    if k < E:
        b_sorted = np.take_along_axis(beta, order, axis=1)
        margin = b_sorted[:, k - 1] - b_sorted[:, k]
    else:
        margin = np.full(T, np.inf)
    return {"idx": idx.astype(np.int64), "w": w, "s": s, "beta": beta, "margin": margin}


def permute(idx: np.ndarray, E: int):
    """Expert histogram, exclusive scan and the (expert, token)-sorted pair list.

    Pairs are numbered p = t * k + j (token t, slot j).  Returns
      counts  [E]      number of pairs routed to each expert;
      offsets [E + 1]  exclusive prefix sum of counts (offsets[E] = T * k);
      perm    [T * k]  perm[r] = pair id placed at row r; rows of expert e are
                       offsets[e] .. offsets[e+1]-1, in ascending token order;
      inv     [T * k]  inv[p] = row of pair p (inverse of perm).
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    # a stable sort of pair ids by expert keeps ascending pair id, hence
    # ascending token, inside each expert's segment
    perm = np.argsort(flat, kind="stable").astype(np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(T * k, dtype=np.int64)
    return {"counts": counts, "offsets": offsets, "perm": perm, "inv": inv}
