"""CPU oracle for the latent routed-expert MXFP4 MoE layer (Kimi-K3 style).

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
NumPy float64 statement of what the layer computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg
may import it.  The product (the CUDA library and its Python binding) never
imports, calls or links anything here, and this package imports nothing from
the product.  It shares no code with the CUDA path; the seeded input
generators in ``synth`` are the only common module and hold no step of the
layer's arithmetic.

Sources (web pages; cited by title and section):

* llama.cpp PR #26185 "model: add Kimi-K3 text model":
  - opening post (pwilkin): the five architecture additions, among them the
    latent MoE ("routed experts run at n_expert_latent") and the undefined
    "situ" activation that replaces SwiGLU;
  - review by GrEarl, section "Dry run: prepare_tensors() completes, all 93
    layers mapped, file type = 38": expert count 896, experts used 16,
    sigmoid expert-score gating, the ``exp_probs_b`` tensor and the
    ``ffn_routed_{down,up,norm}`` tensors;
  - review by GrEarl, section "repack_mxfp4_blocks is bit-exact - 0
    mismatches over 11,010,048 values": the compressed-tensors MXFP4 source
    format, the ggml 17-byte block, the E2M1 and doubled ggml value tables,
    both scale formulas and the worked check on a [3072, 3584] w1 tensor.
* Lucebox PR #573 "feat(kimi-k3): add DSpark Q8 artifact and shared
  speculative runtime", section "DSpark acceptance-contract correction": RMS
  epsilon 1e-5; section "Runtime validation": an 8 GiB device expert cache
  in front of SSD-routed experts.
* The K3-Stuff model page, "llama-cpp-patches", change 2: the page cache as
  the hot-expert cache with least-recently-used eviction (``cache.py``, the
  slot policy of the host-resident expert path).

Readings of points the pages leave open are stated in each function.

Parity status per function (what pins it is in ``tests/test_oracle_*.py``):
every function here is pinned by closed forms, worked facts from the pages,
brute force or library special cases, except the E8M0 ``x < 2`` branch of the
ggml half-scale decode, whose value is fixed by the pages only through the
"represented value unchanged" argument - parity unpinned by the pages for
that branch alone.
"""
from .mxfp4 import (E2M1_MAGNITUDES, GGML_KVALUES, decode_ggml, decode_source, e8m0_scale,
                    ggml_e8m0_half, repack_ggml, source_codes, unpack_ggml)
from .routing import bf16_to_f64, permute, router_logits, select_experts, sigmoid
from .layer import (block_forward, block_head, block_tail, expert_ffn, moe_forward, rmsnorm,
                    round_bf16, silu)

__all__ = [
    "E2M1_MAGNITUDES", "GGML_KVALUES", "decode_ggml", "decode_source", "e8m0_scale",
    "ggml_e8m0_half", "repack_ggml", "source_codes", "unpack_ggml", "bf16_to_f64", "permute",
    "router_logits", "select_experts", "sigmoid", "block_forward", "block_head", "block_tail",
    "expert_ffn", "moe_forward",
    "rmsnorm", "round_bf16", "silu",
]
