"""GPU parity of the tcgen05 kernels: the dense bf16 GEMM (latent projections,
router logits at large T) and the grouped expert path of k3moe_forward.

Dense GEMM: fp32 accumulation of exact bf16 products; compared with the
float64 product within 1e-5 of the sum of |products| (plus bf16 output
rounding when the output is bf16).  Layer outputs: max |err| per token <=
1e-2 x RMS of the oracle row (the stated tolerance of the dequantising path),
plus half a bf16 ulp for the conversion to the bf16 output.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (bf16_tensor_to_np, make_layer, oracle_forward, oracle_rows_parallel,
                      record_margin, rel_err_rows, sample_rows, to_dev)

pytestmark = pytest.mark.gpu

TOL = 1e-2
TINY = dict()  # the tiny workload at its stated shape (d = f = 64)


@pytest.fixture(scope="module")
def k3():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mxfp4_routed_expert_sigmoid_gb300 as k3mod

    return k3mod


@pytest.mark.parametrize("T,N,K,fp32", [(1, 128, 64, True), (300, 256, 320, False),
                                        (1000, 896, 3584, True), (512, 3584, 1024, False),
                                        (257, 384, 7168, False)])
def test_gemm_bf16(k3, T, N, K, fp32):
    import torch

    rng = np.random.default_rng(T + N + K)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, K)).astype(np.float32))
    w = synth.f32_to_bf16_bits((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    out = k3.k3moe_gemm_bf16(to_dev(x, "cuda"), to_dev(w, "cuda"), out_fp32=fp32)
    got = out.float().cpu().numpy().astype(np.float64)
    xf, wf = oracle.bf16_to_f64(x), oracle.bf16_to_f64(w)
    ref = xf @ wf.T
    bound = np.abs(xf) @ np.abs(wf).T
    tol = 1e-5 * bound + (0 if fp32 else 2.0 ** -8 * np.abs(ref))
    assert np.all(np.abs(got - ref) <= tol + 1e-30), np.max(np.abs(got - ref) - tol)


def compare_forward(k3, cfg, path, tokens=None, bundle=None, tol=TOL, sample=0):
    """The layer on the GPU against the oracle on `tokens` (all by default),
    or, with `sample`, on that many rows chosen from the GPU's routing
    (gpu_util.sample_rows: the heaviest experts' first and last tokens, the
    end of the tile list, seeded random rows), the oracle's expert sum then
    spread over host processes."""
    layer, dense, expert, _ = bundle or make_layer(cfg, path=path)
    x = to_dev(dense["hidden"], "cuda")
    ws = k3.workspace(k3.k3moe_workspace_size(layer, cfg.T))
    out = k3.k3moe_forward(layer, x, ws=ws)
    idx_gpu, _, _ = k3.k3moe_forward_routing(layer, ws, cfg.T)
    assert k3.k3moe_get_status(ws) == 0
    got = bf16_tensor_to_np(out)
    idx_gpu = idx_gpu.cpu().numpy().astype(np.int64)
    if sample:
        tokens = sample_rows(cfg.T, idx_gpu, sample, seed=cfg.seed)
        run = lambda idx=None: oracle_rows_parallel(cfg, dense, tokens, idx=idx)  # noqa: E731
        ref_out, ref = run()
    else:
        tokens = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
        ref = oracle_forward(cfg, dense, expert, tokens=tokens)
        ref_out = ref["out"]
    thr = 1e-3 if cfg.block else 1e-5
    near = ref["margin"] < thr
    same = np.all(ref["idx"] == idx_gpu[tokens], axis=1)
    assert np.all(same | near), "selection differs outside near ties"
    if np.any(~same):
        if sample:
            ref_out, _ = run(idx=idx_gpu[tokens])
        else:
            ref_out = oracle_forward(cfg, dense, expert, tokens=tokens, idx=idx_gpu[tokens])["out"]
    err = rel_err_rows(got[tokens], ref_out)
    record_margin(f"{cfg.name} T={cfg.T} E={cfg.E} d={cfg.d} f={cfg.f} path={path} rows={len(tokens)}",
                  err, tol)
    assert np.all(err <= tol), f"max err/rms {err.max():.3e} at token {tokens[np.argmax(err)]}"
    return out, ws, err


@pytest.mark.parametrize("T", [4, 9, 33])
def test_tiny_grouped(k3, T):
    compare_forward(k3, synth.custom("tiny", T=T, **TINY), 2)


@pytest.mark.parametrize("T", [9, 33])
def test_tiny_units(k3, T):
    """More than 8 tokens on the block-scaled streaming kernels (units of at
    most 16 tokens of one expert)."""
    compare_forward(k3, synth.custom("tiny", T=T, **TINY), 1)


@pytest.mark.parametrize("T,path", [(1024, 1), (1025, 0)])
def test_units_limit(k3, T, path):
    """The largest batch the streaming kernels take (T = 1024; up to 128 tokens
    per expert, eight units of 16) and the first one AUTO sends to the grouped
    GEMMs (T = 1025); 6 seeded token rows checked."""
    cfg = synth.custom("decode_t1", T=T, E=64, k=8, d=768, f=1280, seed_index=26)
    rng = np.random.default_rng(T)
    compare_forward(k3, cfg, path, tokens=np.sort(rng.choice(T, 6, replace=False)))


@pytest.mark.parametrize("T", [4, 20])
def test_every_expert_selected(k3, T):
    """k = E: every expert takes every token (the dense gated MLP special case),
    through the decode path (T = 4) and the units (T = 20, two units per expert)."""
    compare_forward(k3, synth.custom("tiny", T=T, k=8, **TINY), 1)


@pytest.mark.parametrize("T", [40, 300])
def test_mid_units(k3, T):
    # experts with 1..60 tokens: several units per expert, ragged last units
    cfg = synth.custom("decode_t1", T=T, E=64, k=8, d=768, f=1280, seed_index=21)
    compare_forward(k3, cfg, 1)


def test_units_deterministic_and_power_of_two(k3):
    import torch

    cfg = synth.custom("decode_t1", T=64, E=32, k=4, d=512, f=512, seed_index=23)
    layer, dense, expert, ex = make_layer(cfg, path=1)
    x = to_dev(dense["hidden"], "cuda")
    out1 = k3.k3moe_forward(layer, x)
    out2 = k3.k3moe_forward(layer, x)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    ex2 = dict(ex)
    ex2["w2_s"] = ex["w2_s"] + 1
    layer2 = k3.MoELayer(router_w=layer.tensors["router_w"], router_b=layer.tensors["router_b"],
                         k=cfg.k, path=1, **ex2)
    out3 = k3.k3moe_forward(layer2, x)
    assert torch.equal(out3.float(), 2 * out1.float())


def test_units_and_grouped_agree(k3):
    """The streaming (units) and grouped GEMM paths on the same 300 tokens."""
    cfg = synth.custom("decode_t1", T=300, E=64, k=8, d=768, f=1280, seed_index=25)
    bundle = make_layer(cfg, path=1)
    out_u, _, _ = compare_forward(k3, cfg, 1, bundle=bundle)
    layer_g = bundle[0].with_path(2)
    out_g, _, _ = compare_forward(k3, cfg, 2, bundle=(layer_g,) + tuple(bundle[1:]))
    a, b = bf16_tensor_to_np(out_u), bf16_tensor_to_np(out_g)
    assert np.all(rel_err_rows(a, b) <= 2 * TOL + 2.0 ** -8)


@pytest.mark.parametrize("T", [8, 40, 300])
def test_mid_grouped(k3, T):
    # several m-tiles, K stages and units; ragged expert segments
    cfg = synth.custom("decode_t1", T=T, E=64, k=8, d=768, f=1280, seed_index=21)
    compare_forward(k3, cfg, 2)


def test_paths_agree(k3):
    """Decode and grouped paths on the same 8 tokens: both within tolerance of
    the oracle and of each other."""
    import torch

    cfg = synth.custom("decode_t1", T=8, E=64, k=8, d=768, f=1280, seed_index=22)
    bundle = make_layer(cfg, path=1)
    out_d, _, _ = compare_forward(k3, cfg, 1, bundle=bundle)
    layer_g = bundle[0].with_path(2)
    out_g, _, _ = compare_forward(k3, cfg, 2, bundle=(layer_g,) + tuple(bundle[1:]))
    a, b = bf16_tensor_to_np(out_d), bf16_tensor_to_np(out_g)
    assert np.all(rel_err_rows(a, b) <= 2 * TOL + 2.0 ** -8)


def test_grouped_deterministic_and_power_of_two(k3):
    import torch

    cfg = synth.custom("decode_t1", T=64, E=32, k=4, d=512, f=512, seed_index=23)
    layer, dense, expert, ex = make_layer(cfg, path=2)
    x = to_dev(dense["hidden"], "cuda")
    out1 = k3.k3moe_forward(layer, x)
    out2 = k3.k3moe_forward(layer, x)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    ex2 = dict(ex)
    ex2["w2_s"] = ex["w2_s"] + 1
    layer2 = k3.MoELayer(router_w=layer.tensors["router_w"], router_b=layer.tensors["router_b"],
                         k=cfg.k, path=2, **ex2)
    out3 = k3.k3moe_forward(layer2, x)
    assert torch.equal(out3.float(), 2 * out1.float())


def staged_block_check(k3, cfg, layer, ws, out, idx_gpu, dense, expert, tokens):
    """The block step by step, each step against the oracle's definition
    applied to the GPU's own previous step (so a bf16 hand-off that rounds a
    value the other way than the oracle does is not carried into the next
    step's comparison):
      hn = bf16(RMSNorm(h) gamma)         within half a bf16 ulp of the exact value;
      z  = bf16(hn W_down^T)              within half an ulp plus fp32 accumulation;
      m  = bf16(MoE layer(hn -> router, z -> experts))
                                          the layer's bound (1e-2 x row RMS + half an ulp);
      out = bf16(m W_up^T)                within half an ulp plus fp32 accumulation.
    Returns the layer step's err / RMS per row."""
    T = cfg.T
    hn, z, m = (bf16_tensor_to_np(t)[tokens] for t in k3.k3moe_forward_intermediates(layer, ws, T))
    got = bf16_tensor_to_np(out)[tokens]
    q = 2.0 ** -8
    h = oracle.bf16_to_f64(dense["hidden"][tokens])
    gamma = oracle.bf16_to_f64(dense["norm_gamma"])
    hn_ref = oracle.rmsnorm(h, gamma, dense["eps"])
    assert np.all(np.abs(hn - hn_ref) <= q * np.abs(hn_ref) + 1e-6 * np.abs(hn_ref) + 1e-30)
    w_down = oracle.bf16_to_f64(dense["w_down"])
    z_ref = hn @ w_down.T
    acc = np.abs(hn) @ np.abs(w_down).T
    assert np.all(np.abs(z - z_ref) <= q * np.abs(z_ref) + 1e-5 * acc + 1e-30)
    idx_gpu = idx_gpu[tokens]
    if len(tokens) > 32:
        moe_ref, r = oracle_rows_parallel(cfg, dense, tokens, moe_inputs=(hn, z))
    else:
        r = oracle.moe_forward(hn, oracle.bf16_to_f64(dense["router_w"]), dense["router_b"], cfg.k, z, expert)
        moe_ref = r["out"]
    same = np.all(r["idx"] == idx_gpu, axis=1)
    assert np.all(same | (r["margin"] < 1e-5)), "selection differs outside near ties"
    if not np.all(same):
        if len(tokens) > 32:
            moe_ref, _ = oracle_rows_parallel(cfg, dense, tokens, idx=idx_gpu, moe_inputs=(hn, z))
        else:
            moe_ref = oracle.moe_forward(hn, oracle.bf16_to_f64(dense["router_w"]), dense["router_b"], cfg.k,
                                         z, expert, idx=idx_gpu)["out"]
    err = rel_err_rows(m, moe_ref)
    record_margin(f"{cfg.name} T={T} block step: MoE layer on the GPU's hn, z (rows={len(tokens)})", err, TOL)
    assert np.all(err <= TOL), f"MoE step max err/rms {err.max():.3e}"
    w_up = oracle.bf16_to_f64(dense["w_up"])
    o_ref = m @ w_up.T
    acc = np.abs(m) @ np.abs(w_up).T
    assert np.all(np.abs(got - o_ref) <= q * np.abs(o_ref) + 1e-5 * acc + 1e-30)
    return err


def run_block(k3, cfg, path, sample=0, tokens=None):
    """The end-to-end check (compare_forward), then the step-by-step check on
    the same forward's intermediates."""
    bundle = make_layer(cfg, path=path)
    out, ws, _ = compare_forward(k3, cfg, path, bundle=bundle, sample=sample, tokens=tokens)
    layer, dense, expert, _ = bundle
    idx_gpu = k3.k3moe_forward_routing(layer, ws, cfg.T)[0].cpu().numpy().astype(np.int64)
    rows = (sample_rows(cfg.T, idx_gpu, sample, seed=cfg.seed) if sample else
            np.arange(cfg.T) if tokens is None else np.asarray(tokens))
    staged_block_check(k3, cfg, layer, ws, out, idx_gpu, dense, expert, rows)


@pytest.mark.parametrize("T,path", [(4, 1), (4, 2), (300, 1), (300, 2)])
def test_block_small(k3, T, path):
    """Full latent block (RMSNorm, projections, router at the model width)."""
    cfg = synth.custom("block_t8192", T=T, E=32, k=4, d=256, f=512, D=512, seed_index=24)
    run_block(k3, cfg, path)


def test_chunk_t512_full_sampled(k3):
    """The T = 512 chunk at the K3 shape on the unit-grouped streaming path:
    256 token rows checked (every expert's units, their first and last tokens
    for the most loaded ones)."""
    compare_forward(k3, synth.CONFIGS["chunk_t512"], 0, sample=256)


def test_block_t8192_full_sampled(k3):
    """The full latent block at T = 8192, D = 7168 (Zipf-skewed routing): the
    whole batch runs on the GPU; 256 token rows are checked, among them the
    first and last tokens of the 8 most-loaded experts (their first and last
    tiles of the grouped GEMMs) and the last tile of the tile list."""
    run_block(k3, synth.CONFIGS["block_t8192"], 0, sample=256)


@pytest.mark.parametrize("T", [95, 97, 200, 385])
def test_grouped_tile_edges(k3, T):
    """Token counts around the grouped GEMMs' tile size (192 token rows per
    tile, split 96 / 96 between the two issuers of the down projection):
    experts with one partial tile, several full tiles and a ragged last one
    (k = E, so every expert takes every token)."""
    cfg = synth.custom("decode_t1", T=T, E=4, k=4, d=512, f=768, seed_index=61)
    compare_forward(k3, cfg, 2)


@pytest.mark.parametrize("path", [1, 2])
def test_reduction_tails(k3, path):
    """Reduction lengths that are multiples of 64 but not of 256 (d = 320,
    f = 448): the grouped GEMMs read their weights 256 inputs at a time, so
    the last read of each row is partial (one and three 64-input stages) and
    the last prepared scale atom of a row is half used.  Token counts span a
    64-row box plus 16-row boxes (k = E, T = 150)."""
    cfg = synth.custom("decode_t1", T=150, E=4, k=4, d=320, f=448, seed_index=62)
    compare_forward(k3, cfg, path)


def test_verify_t8_grouped_path(k3):
    """The full-size K3 layer through the tcgen05 path at T = 8 (hot experts)."""
    compare_forward(k3, synth.CONFIGS["verify_t8"], 2)
