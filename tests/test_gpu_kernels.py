"""GPU parity of the integer and routing kernels against the oracle.

Repack / unpack and the permutation are bit-exact; routing indices are exact
for every token whose selection margin is above the fp32 rounding level (and
valid for the rest); weights and logits within fp32 rounding.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def k3():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mxfp4_routed_expert_sigmoid_gb300 as k3mod

    return k3mod


def _repack_case(k3, packed, scale, misalign_out=False):
    import torch

    rows, cols = packed.shape[0], packed.shape[1] * 2
    pd, sd = to_dev(packed, "cuda"), to_dev(scale, "cuda")
    if misalign_out:
        buf = torch.empty(rows * (cols // 32) * 17 + 1, dtype=torch.uint8, device="cuda")
        out = buf[1:].view(rows, cols // 32, 17)
        blocks = k3.k3moe_repack_mxfp4(pd, sd, out=out)
    else:
        blocks = k3.k3moe_repack_mxfp4(pd, sd)
    want = oracle.repack_ggml(packed, scale)
    got = blocks.cpu().numpy()
    assert np.array_equal(got, want)
    p2, s2 = k3.k3moe_unpack_mxfp4(blocks.contiguous() if misalign_out else blocks)
    assert np.array_equal(p2.cpu().numpy(), packed)
    assert np.array_equal(s2.cpu().numpy(), scale)


@pytest.mark.parametrize("rows,cols", [(1, 32), (37, 96), (255, 64), (300, 2048)])
def test_repack_unpack_bit_exact(k3, rows, cols):
    packed = synth.random_bytes(rows * 7 + cols, rows * cols // 2).reshape(rows, cols // 2)
    scale = synth.random_bytes(rows * 11 + cols, rows * cols // 32).reshape(rows, cols // 32)
    scale[scale == 255] = 254
    _repack_case(k3, packed, scale)
    _repack_case(k3, packed, scale, misalign_out=True)


def prepared_atoms_np(s):
    """The prepared scale layout written out with numpy: per expert, rows
    padded to whole tiles of 128 and blocks to whole groups of 4 with zeros;
    per (tile, 128-wide input group) a 512-byte atom with row m = 32 q + r,
    block b at byte 16 r + 4 q + b."""
    E, R, nb = s.shape
    tiles, G = -(-R // 128), -(-nb // 4)
    pad = np.zeros((E, tiles * 128, G * 4), np.uint8)
    pad[:, :R, :nb] = s
    return pad.reshape(E, tiles, 4, 32, G, 4).transpose(0, 1, 4, 3, 2, 5).reshape(-1)


@pytest.mark.parametrize("E,rows,cols", [(1, 128, 128), (3, 384, 256), (5, 1152, 768), (8, 64, 64),
                                         (2, 192, 320), (3, 64, 448)])
def test_prepare_scales_bit_exact(k3, E, rows, cols):
    s = synth.random_bytes(E * rows * 3 + cols, E * rows * cols // 32).reshape(E, rows, cols // 32)
    sf = k3.k3moe_prepare_scales(to_dev(s, "cuda"))
    assert sf.numel() == k3.k3moe_prepared_scales_size(E, rows, cols)
    assert np.array_equal(sf.cpu().numpy(), prepared_atoms_np(s))
    back = k3.k3moe_unprepare_scales(sf, s.shape)
    assert np.array_equal(back.cpu().numpy(), s)


def test_repack_worked_check_shape(k3):
    """The pages' [3072, 3584] check: GPU blocks decode to the same values."""
    rows, cols = 3072, 3584
    packed = synth.random_bytes(2026, rows * cols // 2).reshape(rows, cols // 2)
    scale = synth.random_exponents(2027, rows * cols // 32, 120, 122).reshape(rows, cols // 32)
    import torch

    blocks = k3.k3moe_repack_mxfp4(to_dev(packed, "cuda"), to_dev(scale, "cuda")).cpu().numpy()
    assert blocks.nbytes == 5849088
    assert np.array_equal(blocks, oracle.repack_ggml(packed, scale))
    ref = oracle.decode_source(packed, scale)
    assert int((oracle.decode_ggml(blocks) != ref).sum()) == 0


def _route_case(k3, cfg, T=None):
    dense = synth.dense_inputs(cfg if T is None else synth.custom(cfg.name, T=T))
    x = dense["hidden"]
    idx, w, logits = k3.k3moe_route(to_dev(x, "cuda"), to_dev(dense["router_w"], "cuda"),
                                    to_dev(dense["router_b"], "cuda"), cfg.k)
    idx, w, logits = idx.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy()
    # logits: fp32 accumulation of exact bf16 products vs the fp64 oracle
    ref_l = oracle.router_logits(oracle.bf16_to_f64(x), oracle.bf16_to_f64(dense["router_w"]))
    scale = np.abs(oracle.bf16_to_f64(x)) @ np.abs(oracle.bf16_to_f64(dense["router_w"])).T
    assert np.all(np.abs(logits - ref_l) <= 1e-5 * scale + 1e-30)
    # selection: the oracle's rule applied to the kernel's own logits
    r = oracle.select_experts(logits.astype(np.float64), dense["router_b"], cfg.k)
    sure = r["margin"] > 1e-6
    assert np.array_equal(idx[sure], r["idx"][sure])
    for t in np.nonzero(~sure)[0]:  # near ties: any valid top-k
        sel = set(idx[t].tolist())
        assert len(sel) == cfg.k
        uns = [r["beta"][t, e] for e in range(cfg.E) if e not in sel]
        assert min(r["beta"][t, idx[t]]) >= max(uns) - 1e-6
    s_sel = np.take_along_axis(r["s"], idx.astype(np.int64), axis=1)
    assert np.allclose(w, s_sel / s_sel.sum(1, keepdims=True), rtol=2e-6, atol=1e-7)
    assert np.allclose(w.sum(1), 1.0, atol=1e-6)
    return idx


@pytest.mark.parametrize("name,T", [("tiny", None), ("decode_t1", None), ("verify_t8", None),
                                    ("decode_t1", 3), ("chunk_t512", 40), ("chunk_t512", 100),
                                    ("chunk_t512", 3000)])
def test_route_matches_oracle(k3, name, T):
    """T = 3000 goes through the warp-per-token top-k (beyond 2048 tokens)."""
    _route_case(k3, synth.CONFIGS[name], T)


def test_route_warp_topk_equals_block_topk(k3):
    """The two top-k kernels give bitwise the same slots and weights: the first
    2048 tokens of a 3000-token batch on their own (one block per token)
    against the same rows inside the whole batch (one warp per token)."""
    import torch
    cfg = synth.custom("chunk_t512", T=3000)
    dense = synth.dense_inputs(cfg)
    x = to_dev(dense["hidden"], "cuda")
    args = (to_dev(dense["router_w"], "cuda"), to_dev(dense["router_b"], "cuda"), cfg.k)
    i_all, w_all, _ = k3.k3moe_route(x, *args)
    i_blk, w_blk, _ = k3.k3moe_route(x[:2048].contiguous(), *args)
    torch.cuda.synchronize()
    assert torch.equal(i_all[:2048], i_blk)
    assert torch.equal(w_all[:2048], w_blk)


def test_route_hot_experts(k3):
    cfg = synth.CONFIGS["verify_t8"]
    idx = _route_case(k3, cfg)
    hot = set(synth.hot_experts(cfg).tolist())
    assert all(e in hot for e in idx.reshape(-1).tolist())


def test_route_ties_lower_index(k3):
    import torch

    E, k, T, d = 64, 8, 4, 64
    x = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((E, d), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(E, dtype=torch.float32, device="cuda")
    b[40:] = 0.5
    idx, wts, _ = k3.k3moe_route(x, w, b, k)
    assert idx.cpu().tolist() == [list(range(40, 48))] * T
    assert np.allclose(wts.cpu().numpy(), 1.0 / k)


@pytest.mark.parametrize("T", [2, 2100])
@pytest.mark.parametrize("case", ["all_equal", "one_tied_per_warp"])
def test_route_ties_wide(k3, case, T):
    """Equal scores at the decode width (896 experts, top-16), both ways each
    top-k kernel can run: all scores equal puts hundreds of keys above the
    maximum bound (bisection in the block kernel, k extraction rounds in the
    warp kernel), one tied expert per warp puts exactly k there (ranked
    directly).  Ties go to the lower index in all four.  T = 2 runs the
    block-per-token kernel, T = 2100 the warp-per-token one."""
    import torch

    E, k, d = 896, 16, 64
    x = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((E, d), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(E, dtype=torch.float32, device="cuda")
    if case == "one_tied_per_warp":
        b[5::32] = 1.0
    idx, wts, _ = k3.k3moe_route(x, w, b, k)
    want = list(range(k)) if case == "all_equal" else [32 * j + 5 for j in range(k)]
    assert idx.cpu().tolist() == [want] * T
    assert np.allclose(wts.cpu().numpy(), 1.0 / k)
    r = oracle.select_experts(np.zeros((T, E)), b.cpu().numpy().astype(np.float32), k)
    assert r["idx"].tolist() == [want] * T


@pytest.mark.parametrize("T", [None, 2100])
def test_route_nonfinite_flag(k3, T):
    import torch

    cfg = synth.CONFIGS["tiny"] if T is None else synth.custom("tiny", T=T)
    dense = synth.dense_inputs(cfg)
    x = to_dev(dense["hidden"], "cuda").clone()
    x[1, 3] = float("nan")
    ws = k3.workspace(k3.k3moe_route_workspace_size(cfg.T, cfg.E))
    k3.k3moe_route(x, to_dev(dense["router_w"], "cuda"), to_dev(dense["router_b"], "cuda"),
                   cfg.k, ws=ws)
    assert k3.k3moe_get_status(ws) == 6
    assert k3.k3moe_get_status(ws) == 0  # cleared by the read


@pytest.mark.parametrize("T,k,E", [(1, 16, 896), (37, 5, 23), (8, 16, 896), (1000, 16, 896),
                                   (200, 2, 8)])
def test_permute_exact(k3, T, k, E):
    import torch

    rng = np.random.default_rng(T * 31 + E)
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    got = k3.k3moe_permute(torch.from_numpy(idx).cuda(), E)
    want = oracle.permute(idx, E)
    for key in ("counts", "offsets", "perm", "inv"):
        assert np.array_equal(got[key].cpu().numpy(), want[key]), key
