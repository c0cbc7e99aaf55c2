"""GPU parity of the streaming kernels on llama.cpp's MXFP4 blocks
(descriptor format K3MOE_FORMAT_GGML: 17 bytes per 32 inputs, the E8M0 byte
then element j in the low and element j + 16 in the high nibble of byte j;
llama.cpp PR #26185, review by GrEarl, "repack_mxfp4_blocks is bit-exact").

The kernels convert the blocks in shared memory to the operands the split
(compressed-tensors) format feeds the tensor cores, so the output must be
bitwise that of the split format on the same weights.  The first call is
also compared with the layer oracle run on the ggml bytes themselves (each
expert decoded by the oracle's own unpack of the blocks): max |err| <= 1e-2
x row RMS + half a bf16 ulp.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import bf16_tensor_to_np, make_layer, oracle_forward, rel_err_rows, to_dev

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


def layers(k3, cfg):
    layer, dense, expert, _ = make_layer(cfg, on_device_experts=False)
    return layer, k3.ggml_layer(layer), dense


def ggml_expert(k3, glayer):
    """Oracle accessor: expert e of matrix m from the device blocks, unpacked by the oracle."""
    names = ("w1_q", "w3_q", "w2_q")
    cache = {}

    def expert(m, e):
        if (m, e) not in cache:
            blocks = glayer.tensors[names[m]][e].cpu().numpy()
            cache[(m, e)] = oracle.unpack_ggml(blocks)
        return cache[(m, e)]

    return expert


def run(k3, cfg, layer, glayer, dense, T, n, seed, check_oracle=True):
    import torch

    big = synth.custom(cfg.name, T=T * n, E=cfg.E, k=cfg.k, d=cfg.d, f=cfg.f, D=cfg.D, seed_index=seed)
    xs = synth.hidden(big).reshape(n, T, -1)
    ws_g = k3.workspace(k3.k3moe_workspace_size(glayer, T))
    ws_s = k3.workspace(k3.k3moe_workspace_size(layer, T))
    for i in range(n):
        x = to_dev(xs[i], "cuda")
        got = k3.k3moe_forward(glayer, x, ws=ws_g)
        ref = k3.k3moe_forward(layer, x, ws=ws_s)
        assert k3.k3moe_get_status(ws_g) == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"batch {i}"
        if i == 0 and check_oracle:
            o = oracle_forward(cfg, dict(dense, hidden=xs[0]), ggml_expert(k3, glayer))
            idx, _, _ = k3.k3moe_forward_routing(glayer, ws_g, T)
            same = np.all(o["idx"] == idx.cpu().numpy(), axis=1)
            assert np.all(same | (o["margin"] < 1e-5))
            err = rel_err_rows(bf16_tensor_to_np(got)[same], o["out"][same])
            assert np.all(err <= 1e-2), err.max()


@pytest.fixture(scope="module")
def small(k3):
    cfg = synth.custom("decode_t1", T=1, E=64, k=4, d=512, f=512)
    return (cfg,) + layers(k3, cfg)


@pytest.mark.parametrize("T", [1, 2, 5, 8, 20, 64])
def test_ggml_small(k3, small, T):
    cfg, layer, glayer, dense = small
    run(k3, cfg, layer, glayer, dense, T, n=3, seed=200 + T)


def test_ggml_blocks_are_the_oracle_repack(k3, small):
    """The bytes the kernels read are the oracle's repack of the source expert."""
    cfg, layer, glayer, _ = small
    for m, name in enumerate(synth.MATRIX_NAMES):
        for e in (0, cfg.E - 1):
            q, s = synth.expert_matrix_np(cfg, m, e)
            want = oracle.repack_ggml(q, s)
            assert np.array_equal(glayer.tensors[name + "_q"][e].cpu().numpy(), want)


@pytest.mark.parametrize("T", [1, 8, 24])
def test_ggml_k3_shapes(k3, T):
    """The K3 widths (d = 3584, f = 3072: 7 and 6 stages of 16 blocks per row)."""
    cfg = synth.custom("decode_t1", T=1, E=32, k=8)
    run(k3, cfg, *layers(k3, cfg), T=T, n=2, seed=300 + T, check_oracle=(T == 1))


def test_ggml_rejections(k3, small):
    cfg, layer, glayer, _ = small
    import torch

    x = torch.zeros((2000, cfg.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(k3.K3MoEError) as ex:  # beyond the streaming kernels
        k3.k3moe_forward(glayer, x)
    assert ex.value.status == 8
    cache = k3.ExpertCache(layer, 8)
    with pytest.raises(k3.K3MoEError) as ex:  # no expert cache over ggml blocks
        k3.k3moe_forward_cached(glayer, cache, x[:1])
    assert ex.value.status == 8


@pytest.mark.parametrize("T", [1, 6, 12])
def test_ggml_block_mode(k3, T):
    """The full latent block over ggml blocks: bitwise the split-layout block."""
    cfg = synth.custom("block_t8192", T=T, E=32, k=4, d=512, f=512, D=1024, seed_index=29)
    layer, glayer, dense = layers(k3, cfg)
    run(k3, cfg, layer, glayer, dense, T, n=2, seed=400 + T, check_oracle=False)
