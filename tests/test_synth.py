"""The seeded input generators: NumPy and PyTorch SplitMix64 agree; recipe facts."""
import numpy as np
import pytest

import synth


def test_splitmix64_reference_value():
    # first output of SplitMix64 seeded with 0 (published test value)
    assert int(synth.words_np(0, 1)[0]) == 0xE220A8397B1DCDAF
    assert synth.mix64(synth.GAMMA) == 0xE220A8397B1DCDAF


def test_numpy_and_torch_expert_bytes_agree():
    torch = pytest.importorskip("torch")
    cfg = synth.custom("decode_t1", E=2, d=256, f=128)
    ex = synth.experts_torch(cfg, "cpu")
    for m, name in enumerate(synth.MATRIX_NAMES):
        for e in range(cfg.E):
            q, s = synth.expert_matrix_np(cfg, m, e)
            assert np.array_equal(q, ex[name + "_q"][e].numpy())
            assert np.array_equal(s, ex[name + "_s"][e].numpy())
            assert s.min() >= cfg.e_lo and s.max() <= cfg.e_hi


def test_tiny_recipe():
    cfg = synth.CONFIGS["tiny"]
    d = synth.dense_inputs(cfg)
    assert d["hidden"].shape == (4, 64) and d["hidden"].dtype == np.uint16
    assert d["router_w"].shape == (8, 64)
    ex = synth.experts_np(cfg)
    assert ex["w1_q"].shape == (8, 64, 32) and ex["w2_s"].shape == (8, 64, 2)


def test_hot_bias_recipe():
    cfg = synth.CONFIGS["verify_t8"]
    b = synth.router_bias(cfg)
    hot = synth.hot_experts(cfg)
    assert len(hot) == 32 and np.all(b[hot] == 1.0)
    assert np.sum(b == 1.0) == 32


def test_bf16_rounding_helper_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f32_to_bf16_bits(x), want)
