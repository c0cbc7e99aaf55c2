"""Pins for the oracle's expert FFN, MoE layer and latent block (CPU only)."""
import math

import numpy as np
import pytest

import oracle
import synth

E2M1_CODE = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}


def encode_exact(mat: np.ndarray):
    """Hand encoding of a matrix whose entries are +-E2M1 magnitudes (scale 2**0)."""
    rows, cols = mat.shape
    codes = np.zeros((rows, cols), np.uint8)
    for (r, c), v in np.ndenumerate(mat):
        codes[r, c] = E2M1_CODE[abs(v)] | (8 if v < 0 else 0)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, np.full((rows, cols // 32), 127, np.uint8)


def test_silu_closed_forms():
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(oracle.silu(np.array([-30.0]))[0]) < 1e-11


def test_expert_ffn_hand_example_catches_transposes_and_swaps():
    # d = f = 32, sparse weights; x = e0 + 2 e1
    d = f = 32
    x = np.zeros((1, d))
    x[0, 0], x[0, 1] = 1.0, 2.0
    w1 = np.zeros((f, d)); w1[0, 1] = 1.0          # g0 = x1 = 2
    w3 = np.zeros((f, d)); w3[0, 0] = 3.0; w3[1, 1] = 1.0   # u0 = 3, u1 = 2
    w2 = np.zeros((d, f)); w2[1, 0] = 1.0          # y1 = h0
    y = oracle.expert_ffn(x, w1, w3, w2)
    want = np.zeros(d); want[1] = 3.0 * 2.0 / (1.0 + math.exp(-2.0))
    assert np.allclose(y[0], want, atol=1e-15, rtol=0)
    # the same through the MXFP4 encoding and the MoE layer (one expert, k = 1)
    mats = {0: encode_exact(w1), 1: encode_exact(w3), 2: encode_exact(w2)}
    r = oracle.moe_forward(x, np.zeros((1, d)), np.zeros(1), 1, x, lambda m, e: mats[m])
    assert r["idx"].tolist() == [[0]] and r["w"][0, 0] == 1.0
    assert np.allclose(r["out"][0], want, atol=1e-15, rtol=0)


def tiny_layer():
    cfg = synth.CONFIGS["tiny"]
    ex = synth.experts_np(cfg)
    dense = synth.dense_inputs(cfg)
    names = synth.MATRIX_NAMES
    expert = lambda m, e: (ex[names[m] + "_q"][e], ex[names[m] + "_s"][e])
    x = oracle.bf16_to_f64(dense["hidden"])
    wr = oracle.bf16_to_f64(dense["router_w"])
    return cfg, ex, dense, expert, x, wr


def test_tiny_sparse_equals_dense_loop_over_all_experts():
    cfg, ex, dense, expert, x, wr = tiny_layer()
    r = oracle.moe_forward(x, wr, dense["router_b"], cfg.k, x, expert)
    # brute force: every expert on every token, gate zero outside the selection
    out = np.zeros_like(x)
    for t in range(cfg.T):
        logits = [sum(x[t, i] * wr[e, i] for i in range(cfg.d)) for e in range(cfg.E)]
        s = [1.0 / (1.0 + math.exp(-l)) for l in logits]
        beta = [s[e] + float(dense["router_b"][e]) for e in range(cfg.E)]
        chosen = sorted(range(cfg.E), key=lambda e: (-beta[e], e))[: cfg.k]
        norm = sum(s[e] for e in chosen)
        for e in range(cfg.E):
            gate = s[e] / norm if e in chosen else 0.0
            w1 = oracle.decode_source(*expert(0, e))
            w3 = oracle.decode_source(*expert(1, e))
            w2 = oracle.decode_source(*expert(2, e))
            g = w1 @ x[t]
            u = w3 @ x[t]
            h = g / (1.0 + np.exp(-g)) * u
            out[t] += gate * (w2 @ h)
    scale = np.sqrt(np.mean(out ** 2))
    assert np.max(np.abs(out - r["out"])) <= 1e-12 * scale


def test_tiny_has_small_exponent_blocks():
    cfg, ex, *_ = tiny_layer()
    for name in synth.MATRIX_NAMES:
        s = ex[name + "_s"]
        assert (s == 0).sum() == 1 and (s == 1).sum() == 1
        assert ((s >= 119) & (s <= 123)).sum() == s.size - 2


def test_k_equals_E_is_dense_gated_mlp():
    cfg, ex, dense, expert, x, wr = tiny_layer()
    r = oracle.moe_forward(x, wr, dense["router_b"], cfg.E, x, expert)
    s = oracle.sigmoid(x @ wr.T)
    out = np.zeros_like(x)
    for e in range(cfg.E):
        W = [oracle.decode_source(*expert(m, e)) for m in range(3)]
        out += (s[:, e] / s.sum(1))[:, None] * oracle.expert_ffn(x, *W)
    assert np.max(np.abs(out - r["out"])) <= 1e-12 * np.sqrt(np.mean(out ** 2))


def test_power_of_two_invariant_exact():
    cfg, ex, dense, expert, x, wr = tiny_layer()
    names = synth.MATRIX_NAMES

    def expert2(m, e):
        q, s = expert(m, e)
        return (q, s + 1) if m == 2 else (q, s)

    a = oracle.moe_forward(x, wr, dense["router_b"], cfg.k, x, expert)["out"]
    b = oracle.moe_forward(x, wr, dense["router_b"], cfg.k, x, expert2)["out"]
    assert np.array_equal(b, 2 * a)


def test_idx_override_recomputes_weights_from_scores():
    cfg, ex, dense, expert, x, wr = tiny_layer()
    r = oracle.moe_forward(x, wr, dense["router_b"], cfg.k, x, expert)
    other = np.array([[0, 1]] * cfg.T)
    r2 = oracle.moe_forward(x, wr, dense["router_b"], cfg.k, x, expert, idx=other)
    s = r["s"]
    assert np.allclose(r2["w"], s[:, :2] / s[:, :2].sum(1, keepdims=True), rtol=0, atol=1e-15)


def test_rmsnorm_closed_forms():
    h = np.full((2, 8), -3.0)
    gamma = np.arange(1, 9, dtype=np.float64)
    y = oracle.rmsnorm(h, gamma, 1e-5)
    assert np.allclose(y, -3.0 / math.sqrt(9.0 + 1e-5) * gamma, rtol=1e-15, atol=0)
    rng = np.random.default_rng(1)
    h = rng.standard_normal((3, 16))
    assert np.allclose(oracle.rmsnorm(5.0 * h, np.ones(16), 0.0),
                       oracle.rmsnorm(h, np.ones(16), 0.0), rtol=1e-14)


def test_round_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-39).astype(np.float32),   # float32 subnormals
        np.array([3.3895314e38, 3.4e38, -3.39e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8,
                  2 ** -126, 2 ** -133, 2 ** -134, 3 * 2 ** -135, 0.0, -0.0], np.float32),
    ])
    want = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(vals.astype(np.float64))
    same = (got == want) | (np.isinf(got) & np.isinf(want) & (np.sign(got) == np.sign(want)))
    assert np.all(same), vals[~same]


def test_block_forward_reduces_to_moe_with_identity_projections():
    cfg, ex, dense, expert, x, wr = tiny_layer()
    D, d = 2 * cfg.d, cfg.d
    rng = np.random.default_rng(8)
    h = oracle.round_bf16(rng.standard_normal((cfg.T, D)))
    w_down = np.zeros((d, D)); w_down[:, :d] = np.eye(d)
    w_up = np.zeros((D, d)); w_up[:d, :] = np.eye(d)
    wr_full = np.zeros((cfg.E, D)); wr_full[:, :d] = wr
    r = oracle.block_forward(h, np.ones(D), 1e-5, w_down, w_up, wr_full, dense["router_b"],
                             cfg.k, expert)
    hn = oracle.round_bf16(oracle.rmsnorm(h, np.ones(D), 1e-5))
    m = oracle.moe_forward(hn[:, :d], wr, dense["router_b"], cfg.k, hn[:, :d], expert)
    assert np.array_equal(r["idx"], m["idx"])
    assert np.array_equal(r["out"][:, :d], oracle.round_bf16(m["out"]))
    assert np.all(r["out"][:, d:] == 0)
