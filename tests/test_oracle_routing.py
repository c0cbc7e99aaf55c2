"""Pins for the oracle's router and permutation (CPU only)."""
import itertools
import math

import numpy as np

import oracle
import synth


def test_sigmoid_closed_forms():
    assert oracle.sigmoid(np.array([0.0]))[0] == 0.5
    assert abs(oracle.sigmoid(np.array([math.log(3.0)]))[0] - 0.75) < 1e-15
    l = np.linspace(-20, 20, 101)
    assert np.allclose(oracle.sigmoid(l) + oracle.sigmoid(-l), 1.0, atol=1e-15)


def test_logits_identity_weights():
    x = np.arange(12, dtype=np.float64).reshape(3, 4)
    assert np.array_equal(oracle.router_logits(x, np.eye(4)), x)
    w = np.array([[1.0, 0, 0, 0], [0, 0, 2.0, 0]])
    assert np.array_equal(oracle.router_logits(x, w), np.stack([x[:, 0], 2 * x[:, 2]], 1))


def test_selection_hand_example_bias_selects_weights_unbiased():
    # s = [0.5, 0.75, 0.25], bias lifts expert 2 to the top
    logits = np.array([[0.0, math.log(3.0), -math.log(3.0)]])
    r = oracle.select_experts(logits, np.array([0.0, 0.0, 10.0]), 2)
    assert r["idx"].tolist() == [[2, 1]]
    assert np.allclose(r["w"], [[0.25, 0.75]], atol=1e-15)


def test_selection_ties_go_to_lower_index():
    r = oracle.select_experts(np.zeros((2, 6)), np.zeros(6), 3)
    assert r["idx"].tolist() == [[0, 1, 2], [0, 1, 2]]
    assert np.allclose(r["w"], 1.0 / 3)
    # equal beta from different (s, b) splits: still index order
    l = np.array([[0.0, 0.0, 0.0]])
    r = oracle.select_experts(l, np.array([0.1, 0.3, 0.3]), 2)
    assert r["idx"].tolist() == [[1, 2]]


def brute_force_topk(beta_row, k):
    """Python tuple sort over (-beta, index): the definition written out."""
    keyed = sorted(((-b, i) for i, b in enumerate(beta_row)))
    return [i for _, i in keyed[:k]]


def test_selection_brute_force_and_lexsort():
    cfg = synth.CONFIGS["tiny"]
    rng = np.random.default_rng(5)
    for trial in range(50):
        E = int(rng.integers(2, 12))
        k = int(rng.integers(1, E + 1))
        l = rng.standard_normal((3, E))
        if trial % 3 == 0:  # force exact ties
            l = np.round(l)
        b = np.round(rng.standard_normal(E) * 0.1, 1)
        r = oracle.select_experts(l, b, k)
        beta = oracle.sigmoid(l) + b
        for t in range(3):
            assert r["idx"][t].tolist() == brute_force_topk(beta[t], k)
            # library special case: lexsort with the index as the secondary key
            lex = np.lexsort((np.arange(E), -beta[t]))[:k]
            assert r["idx"][t].tolist() == lex.tolist()
            # every selected beta >= every unselected beta
            sel = set(r["idx"][t].tolist())
            uns = [beta[t, e] for e in range(E) if e not in sel]
            if uns:
                assert min(beta[t, list(sel)]) >= max(uns)
            assert abs(r["w"][t].sum() - 1.0) < 1e-12
            assert np.all(r["w"][t] > 0)
    assert cfg.k <= cfg.E


def test_selection_subset_enumeration_tiny():
    """Top-k set = the k-subset with the largest sum of beta (distinct betas)."""
    rng = np.random.default_rng(9)
    l = rng.standard_normal((4, 8))
    b = rng.standard_normal(8) * 0.01
    r = oracle.select_experts(l, b, 2)
    beta = oracle.sigmoid(l) + b
    for t in range(4):
        best = max(itertools.combinations(range(8), 2), key=lambda c: beta[t, list(c)].sum())
        assert sorted(best) == sorted(r["idx"][t].tolist())


def test_margin():
    l = np.array([[0.0, 1.0, 2.0, 3.0]])
    r = oracle.select_experts(l, np.zeros(4), 2)
    s = oracle.sigmoid(l[0])
    assert abs(r["margin"][0] - (s[2] - s[1])) < 1e-15
    assert np.isinf(oracle.select_experts(l, np.zeros(4), 4)["margin"][0])


def test_permute_hand_example():
    # pairs: p0=(t0,j0)->e2, p1=(t0,j1)->e0, p2=(t1,j0)->e0, p3=(t1,j1)->e1
    p = oracle.permute(np.array([[2, 0], [0, 1]]), 3)
    assert p["counts"].tolist() == [2, 1, 1]
    assert p["offsets"].tolist() == [0, 2, 3, 4]
    assert p["perm"].tolist() == [1, 2, 3, 0]
    assert p["inv"].tolist() == [3, 0, 1, 2]


def test_permute_invariants_random():
    rng = np.random.default_rng(3)
    T, k, E = 37, 5, 23
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    p = oracle.permute(idx, E)
    assert p["counts"].sum() == T * k
    assert np.array_equal(p["offsets"][1:], np.cumsum(p["counts"]))
    assert sorted(p["perm"].tolist()) == list(range(T * k))
    assert np.array_equal(p["inv"][p["perm"]], np.arange(T * k))
    flat = idx.reshape(-1)
    for e in range(E):
        rows = p["perm"][p["offsets"][e]:p["offsets"][e + 1]]
        assert np.all(flat[rows] == e)
        assert np.all(np.diff(rows // k) > 0)  # ascending tokens


def test_bf16_to_f64_hand_bit_patterns():
    """bf16 is the top half of an IEEE binary32: sign bit 15, 8 exponent bits
    (bias 127), 7 mantissa bits.  Values worked out by hand from that
    definition; a shift or mask error in the widening fails one of them."""
    cases = {
        0x3F80: 1.0,                     # exponent 127, mantissa 0
        0xC000: -2.0,                    # sign, exponent 128
        0x4049: 3.140625,                # 2 * (1 + 73/128)
        0x3F81: 1.0 + 2.0 ** -7,         # lowest mantissa bit
        0x0080: 2.0 ** -126,             # smallest normal
        0x0001: 2.0 ** -133,             # smallest subnormal: 2^-126 * 2^-7
        0x007F: 127 * 2.0 ** -133,       # largest subnormal
        0x7F7F: (2.0 - 2.0 ** -7) * 2.0 ** 127,  # largest finite
        0x0000: 0.0,
    }
    bits = np.array(list(cases), dtype=np.uint16)
    got = oracle.bf16_to_f64(bits)
    assert got.tolist() == list(cases.values())
    neg0 = oracle.bf16_to_f64(np.array([0x8000], np.uint16))[0]
    assert neg0 == 0.0 and math.copysign(1.0, neg0) == -1.0
    inf = oracle.bf16_to_f64(np.array([0x7F80, 0xFF80], np.uint16))
    assert inf.tolist() == [math.inf, -math.inf]
    assert math.isnan(oracle.bf16_to_f64(np.array([0x7FC0], np.uint16))[0])
