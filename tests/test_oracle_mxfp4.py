"""Pins for the oracle's MXFP4 formats (CPU only).

Each check ties the oracle to something other than itself: the OCP E2M1 bit
definition, the value tables and worked result the pages print
(tests/golden/), hand-built byte patterns, and brute force over every code and
exponent.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from conftest import golden


def e2m1_from_bits(code: int) -> float:
    """OCP MX E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0."""
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        return s * 0.5 * m
    return s * 2.0 ** (e - 1) * (1.0 + 0.5 * m)


def test_tables_match_pages_and_bit_definition():
    g = golden("format_tables.json")
    assert oracle.E2M1_MAGNITUDES.tolist() == g["e2m1_magnitudes"]
    assert oracle.GGML_KVALUES.tolist() == g["ggml_kvalues"]
    for c in range(16):
        assert abs(e2m1_from_bits(c)) == oracle.E2M1_MAGNITUDES[c & 7]
        # ggml table = doubled E2M1 with the sign folded in
        assert oracle.GGML_KVALUES[c] == 2 * e2m1_from_bits(c)


def test_nibble_order_low_is_even_element():
    # byte 0x21: element 0 = code 1 (0.5), element 1 = code 2 (1.0)
    packed = np.zeros((1, 16), np.uint8)
    packed[0, 0] = 0x21
    packed[0, 1] = 0xF8  # element 2 = code 8 (-0), element 3 = code 15 (-6)
    scale = np.array([[127]], np.uint8)
    v = oracle.decode_source(packed, scale)
    assert v[0, 0] == 0.5 and v[0, 1] == 1.0
    assert v[0, 2] == 0.0 and math.copysign(1, v[0, 2]) == -1.0
    assert v[0, 3] == -6.0
    assert np.all(v[0, 4:] == 0)


def test_decode_source_exhaustive_codes_and_exponents():
    # every (code, e) with e in 0..254, one code per element: rows = exponents
    es = np.arange(255, dtype=np.uint8)
    codes = np.tile(np.arange(32) % 16, (255, 1)).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    v = oracle.decode_source(packed, es[:, None])
    for e in range(255):
        for j in range(32):
            want = math.ldexp(e2m1_from_bits(j % 16), e - 127)
            assert v[e, j] == want, (e, j)


def test_e8m0_scale_values():
    assert oracle.e8m0_scale(np.array([127]))[0] == 1.0
    assert oracle.e8m0_scale(np.array([128]))[0] == 2.0
    assert oracle.e8m0_scale(np.array([0]))[0] == 2.0 ** -127
    assert oracle.e8m0_scale(np.array([254]))[0] == 2.0 ** 127
    assert np.isnan(oracle.e8m0_scale(np.array([255]))[0])


def test_ggml_half_scale_printed_branch():
    # printed for x >= 2: the float32 whose bits are (x - 1) << 23
    for x in range(2, 255):
        bits = np.array([(x - 1) << 23], np.uint32).view(np.float32)[0]
        assert oracle.ggml_e8m0_half(np.array([x]))[0] == float(bits)
    # x < 2 (not printed): the value that leaves the represented value unchanged
    assert oracle.ggml_e8m0_half(np.array([1]))[0] == 2.0 ** -127
    assert oracle.ggml_e8m0_half(np.array([0]))[0] == 2.0 ** -128


def test_repack_hand_built_block():
    # codes j % 16 over one block: qs[j] = code[j] | code[j+16] << 4 = j | j << 4
    codes = (np.arange(32) % 16).astype(np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)[None, :]
    blk = oracle.repack_ggml(packed, np.array([[121]], np.uint8))
    assert blk.shape == (1, 1, 17)
    assert blk[0, 0, 0] == 121
    assert blk[0, 0, 1:].tolist() == [j | (j << 4) for j in range(16)]
    # a block whose two halves differ: codes 0..15 then 15..0
    codes2 = np.concatenate([np.arange(16), np.arange(15, -1, -1)]).astype(np.uint8)
    packed2 = (codes2[0::2] | (codes2[1::2] << 4)).astype(np.uint8)[None, :]
    blk2 = oracle.repack_ggml(packed2, np.array([[7]], np.uint8))
    assert blk2[0, 0, 1:].tolist() == [j | ((15 - j) << 4) for j in range(16)]


def test_repack_value_equality_exhaustive():
    """The pages' check: kvalues doubled + scale halved leaves every value unchanged,
    for all 16 codes and every exponent 0..254 (x < 2 included)."""
    es = np.arange(255, dtype=np.uint8)
    rng = np.random.default_rng(7)
    packed = rng.integers(0, 256, size=(255, 64), dtype=np.uint8)
    packed[:, :16] = (np.arange(32) % 16)[0::2] | ((np.arange(32) % 16)[1::2] << 4)
    scale = np.repeat(es[:, None], 4, axis=1)
    ref = oracle.decode_source(packed, scale)
    got = oracle.decode_ggml(oracle.repack_ggml(packed, scale))
    assert int((ref != got).sum()) == 0


def test_round_trip_bytes():
    packed = synth.random_bytes(11, 40 * 48).reshape(40, 48)
    scale = synth.random_bytes(12, 40 * 3).reshape(40, 3)
    blocks = oracle.repack_ggml(packed, scale)
    p2, s2 = oracle.unpack_ggml(blocks)
    assert np.array_equal(p2, packed) and np.array_equal(s2, scale)
    # and the other way round on arbitrary blocks
    blk = synth.random_bytes(13, 5 * 7 * 17).reshape(5, 7, 17)
    assert np.array_equal(oracle.repack_ggml(*oracle.unpack_ggml(blk)), blk)


def test_worked_check_counts():
    """Reproduce the printed result of the pages' repack check on a synthetic
    tensor of the same shape and exponent range."""
    g = golden("repack_worked_check.json")
    rows, cols = g["logical_shape"]
    packed = synth.random_bytes(2026, rows * cols // 2).reshape(rows, cols // 2)
    scale = synth.random_exponents(2027, rows * cols // 32, g["e8m0_min"],
                                   g["e8m0_max"]).reshape(rows, cols // 32)
    ref = oracle.decode_source(packed, scale)
    blk = oracle.repack_ggml(packed, scale)
    got = oracle.decode_ggml(blk)
    assert ref.size == g["total_elements"]
    assert int((ref != got).sum()) == g["mismatched_elements"]
    assert float(np.abs(ref - got).max()) == g["max_abs_error"]
    assert packed.nbytes + scale.nbytes == g["bytes_in"]
    assert blk.nbytes == g["bytes_out"]
    assert blk.nbytes * 8 / (rows * cols) == g["bpw"]


def test_negative_zero_code():
    # code 8 is -0 in the source and +0 in ggml: equal as values
    packed = np.full((1, 16), 0x88, np.uint8)
    v_src = oracle.decode_source(packed, np.array([[127]], np.uint8))
    v_ggml = oracle.decode_ggml(oracle.repack_ggml(packed, np.array([[127]], np.uint8)))
    assert np.all(v_src == 0) and np.all(np.signbit(v_src))
    assert np.all(v_ggml == 0) and not np.any(np.signbit(v_ggml))
    assert np.all(v_src == v_ggml)


def test_shape_facts():
    g = golden("k3_shapes.json")
    assert g["moe_layers"] * g["expert_count"] * 3 == g["block_scale_pairs"]
    cfg = synth.CONFIGS["decode_t1"]
    assert (cfg.E, cfg.k, cfg.f, cfg.d) == (g["expert_count"], g["experts_used"],
                                            *g["w1_logical_shape"])
    assert synth.CONFIGS["block_t8192"].D == g["embedding_length"]
    # bytes of one expert matrix = the worked check's bytes in
    rows, cols = cfg.matrix_shape(synth.W1)
    assert rows * cols // 2 + rows * cols // 32 == golden("repack_worked_check.json")["bytes_in"]


def test_bad_shapes_rejected():
    with pytest.raises(ValueError):
        oracle.decode_source(np.zeros((1, 8), np.uint8), np.zeros((1, 1), np.uint8))
