"""MXFP4 formats: the compressed-tensors source layout and the ggml 17-byte block.

Test infrastructure (see the package docstring); float64 throughout.

Source: llama.cpp PR #26185 "model: add Kimi-K3 text model", review by
GrEarl, section "repack_mxfp4_blocks is bit-exact - 0 mismatches over
11,010,048 values" (the format facts and the reproduction script's decode
steps, restated here in my own code).

Source format (compressed-tensors):
  * ``packed[rows, cols // 2]`` uint8: element 2i of a row in the low nibble of
    byte i, element 2i+1 in the high nibble;
  * a nibble is an E2M1 code: bit 3 is the sign, bits 0-2 index the
    magnitudes [0, .5, 1, 1.5, 2, 3, 4, 6];
  * ``scale[rows, cols // 32]`` uint8 E8M0: block b of a row (elements
    32b .. 32b+31) is multiplied by 2**(e - 127).

ggml block (``block_mxfp4``, 17 bytes per 32 elements):
  * byte 0: the E8M0 exponent e, unchanged;
  * bytes 1..16 (``qs``): element j (0..15) in the low nibble of qs[j],
    element j + 16 in the high nibble of qs[j];
  * value = kvalues[code] * 2**(e - 128), kvalues = the E2M1 table doubled
    with the sign folded in: [0,1,2,3,4,6,8,12, 0,-1,-2,-3,-4,-6,-8,-12].
    "kvalues doubled, scale halved": the represented value is unchanged.
"""
from __future__ import annotations

import numpy as np

#: E2M1 magnitudes indexed by the low three bits of a code (page table).
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)

#: ggml ``kvalues_fp4``: doubled E2M1 values with the sign folded in (page table).
GGML_KVALUES = np.array([0, 1, 2, 3, 4, 6, 8, 12, 0, -1, -2, -3, -4, -6, -8, -12],
                        dtype=np.float64)

BLOCK = 32          # elements per E8M0 scale
GGML_BLOCK_BYTES = 17


def source_codes(packed: np.ndarray) -> np.ndarray:
    """Unpack [rows, cols//2] bytes into [rows, cols] 4-bit codes (element 2i = low nibble)."""
    packed = np.asarray(packed, dtype=np.uint8)
    rows, half = packed.shape
    codes = np.empty((rows, 2 * half), dtype=np.uint8)
    codes[:, 0::2] = packed & 0x0F
    codes[:, 1::2] = packed >> 4
    return codes


def e8m0_scale(e: np.ndarray) -> np.ndarray:
    """Source scale: 2**(e - 127) for e in 0..254; e = 255 is NaN (OCP MX).

    The pages give 2**(e - 127); e = 255 is never produced by the generators.
    """
    e = np.asarray(e).astype(np.int64)
    out = np.ldexp(1.0, e - 127)
    return np.where(e == 255, np.nan, out)


def decode_source(packed: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Decode a compressed-tensors MXFP4 matrix to float64 [rows, cols]."""
    codes = source_codes(packed)
    rows, cols = codes.shape
    if cols % BLOCK:
        raise ValueError("cols must be a multiple of 32")
    mag = E2M1_MAGNITUDES[codes & 7]
    val = np.where((codes & 8) != 0, -mag, mag)
    sc = e8m0_scale(np.asarray(scale).reshape(rows, cols // BLOCK))
    return (val.reshape(rows, cols // BLOCK, BLOCK) * sc[:, :, None]).reshape(rows, cols)


def repack_ggml(packed: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Source (packed, scale) -> ggml blocks uint8 [rows, cols // 32, 17].

    Byte 0 keeps e as stored (the halving lives in the ggml decode); byte 1+j
    holds element j in the low nibble and element j + 16 in the high nibble.
    """
    codes = source_codes(packed)
    rows, cols = codes.shape
    nb = cols // BLOCK
    c = codes.reshape(rows, nb, BLOCK)
    out = np.empty((rows, nb, GGML_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0] = np.asarray(scale, dtype=np.uint8).reshape(rows, nb)
    out[:, :, 1:] = c[:, :, :16] | (c[:, :, 16:] << 4)
    return out


def unpack_ggml(blocks: np.ndarray):
    """ggml blocks [rows, nb, 17] -> (packed [rows, nb*16], scale [rows, nb]); inverse of repack."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    rows, nb, _ = blocks.shape
    scale = blocks[:, :, 0].copy()
    qs = blocks[:, :, 1:]
    codes = np.empty((rows, nb, BLOCK), dtype=np.uint8)
    codes[:, :, :16] = qs & 0x0F
    codes[:, :, 16:] = qs >> 4
    codes = codes.reshape(rows, nb * BLOCK)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scale


def ggml_e8m0_half(x: np.ndarray) -> np.ndarray:
    """ggml's half scale, 2**(x - 128).

    The page prints only the x >= 2 branch (the float with bit pattern
    (x - 1) << 23, i.e. 2**(x - 128)).  Reading for x < 2 (not printed): the
    same value 2**(x - 128), a float32 subnormal, which is the only choice that
    keeps the represented value unchanged after the repack.
    """
    x = np.asarray(x).astype(np.int64)
    return np.ldexp(1.0, x - 128)


def decode_ggml(blocks: np.ndarray) -> np.ndarray:
    """Decode ggml MXFP4 blocks [rows, nb, 17] to float64 [rows, nb*32]."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    rows, nb, _ = blocks.shape
    qs = blocks[:, :, 1:]
    out = np.empty((rows, nb, BLOCK), dtype=np.float64)
    out[:, :, :16] = GGML_KVALUES[qs & 0x0F]
    out[:, :, 16:] = GGML_KVALUES[qs >> 4]
    out *= ggml_e8m0_half(blocks[:, :, 0])[:, :, None]
    return out.reshape(rows, nb * BLOCK)
