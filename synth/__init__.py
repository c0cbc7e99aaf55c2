"""Seeded synthetic inputs for the latent routed-expert MXFP4 MoE layer.

This module holds random draws only: no step of the layer's arithmetic lives
here.  It is the one piece of code that both the CPU oracle (``oracle/``) and
the CUDA path (through the tests and ``bench.py``) use.

Two generators are used:

* Small dense tensors (hidden states, router weights, bias, RMSNorm gain,
  latent projections) come from NumPy's PCG64, seeded by
  ``SeedSequence([config_seed, tag])``, drawn in float64, cast to float32 and
  rounded to bf16 (round-to-nearest-even).  bf16 tensors are carried as their
  uint16 bit patterns.

* Expert bytes (MXFP4 nibbles and E8M0 scales, 15.7 GB for 896 experts) come
  from SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): word j of a stream with seed s is
  ``mix64(s + (j + 1) * 0x9E3779B97F4A7C15 mod 2**64)``.  Because the
  generator is counter-based, any single expert can be regenerated alone (the
  oracle does this on the host with NumPy) and the whole weight set can be
  generated directly in device memory (the tests and the benchmark do this
  with PyTorch integer ops).  Both implementations are written here, from the
  published definition, and are checked against each other on CPU.

Byte layout of one expert matrix with logical shape [rows, cols] (rows =
outputs, cols = inputs): ``packed[rows, cols // 2]`` (two E2M1 codes per byte,
element 2i in the low nibble) and ``scale[rows, cols // 32]`` (one E8M0 byte
per run of 32 inputs).  Nibble bytes are the little-endian bytes of the
stream's words; scale byte j is ``e_lo + (word_j >> 32) % (e_hi - e_lo + 1)``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

# matrix ids of one expert
W1, W3, W2 = 0, 1, 2
MATRIX_NAMES = ("w1", "w3", "w2")

_TAG_NIBBLES = 1
_TAG_SCALES = 2


# --------------------------------------------------------------------------
# SplitMix64
# --------------------------------------------------------------------------
def mix64(z: int) -> int:
    """SplitMix64 output function on a Python int (mod 2**64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def stream_seed(*parts: int) -> int:
    """Derive a 64-bit stream seed from integer parts (config seed, tags, ids)."""
    h = 0
    for p in parts:
        h = mix64((h ^ (int(p) & MASK64)) + GAMMA)
    return h


def words_np(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Words start..start+n-1 of the SplitMix64 stream ``seed`` as uint64."""
    with np.errstate(over="ignore"):
        j = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(seed & MASK64) + j * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
        z = z ^ (z >> np.uint64(31))
    return z


def _signed64(u: int) -> int:
    u &= MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


def words_torch(seeds, n: int, device):
    """SplitMix64 words for a batch of streams, as int64 [len(seeds), n].

    Integer multiply wraps mod 2**64 in PyTorch's int64 kernels on both CPU and
    CUDA; right shifts are arithmetic, so they are masked into logical shifts.
    """
    import torch

    s = torch.tensor([_signed64(x) for x in seeds], dtype=torch.int64, device=device)
    j = torch.arange(1, n + 1, dtype=torch.int64, device=device)
    z = s[:, None] + j[None, :] * _signed64(GAMMA)
    z = (z ^ ((z >> 30) & ((1 << 34) - 1))) * _signed64(_M1)
    z = (z ^ ((z >> 27) & ((1 << 37) - 1))) * _signed64(_M2)
    z = z ^ ((z >> 31) & ((1 << 33) - 1))
    return z


# --------------------------------------------------------------------------
# configurations
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    T: int            # tokens
    E: int            # routed experts
    k: int            # experts used per token
    d: int            # latent width (expert input/output)
    f: int            # expert hidden width
    e_lo: int         # E8M0 exponent range (inclusive)
    e_hi: int
    router_std: float
    bias: str         # "normal", "hot", "zipf"
    bias_std: float
    D: int = 0        # full model width (block mode only)
    seed_index: int = 0
    n_hot: int = 0
    force_small_exponents: bool = False

    @property
    def seed(self) -> int:
        return 20260000 + self.seed_index

    @property
    def block(self) -> bool:
        return self.D > 0

    @property
    def d_router(self) -> int:
        return self.D if self.block else self.d

    def matrix_shape(self, m: int):
        """Logical [rows, cols] of expert matrix m."""
        return (self.f, self.d) if m in (W1, W3) else (self.d, self.f)


CONFIGS = {
    "tiny": Config("tiny", T=4, E=8, k=2, d=64, f=64, e_lo=119, e_hi=123,
                   router_std=1.0 / 8.0, bias="normal", bias_std=0.01, seed_index=0,
                   force_small_exponents=True),
    "decode_t1": Config("decode_t1", T=1, E=896, k=16, d=3584, f=3072, e_lo=120, e_hi=122,
                        router_std=1.0 / math.sqrt(3584), bias="normal", bias_std=0.05,
                        seed_index=1),
    "verify_t8": Config("verify_t8", T=8, E=896, k=16, d=3584, f=3072, e_lo=120, e_hi=122,
                        router_std=1.0 / math.sqrt(3584), bias="hot", bias_std=0.05,
                        seed_index=2, n_hot=32),
    "chunk_t512": Config("chunk_t512", T=512, E=896, k=16, d=3584, f=3072, e_lo=120, e_hi=122,
                         router_std=1.0 / math.sqrt(3584), bias="normal", bias_std=0.05,
                         seed_index=3),
    "block_t8192": Config("block_t8192", T=8192, E=896, k=16, d=3584, f=3072, e_lo=120,
                          e_hi=122, router_std=1.0 / math.sqrt(7168), bias="zipf",
                          bias_std=0.05, D=7168, seed_index=4),
}
CONFIG_ORDER = ["tiny", "decode_t1", "verify_t8", "chunk_t512", "block_t8192"]


def custom(base: str, **over) -> Config:
    """A config derived from a named one (other T, E, k, shapes, seed)."""
    return dataclasses.replace(CONFIGS[base], **over)


# --------------------------------------------------------------------------
# dense draws (host)
# --------------------------------------------------------------------------
def _rng(cfg: Config, tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([cfg.seed, tag])))


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(cfg: Config, tag: int, shape, std: float) -> np.ndarray:
    x = _rng(cfg, tag).standard_normal(size=shape) * std
    return f32_to_bf16_bits(x.astype(np.float32))


def hidden(cfg: Config) -> np.ndarray:
    """Layer input as bf16 bits: [T, d] latent, or [T, D] in block mode; N(0,1)."""
    width = cfg.D if cfg.block else cfg.d
    return _normal_bf16(cfg, 10, (cfg.T, width), 1.0)


def router_weight(cfg: Config) -> np.ndarray:
    """Router weight [E, d_router] as bf16 bits, N(0, router_std)."""
    return _normal_bf16(cfg, 11, (cfg.E, cfg.d_router), cfg.router_std)


def router_bias(cfg: Config) -> np.ndarray:
    """Selection bias [E] float32."""
    g = _rng(cfg, 12)
    noise = g.standard_normal(cfg.E) * cfg.bias_std
    if cfg.bias == "normal":
        b = noise
    elif cfg.bias == "hot":
        hot = g.permutation(cfg.E)[: cfg.n_hot]
        b = noise.copy()
        b[hot] = 1.0
    elif cfg.bias == "zipf":
        rank = g.permutation(cfg.E)  # rank[e] = popularity rank of expert e
        b = 0.1 * (-1.1 * np.log(rank + 1.0)) + noise
    else:
        raise ValueError(cfg.bias)
    return b.astype(np.float32)


def hot_experts(cfg: Config) -> np.ndarray:
    """Experts given the +1.0 bias in the "hot" recipe (sorted)."""
    g = _rng(cfg, 12)
    g.standard_normal(cfg.E)
    return np.sort(g.permutation(cfg.E)[: cfg.n_hot])


def norm_gamma(cfg: Config) -> np.ndarray:
    """RMSNorm gain [D] as bf16 bits, U(0.5, 1.5)."""
    return f32_to_bf16_bits(_rng(cfg, 13).uniform(0.5, 1.5, cfg.D).astype(np.float32))


def w_down(cfg: Config) -> np.ndarray:
    """Latent down-projection [d, D] bf16 bits, N(0, 1/sqrt(D))."""
    return _normal_bf16(cfg, 14, (cfg.d, cfg.D), 1.0 / math.sqrt(cfg.D))


def w_up(cfg: Config) -> np.ndarray:
    """Latent up-projection [D, d] bf16 bits, N(0, 1/sqrt(d))."""
    return _normal_bf16(cfg, 15, (cfg.D, cfg.d), 1.0 / math.sqrt(cfg.d))


RMS_EPS = 1e-5


# --------------------------------------------------------------------------
# expert bytes
# --------------------------------------------------------------------------
def _nibble_seed(cfg: Config, m: int, e: int) -> int:
    return stream_seed(cfg.seed, _TAG_NIBBLES, m, e)


def _scale_seed(cfg: Config, m: int, e: int) -> int:
    return stream_seed(cfg.seed, _TAG_SCALES, m, e)


def _forced_blocks(cfg: Config, m: int):
    """(expert, row, block, exponent) overrides for the tiny config: one block
    per matrix gets E8M0 = 1 and another gets E8M0 = 0."""
    if not cfg.force_small_exponents:
        return []
    rows, cols = cfg.matrix_shape(m)
    nb = cols // 32
    out = []
    for i, ev in enumerate((1, 0)):
        w = int(words_np(stream_seed(cfg.seed, 3, m, i), 1)[0])
        e = w % cfg.E
        r = (w >> 16) % rows
        b = (w >> 40) % nb
        out.append((e, r, b, ev))
    if out[0][:3] == out[1][:3]:  # keep the two blocks distinct
        e, r, b, ev = out[1]
        out[1] = (e, r, (b + 1) % nb, ev)
    return out


def expert_matrix_np(cfg: Config, m: int, e: int):
    """(packed [rows, cols//2] uint8, scale [rows, cols//32] uint8) of matrix m of expert e."""
    rows, cols = cfg.matrix_shape(m)
    nbytes = rows * cols // 2
    nw = (nbytes + 7) // 8
    packed = words_np(_nibble_seed(cfg, m, e), nw).view(np.uint8)[:nbytes].reshape(rows, cols // 2)
    ns = rows * (cols // 32)
    span = cfg.e_hi - cfg.e_lo + 1
    sw = words_np(_scale_seed(cfg, m, e), ns)
    scale = (cfg.e_lo + (sw >> np.uint64(32)) % np.uint64(span)).astype(np.uint8)
    scale = scale.reshape(rows, cols // 32)
    for (fe, r, b, ev) in _forced_blocks(cfg, m):
        if fe == e:
            scale[r, b] = ev
    return np.ascontiguousarray(packed), np.ascontiguousarray(scale)


def experts_np(cfg: Config):
    """All expert bytes on the host: dict name -> array [E, ...] (small configs)."""
    out = {}
    for m, name in enumerate(MATRIX_NAMES):
        qs, ss = zip(*(expert_matrix_np(cfg, m, e) for e in range(cfg.E)))
        out[name + "_q"] = np.stack(qs)
        out[name + "_s"] = np.stack(ss)
    return out


def experts_torch(cfg: Config, device, chunk: int = 16):
    """All expert bytes generated in place on ``device`` (same bytes as experts_np)."""
    import torch

    out = {}
    span = cfg.e_hi - cfg.e_lo + 1
    for m, name in enumerate(MATRIX_NAMES):
        rows, cols = cfg.matrix_shape(m)
        nbytes = rows * cols // 2
        nw = (nbytes + 7) // 8
        ns = rows * (cols // 32)
        q = torch.empty((cfg.E, rows, cols // 2), dtype=torch.uint8, device=device)
        s = torch.empty((cfg.E, rows, cols // 32), dtype=torch.uint8, device=device)
        for e0 in range(0, cfg.E, chunk):
            e1 = min(cfg.E, e0 + chunk)
            w = words_torch([_nibble_seed(cfg, m, e) for e in range(e0, e1)], nw, device)
            q[e0:e1] = w.view(torch.uint8).reshape(e1 - e0, nw * 8)[:, :nbytes].reshape(
                e1 - e0, rows, cols // 2)
            del w
            w = words_torch([_scale_seed(cfg, m, e) for e in range(e0, e1)], ns, device)
            sc = cfg.e_lo + ((w >> 32) & 0xFFFFFFFF) % span
            s[e0:e1] = sc.to(torch.uint8).reshape(e1 - e0, rows, cols // 32)
            del w, sc
        for (fe, r, b, ev) in _forced_blocks(cfg, m):
            s[fe, r, b] = ev
        out[name + "_q"] = q
        out[name + "_s"] = s
    return out


def dense_inputs(cfg: Config) -> dict:
    """Every non-expert input of the config, on the host."""
    d = {
        "hidden": hidden(cfg),
        "router_w": router_weight(cfg),
        "router_b": router_bias(cfg),
    }
    if cfg.block:
        d["norm_gamma"] = norm_gamma(cfg)
        d["w_down"] = w_down(cfg)
        d["w_up"] = w_up(cfg)
        d["eps"] = RMS_EPS
    return d


def random_bytes(seed: int, n: int) -> np.ndarray:
    """n uniform bytes from the SplitMix64 stream ``seed`` (for standalone repack inputs)."""
    return words_np(seed, (n + 7) // 8).view(np.uint8)[:n].copy()


def random_exponents(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n E8M0 bytes uniform in [lo, hi]."""
    w = words_np(seed, n)
    return (lo + (w >> np.uint64(32)) % np.uint64(hi - lo + 1)).astype(np.uint8)
