"""The parallel evaluation used by the full-size sampled parity tests
(gpu_util.oracle_rows_parallel) against the serial oracle (CPU only): the
layer output is a sum of per-expert terms, so splitting the used experts over
processes and adding the parts must give the serial result up to float64
summation order, in latent and in block mode, with and without a forced
selection."""
import numpy as np

import oracle
import synth
from gpu_util import oracle_forward, oracle_rows_parallel, sample_rows


def _expert(cfg):
    return lambda m, e: synth.expert_matrix_np(cfg, m, e)


def test_parallel_matches_serial_latent():
    cfg = synth.custom("decode_t1", T=12, E=16, k=4, d=128, f=192, seed_index=41)
    dense = synth.dense_inputs(cfg)
    rows = np.array([0, 3, 4, 9, 11])
    ref = oracle_forward(cfg, dense, _expert(cfg), tokens=rows)
    got, r = oracle_rows_parallel(cfg, dense, rows, workers=3)
    assert np.array_equal(r["idx"], ref["idx"])
    assert np.allclose(got, ref["out"], rtol=1e-12, atol=1e-14)
    # a forced selection is used as given
    idx = np.roll(ref["idx"], 1, axis=1)
    ref2 = oracle_forward(cfg, dense, _expert(cfg), tokens=rows, idx=idx)
    got2, _ = oracle_rows_parallel(cfg, dense, rows, idx=idx, workers=2)
    assert np.allclose(got2, ref2["out"], rtol=1e-12, atol=1e-14)


def test_parallel_matches_serial_block():
    cfg = synth.custom("block_t8192", T=6, E=16, k=4, d=128, f=128, D=256, seed_index=42)
    dense = synth.dense_inputs(cfg)
    rows = np.arange(6)
    ref = oracle_forward(cfg, dense, _expert(cfg), tokens=rows)
    got, _ = oracle_rows_parallel(cfg, dense, rows, workers=4)
    # the combined latent row is rounded to bf16 before the up-projection: the
    # parts' summation order can move a value across a rounding boundary, so
    # compare within one bf16 step of that row, carried through W_up
    w_up = oracle.bf16_to_f64(dense["w_up"])
    step = np.abs(ref["moe_out"]) * 2.0 ** -7 @ np.abs(w_up).T
    assert np.all(np.abs(got - ref["out"]) <= step + 1e-12)


def test_sample_rows_covers_heavy_experts_and_tail():
    rng = np.random.default_rng(0)
    T, k, E = 500, 4, 40
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    idx[:200, 0] = 7  # a heavy expert
    rows = sample_rows(T, idx, 64, seed=1)
    assert len(rows) == 64 and len(np.unique(rows)) == 64
    heavy = np.nonzero((idx == 7).any(axis=1))[0]
    assert heavy[0] in rows and heavy[-1] in rows
    last = idx.max()
    assert np.nonzero((idx == last).any(axis=1))[0][-1] in rows
