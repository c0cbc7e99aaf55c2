"""Failure detection on the GPU, without faulting it.

Every wait inside the library's kernels is bounded; on expiry the kernel
records K3MOE_ERR_TIMEOUT in the workspace status word, every role of the CTA
stops, its copies in flight land, tensor memory is released and the kernel
returns.  k3moe_inject_fault arms the one fault that exercises this: a
pipeline stage of the W1/W3 stream that is never signalled, with the wait
limit cut to 1 ms.  The tests check that the call returns promptly with the
timeout status and that the next call on the same workspace is correct.
Host-side injections: a NaN router input, a NaN selection bias (status
NONFINITE), a bias of +inf (a valid key: that expert is always selected), and
a workspace one byte short (rejected before any launch).
"""
import time

import numpy as np
import pytest

import synth
from gpu_util import bf16_tensor_to_np, make_layer, oracle_forward, record_margin, rel_err_rows, to_dev

pytestmark = pytest.mark.gpu

SHAPE = dict(E=32, k=4, d=512, f=512)


@pytest.fixture(scope="module")
def k3():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mxfp4_routed_expert_sigmoid_gb300 as k3mod

    return k3mod


@pytest.mark.parametrize("T", [1, 8, 20])
def test_dropped_signal_times_out_and_recovers(k3, T):
    import torch

    cfg = synth.custom("decode_t1", T=T, seed_index=51, **SHAPE)
    layer, dense, expert, _ = make_layer(cfg, path=1)
    x = to_dev(dense["hidden"], "cuda")
    ws = k3.workspace(k3.k3moe_workspace_size(layer, T))
    ref = k3.k3moe_forward(layer, x, ws=ws).clone()
    assert k3.k3moe_get_status(ws) == 0
    assert k3.k3moe_inject_fault(k3.FAULT_DROP_SIGNAL) == 0
    t0 = time.perf_counter()
    k3.k3moe_forward(layer, x, ws=ws)
    status = k3.k3moe_get_status(ws)  # synchronises: the kernels have returned
    elapsed = time.perf_counter() - t0
    assert status == 7, k3.STATUS.get(status, status)
    assert elapsed < 1.0  # one 1 ms wait, not the 2 s default
    assert k3.k3moe_inject_fault(0) == 0  # consumed by that forward
    out = k3.k3moe_forward(layer, x, ws=ws)
    assert k3.k3moe_get_status(ws) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_nonfinite_router_input_flagged(k3):
    cfg = synth.custom("decode_t1", T=3, seed_index=52, **SHAPE)
    layer, dense, expert, _ = make_layer(cfg, path=1)
    h = dense["hidden"].copy()
    h[1, 17] = 0x7FC0  # NaN
    ws = k3.workspace(k3.k3moe_workspace_size(layer, cfg.T))
    k3.k3moe_forward(layer, to_dev(h, "cuda"), ws=ws)
    assert k3.k3moe_get_status(ws) == 6
    k3.k3moe_forward(layer, to_dev(dense["hidden"], "cuda"), ws=ws)
    assert k3.k3moe_get_status(ws) == 0


def test_nan_bias_flagged(k3):
    cfg = synth.custom("decode_t1", T=2, seed_index=53, **SHAPE)
    layer, dense, expert, _ = make_layer(cfg, path=1)
    b = layer.tensors["router_b"]
    keep = b[5].item()
    b[5] = float("nan")
    ws = k3.workspace(k3.k3moe_workspace_size(layer, cfg.T))
    k3.k3moe_forward(layer, to_dev(dense["hidden"], "cuda"), ws=ws)
    assert k3.k3moe_get_status(ws) == 6
    b[5] = keep


@pytest.mark.parametrize("path", [1, 2])
def test_infinite_bias_selects_first(k3, path):
    """b = +inf is a valid selection key: the expert takes slot 0 of every
    token, its weight stays the unbiased renormalised score, and the output
    matches the oracle on the same bias."""
    cfg = synth.custom("decode_t1", T=5, seed_index=54, **SHAPE)
    layer, dense, expert, _ = make_layer(cfg, path=path)
    dense = dict(dense)
    dense["router_b"] = dense["router_b"].copy()
    dense["router_b"][11] = np.inf
    import torch

    layer.tensors["router_b"].copy_(torch.from_numpy(dense["router_b"]))
    x = to_dev(dense["hidden"], "cuda")
    ws = k3.workspace(k3.k3moe_workspace_size(layer, cfg.T))
    out = k3.k3moe_forward(layer, x, ws=ws)
    assert k3.k3moe_get_status(ws) == 0
    idx, _, _ = k3.k3moe_forward_routing(layer, ws, cfg.T)
    assert np.all(idx.cpu().numpy()[:, 0] == 11)
    ref = oracle_forward(cfg, dense, expert)
    assert np.all(ref["idx"][:, 0] == 11)
    err = rel_err_rows(bf16_tensor_to_np(out), ref["out"])
    record_margin(f"bias +inf path={path}", err, 1e-2)
    assert np.all(err <= 1e-2)


def test_short_workspace_rejected(k3):
    import torch

    cfg = synth.custom("decode_t1", T=4, seed_index=55, **SHAPE)
    layer, dense, expert, _ = make_layer(cfg, path=1)
    x = to_dev(dense["hidden"], "cuda")
    need = k3.k3moe_workspace_size(layer, cfg.T)
    ws = k3.workspace(need)
    out = torch.full_like(x, 7.0)
    with pytest.raises(k3.K3MoEError) as ex:
        k3.k3moe_forward(layer, x, out=out, ws=ws[: need - 1])
    assert ex.value.status == 4
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)  # nothing was launched
    k3.k3moe_forward(layer, x, out=out, ws=ws)
    assert k3.k3moe_get_status(ws) == 0
