"""GPU parity of the decode path (T <= 8) of k3moe_forward against the oracle.

Tolerance (the layer's stated bound): max |err| per token <= 1e-2 x RMS of
the oracle's output row on the computed value, plus half a bf16 ulp for the
conversion to the bf16 output (see gpu_util.rel_err_rows).  Tokens whose
oracle selection is a
near tie (margin below 1e-5) are compared with the oracle run on the kernel's
selection, which is then also a valid top-k.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import bf16_tensor_to_np, make_layer, oracle_forward, rel_err_rows, to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-2
# the tiny workload at the smallest width the tensor-core stages take (128)
TINY = dict(d=256, f=256)


@pytest.fixture(scope="module")
def k3():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mxfp4_routed_expert_sigmoid_gb300 as k3mod

    return k3mod


def run_and_compare(k3, cfg, path, tokens=None, tol=TOL, layer_bundle=None):
    import torch

    layer, dense, expert, _ = layer_bundle or make_layer(cfg, path=path)
    x = to_dev(dense["hidden"], "cuda")
    ws = k3.workspace(k3.k3moe_workspace_size(layer, cfg.T))
    out = k3.k3moe_forward(layer, x, ws=ws)
    idx_gpu, _, _ = k3.k3moe_forward_routing(layer, ws, cfg.T)
    assert k3.k3moe_get_status(ws) == 0
    got = bf16_tensor_to_np(out)
    idx_gpu = idx_gpu.cpu().numpy().astype(np.int64)
    tokens = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    ref = oracle_forward(cfg, dense, expert, tokens=tokens)
    near = ref["margin"] < 1e-5
    same = np.all(ref["idx"] == idx_gpu[tokens], axis=1)
    assert np.all(same | near), "selection differs outside near ties"
    if np.any(~same):
        ref = oracle_forward(cfg, dense, expert, tokens=tokens, idx=idx_gpu[tokens])
    err = rel_err_rows(got[tokens], ref["out"])
    assert np.all(err <= tol), f"max err/rms {err.max():.3e}"
    return out, ws, err


@pytest.mark.parametrize("T", [1, 3, 4, 8])
def test_tiny_decode(k3, T):
    cfg = synth.custom("tiny", T=T, **TINY)
    run_and_compare(k3, cfg, 1)


@pytest.mark.parametrize("T", [1, 5, 8])
def test_mid_decode(k3, T):
    # several row tiles per expert, ragged lane use (K/32 = 24 blocks), many experts
    cfg = synth.custom("decode_t1", T=T, E=64, k=8, d=768, f=1280, seed_index=11)
    run_and_compare(k3, cfg, 1)


def test_decode_t1_full(k3):
    run_and_compare(k3, synth.CONFIGS["decode_t1"], 0)


def test_verify_t8_full_and_deterministic(k3):
    import torch

    cfg = synth.CONFIGS["verify_t8"]
    bundle = make_layer(cfg, path=0)
    out1, ws, _ = run_and_compare(k3, cfg, 0, layer_bundle=bundle)
    out2 = k3.k3moe_forward(bundle[0], to_dev(bundle[1]["hidden"], "cuda"), ws=ws)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_power_of_two_invariant_decode(k3):
    """Adding 1 to every W2 exponent doubles the output bit-exactly."""
    import torch

    cfg = synth.custom("decode_t1", T=4, E=32, k=4, d=512, f=512, seed_index=12)
    layer, dense, expert, ex = make_layer(cfg, path=1)
    x = to_dev(dense["hidden"], "cuda")
    out1 = k3.k3moe_forward(layer, x)
    ex2 = dict(ex)
    ex2["w2_s"] = ex["w2_s"] + 1
    layer2 = k3.MoELayer(router_w=layer.tensors["router_w"], router_b=layer.tensors["router_b"],
                         k=cfg.k, path=1, **ex2)
    out2 = k3.k3moe_forward(layer2, x)
    assert torch.equal(out2.float(), 2 * out1.float())


def test_forward_host_buffers(k3):
    import torch

    cfg = synth.custom("tiny", T=2, **TINY)
    layer, dense, expert, _ = make_layer(cfg, path=1)
    x_host = torch.from_numpy(dense["hidden"].view(np.int16)).view(torch.bfloat16).pin_memory()
    out_host = k3.k3moe_forward_host(layer, x_host)
    out_dev = k3.k3moe_forward(layer, x_host.cuda())
    assert torch.equal(out_host.view(torch.int16), out_dev.cpu().view(torch.int16))


def test_graph_replay_matches_forward(k3):
    """k3moe_graph_create / k3moe_graph_launch reproduce k3moe_forward bit for bit."""
    import torch

    cfg = synth.custom("decode_t1", T=3, E=64, k=8, d=768, f=1280, seed_index=13)
    layer, dense, expert, _ = make_layer(cfg, path=0)
    x = to_dev(dense["hidden"], "cuda")
    ws = k3.workspace(k3.k3moe_workspace_size(layer, cfg.T))
    ref = k3.k3moe_forward(layer, x, ws=ws).clone()
    out = torch.zeros_like(ref)
    graph = k3.ForwardGraph(layer, x, out, ws)
    out.zero_()
    graph.launch()
    graph.launch()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    graph.close()


def test_trace_of_graph_replay(k3):
    """Kernel tracing inside a library graph: every kernel of the forward
    reports a positive duration after a replay."""
    import torch

    cfg = synth.custom("decode_t1", T=2, E=64, k=8, d=768, f=1280, seed_index=14)
    layer, dense, expert, _ = make_layer(cfg, path=0)
    x = to_dev(dense["hidden"], "cuda")
    ws = k3.workspace(k3.k3moe_workspace_size(layer, cfg.T))
    out = torch.empty_like(x)
    k3.k3moe_trace(True)
    graph = k3.ForwardGraph(layer, x, out, ws)
    k3.k3moe_trace(False)
    graph.launch()
    tr = k3.k3moe_trace_read()
    torch.cuda.synchronize()
    names = [n for n, _ in tr]
    assert "route_small" in names and "decode_up" in names and "combine" in names
    assert all(ms > 0 for _, ms in tr)
    graph.close()
