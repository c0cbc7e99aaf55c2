"""Expert parallelism with the library's kernels on one GPU (a one-rank NCCL
group): k3moe_route routes, the dispatch sends every (token, slot) pair to
the owner (this rank), k3moe_forward_routed runs the experts with k = 1 on
the received rows, and the combine adds each token's rows in slot order.
Checked against the oracle.  The bound: the layer's 1e-2 x row RMS, plus half
a bf16 ulp of each of the k weighted rows, which the routed forward returns
as bf16 before the combine adds them (tests/test_ep_dist.py checks the
exchange itself on several gloo ranks)."""
import os
import socket

import numpy as np
import pytest

import oracle
import synth
from gpu_util import make_layer, record_margin, to_dev

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


@pytest.mark.parametrize("T", [3, 40])
def test_one_rank_expert_parallel(k3, T):
    import torch
    import torch.distributed as dist

    from mxfp4_routed_expert_sigmoid_gb300.ep import ExpertParallel, routed_experts_fn

    cfg = synth.custom("decode_t1", T=T, E=16, k=4, d=512, f=512, seed_index=72)
    layer, dense, expert, ex = make_layer(cfg, path=0)
    local = k3.MoELayer(router_w=layer.tensors["router_w"], router_b=layer.tensors["router_b"], k=1, **ex)
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        ep = ExpertParallel(cfg.E, cfg.k)
        x = to_dev(dense["hidden"], "cuda")

        def route_fn(h):
            idx, w, _ = k3.k3moe_route(h, layer.tensors["router_w"], layer.tensors["router_b"], cfg.k,
                                       with_logits=False)
            return idx, w

        out = ep.forward(x, route_fn, routed_experts_fn(local)).cpu().numpy().astype(np.float64)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    xr = oracle.bf16_to_f64(dense["hidden"])
    ref = oracle.moe_forward(xr, oracle.bf16_to_f64(dense["router_w"]), dense["router_b"], cfg.k, xr, expert)
    terms = np.zeros_like(ref["out"])  # sum over slots of |w_j y_j|
    for e in np.unique(ref["idx"]):
        tok, slot = np.nonzero(ref["idx"] == e)
        W = [oracle.decode_source(*expert(m, int(e))) for m in range(3)]
        terms[tok] += np.abs(ref["w"][tok, slot][:, None] * oracle.expert_ffn(xr[tok], *W))
    rms = np.sqrt(np.mean(ref["out"] ** 2, axis=1))
    err = np.max((np.abs(out - ref["out"]) - 2.0 ** -8 * terms) / rms[:, None], axis=1)
    record_margin(f"expert parallel, one rank, T={T}", err, 1e-2)
    assert np.all(err <= 1e-2)
