"""Expert parallelism (mxfp4_routed_expert_sigmoid_gb300.ep) on gloo ranks.

Two (and three) CPU ranks split the tiny layer's experts; every rank routes
its own tokens, dispatches each (token, slot) pair to the rank that owns the
expert, the owner computes w * expert(row), and the rows come back and are
added in slot order.  The routing and the expert FFN here are the oracle's
(float64), so each rank's output must equal oracle.moe_forward on its tokens
up to the order of a float64 sum.  Multi-GPU runs are not available to these
tests: the GPU compute step (k3moe_forward_routed) is checked on one GPU in
tests/test_gpu_decode.py, the exchange only here."""
import os
import socket

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, E, counts, results):
    import torch.distributed as dist

    from mxfp4_routed_expert_sigmoid_gb300.ep import ExpertParallel

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total = sum(counts)
        cfg = synth.custom("tiny", T=total, E=E, k=3, seed_index=71)
        dense = synth.dense_inputs(cfg)
        lo = sum(counts[:rank])
        mine = np.arange(lo, lo + counts[rank])
        x_all = oracle.bf16_to_f64(dense["hidden"])
        wr = oracle.bf16_to_f64(dense["router_w"])
        ep = ExpertParallel(E, cfg.k)
        expert = lambda m, e: synth.expert_matrix_np(cfg, m, e)  # noqa: E731

        def route_fn(x):
            r = oracle.select_experts(oracle.router_logits(x.numpy(), wr), dense["router_b"], cfg.k)
            return torch.from_numpy(r["idx"]), torch.from_numpy(r["w"])

        def experts_fn(rows, local, w):
            y = torch.zeros_like(rows)
            for e_local in torch.unique(local).tolist():
                sel = (local[:, 0] == e_local).nonzero()[:, 0]
                e = ep.owned()[e_local]
                W = [oracle.decode_source(*expert(m, e)) for m in range(3)]
                y[sel] = w[sel].to(torch.float64) * torch.from_numpy(oracle.expert_ffn(rows[sel].numpy(), *W))
            return y

        x = torch.from_numpy(x_all[mine])
        idx, _ = route_fn(x)
        plan = ep.plan(idx)
        out = ep.forward(x, route_fn, experts_fn)
        ref = oracle.moe_forward(x_all[mine], wr, dense["router_b"], cfg.k, x_all[mine], expert)["out"]
        results[rank] = dict(err=float(np.max(np.abs(out.numpy() - ref))) if len(mine) else 0.0,
                             scale=float(np.max(np.abs(ref))) if len(mine) else 1.0,
                             counts=plan["send_counts"].tolist(),
                             order=plan["order"].tolist(), local=plan["local"].tolist(),
                             idx=idx.tolist())
    finally:
        dist.destroy_process_group()


def _run(world, E, counts):
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, E, counts, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    return [results[r] for r in range(world)]


@pytest.mark.parametrize("world,E,counts", [(2, 8, [5, 4]), (2, 8, [6, 0]), (3, 9, [2, 5, 3])])
def test_expert_parallel_matches_oracle(world, E, counts):
    res = _run(world, E, counts)
    El = E // world
    for r, d in enumerate(res):
        # the rank's output is the oracle layer on its tokens
        assert d["err"] <= 1e-12 * max(d["scale"], 1.0), (r, d["err"])
        # plan: every pair once, grouped by owner, tokens then slots ascending
        # within an owner, local indices inside the owner's range
        idx = np.asarray(d["idx"], dtype=np.int64).reshape(-1)
        order = np.asarray(d["order"], dtype=np.int64)
        assert sorted(order.tolist()) == list(range(len(idx)))
        owner = idx[order] // El
        assert np.all(np.diff(owner) >= 0)
        for o in range(world):
            grp = order[owner == o]
            assert np.all(np.diff(grp) > 0)
        assert np.array_equal(np.asarray(d["local"], dtype=np.int64), idx[order] - owner * El)
        assert d["counts"] == np.bincount(idx // El, minlength=world).tolist()
