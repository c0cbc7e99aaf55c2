"""GPU parity of the host-resident expert path (k3moe_forward_cached).

The expert arrays live in page-locked host memory and a device cache of S
slots holds the recently used experts (least recently used eviction, per the
K3-Stuff model page, "llama-cpp-patches", change 2).  Checked per call:
  * the output is bitwise that of k3moe_forward on device-resident weights
    (the same kernels read the same bytes, from a slot instead);
  * the slot maps, stamps and counters equal those of the policy oracle
    (oracle/cache.py) fed with the experts the GPU's routing used;
  * the first call of each sequence also against the layer oracle
    (max |err| <= 1e-2 x row RMS + half a bf16 ulp).
"""
import numpy as np
import pytest

import synth
from gpu_util import bf16_tensor_to_np, make_layer, oracle_forward, rel_err_rows, to_dev
from oracle.cache import CacheState, cache_call

pytestmark = pytest.mark.gpu

SMALL = dict(E=128, k=4, d=512, f=512)


@pytest.fixture(scope="module")
def k3():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mxfp4_routed_expert_sigmoid_gb300 as k3mod

    return k3mod


@pytest.fixture(scope="module")
def small(k3):
    cfg = synth.custom("decode_t1", T=1, **SMALL)
    layer, dense, expert, _ = make_layer(cfg, on_device_experts=False)
    return cfg, layer, k3.host_resident(layer), dense, expert


def batches(cfg, n, T, seed):
    """n distinct seeded token batches [T, d] (bf16 bits) of the config's distribution."""
    big = synth.custom(cfg.name, T=T * n, E=cfg.E, k=cfg.k, d=cfg.d, f=cfg.f, D=cfg.D, seed_index=seed)
    return synth.hidden(big).reshape(n, T, -1)


def check_state(k3, cache, st: CacheState, call: dict):
    slot_of, expert_of, stamp = (t.cpu().numpy() for t in cache.maps())
    assert slot_of.tolist() == st.slot_of
    assert expert_of.tolist() == st.expert_of
    assert stamp.tolist() == st.stamp
    s = cache.stats()
    assert (s["calls"], s["hits"], s["misses"]) == (st.clock, st.hits, st.misses)
    assert (s["last_hits"], s["last_misses"]) == (call["hits"], call["misses"])


def run_sequence(k3, bundle, T, S, n, seed, graph=False):
    import torch

    cfg, layer, hlayer, dense, expert = bundle
    cache = k3.ExpertCache(hlayer, S)
    st = CacheState.empty(cfg.E, S)
    xs = batches(cfg, n, T, seed)
    ws_c = k3.workspace(k3.k3moe_workspace_size(hlayer, T))
    ws_r = k3.workspace(k3.k3moe_workspace_size(layer, T))
    x_buf = to_dev(xs[0], "cuda")
    out_c = torch.empty_like(x_buf)
    g = None
    if graph:
        g = k3.ForwardGraph(hlayer, x_buf, out_c, ws_c, cache=cache)  # runs xs[0] once
        idx, _, _ = k3.k3moe_forward_routing(hlayer, ws_c, T)
        check_state(k3, cache, st, cache_call(st, np.unique(idx.cpu().numpy())))
    seen = set()
    for i in range(n):
        x_buf.copy_(to_dev(xs[i], "cuda"))
        if g is not None:
            g.launch()
        else:
            k3.k3moe_forward_cached(hlayer, cache, x_buf, out=out_c, ws=ws_c)
        assert k3.k3moe_get_status(ws_c) == 0
        ref = k3.k3moe_forward(layer, x_buf, ws=ws_r)
        assert torch.equal(out_c.view(torch.int16), ref.view(torch.int16)), f"call {i}"
        idx, _, _ = k3.k3moe_forward_routing(hlayer, ws_c, T)
        used = np.unique(idx.cpu().numpy())
        seen |= set(used.tolist())
        check_state(k3, cache, st, cache_call(st, used))
        if i == 0:
            o = oracle_forward(cfg, dict(dense, hidden=xs[0]), expert)
            assert np.all(o["idx"] == idx.cpu().numpy()) or np.any(o["margin"] < 1e-5)
            err = rel_err_rows(bf16_tensor_to_np(out_c), o["out"])
            assert np.all(err <= 1e-2), err.max()
    s = cache.stats()
    assert s["bytes"] == s["misses"] * 3 * (cfg.f * cfg.d // 2 + cfg.f * cfg.d // 32)
    return s, seen


@pytest.mark.parametrize("T,S", [(1, 4), (1, 24), (2, 8), (8, 32), (8, 128)])
def test_cached_decode(k3, small, T, S):
    s, seen = run_sequence(k3, small, T, S, n=10, seed=40 + T + S)
    assert s["misses"] >= min(len(seen), S)


@pytest.mark.parametrize("T,S", [(20, 80), (40, 128)])
def test_cached_units(k3, small, T, S):
    run_sequence(k3, small, T, S, n=5, seed=60 + T)


def test_cached_graph(k3, small):
    run_sequence(k3, small, 2, 12, n=6, seed=77, graph=True)


def test_hot_experts_stay_resident(k3):
    """Tokens that all favour the same 8 hot experts (bias +1, as in the
    draft-verification workload) hit the cache after the first call."""
    cfg = synth.custom("verify_t8", T=8, E=64, k=4, d=256, f=256)
    # d = f = 256 are not whole 512-input stages: the cache takes the prepared scales
    layer, dense, expert, _ = make_layer(cfg, on_device_experts=False, prepared=True)
    import torch

    b = torch.zeros(cfg.E, dtype=torch.float32)
    b[:8] = 1.0
    layer.tensors["router_b"].copy_(b)
    hlayer = k3.host_resident(layer)
    cache = k3.ExpertCache(hlayer, 32)
    xs = batches(cfg, 6, 8, 91)
    ws = k3.workspace(k3.k3moe_workspace_size(hlayer, 8))
    seen, used_total = set(), 0
    for x in xs:
        k3.k3moe_forward_cached(hlayer, cache, to_dev(x, "cuda"), ws=ws)
        used = set(np.unique(k3.k3moe_forward_routing(hlayer, ws, 8)[0].cpu().numpy()).tolist())
        assert used <= set(range(8))
        seen |= used
        used_total += len(used)
    s = cache.stats()
    assert s["misses"] == len(seen) and s["hits"] == used_total - len(seen)


def test_cache_errors(k3, small):
    import torch

    cfg, layer, hlayer, dense, _ = small
    x = to_dev(batches(cfg, 1, 1, 5)[0], "cuda")
    ws = k3.workspace(k3.k3moe_workspace_size(hlayer, 1))
    # state never initialised: the device flags it and nothing is fetched
    cache = k3.ExpertCache(hlayer, 8)
    cache.tensors["state"].zero_()
    for t in ("w1_q", "w3_q", "w2_q", "w1_s", "w3_s", "w2_s"):
        cache.tensors[t].zero_()
    k3.k3moe_forward_cached(hlayer, cache, x, ws=ws)
    assert k3.k3moe_get_status(ws) == 1
    # device arrays where host ones are expected
    cache.reset()
    with pytest.raises(k3.K3MoEError) as ex:
        k3.k3moe_forward_cached(layer, cache, x, ws=ws)
    assert ex.value.status == 1
    # too few slots for 8 tokens x 4 experts
    with pytest.raises(k3.K3MoEError) as ex:
        x8 = to_dev(batches(cfg, 1, 8, 6)[0], "cuda")
        k3.k3moe_forward_cached(hlayer, cache, x8, ws=k3.workspace(k3.k3moe_workspace_size(hlayer, 8)))
    assert ex.value.status == 2
    assert torch.cuda.is_available()


@pytest.mark.parametrize("T", [1, 6])
def test_cached_block_mode(k3, T):
    """The full latent block (RMSNorm, down-projection, router on the normed
    width, experts, up-projection) with host-resident experts: bitwise the
    block on device-resident experts, call after call."""
    import torch

    cfg = synth.custom("block_t8192", T=T, E=32, k=4, d=512, f=512, D=1024, seed_index=27)
    layer, dense, expert, _ = make_layer(cfg, on_device_experts=False)
    hlayer = k3.host_resident(layer)
    cache = k3.ExpertCache(hlayer, min(cfg.E, T * cfg.k + 4))
    st = CacheState.empty(cfg.E, cache.slots)
    big = synth.custom(cfg.name, T=T * 4, E=cfg.E, k=cfg.k, d=cfg.d, f=cfg.f, D=cfg.D, seed_index=28)
    xs = synth.hidden(big).reshape(4, T, -1)
    ws_c = k3.workspace(k3.k3moe_workspace_size(hlayer, T))
    ws_r = k3.workspace(k3.k3moe_workspace_size(layer, T))
    for x_np in xs:
        x = to_dev(x_np, "cuda")
        got = k3.k3moe_forward_cached(hlayer, cache, x, ws=ws_c)
        ref = k3.k3moe_forward(layer, x, ws=ws_r)
        assert k3.k3moe_get_status(ws_c) == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
        idx, _, _ = k3.k3moe_forward_routing(hlayer, ws_c, T)
        check_state(k3, cache, st, cache_call(st, np.unique(idx.cpu().numpy())))


def test_graph_after_queued_calls(k3, small):
    """Graph creation right after eager calls still queued on the caller's
    stream: its set-up forward (on a private stream) must not overlap them."""
    import torch

    cfg, layer, hlayer, dense, expert = small
    T, S = 1, 8
    cache = k3.ExpertCache(hlayer, S)
    xs = batches(cfg, 5, T, 88)
    ws = k3.workspace(k3.k3moe_workspace_size(hlayer, T))
    out = torch.empty((T, cfg.d), dtype=torch.bfloat16, device="cuda")
    idxs = []
    for i in range(4):  # no synchronisation in between
        k3.k3moe_forward_cached(hlayer, cache, to_dev(xs[i], "cuda"), out=out, ws=ws)
        idxs.append(k3.k3moe_forward_routing(hlayer, ws, T, with_logits=False)[0])
    g = k3.ForwardGraph(hlayer, to_dev(xs[4], "cuda"), out, ws, cache=cache)
    idxs.append(k3.k3moe_forward_routing(hlayer, ws, T, with_logits=False)[0])
    assert k3.k3moe_get_status(ws) == 0
    st = CacheState.empty(cfg.E, S)
    for idx in idxs:
        call = cache_call(st, np.unique(idx.cpu().numpy()))
    check_state(k3, cache, st, call)
    g.close()
