"""k3moe_route_noalloc: the router entry point that allocates nothing.

Some callers cannot give the library device memory: everything they allocate
must come from a memory pool their framework owns, or they run inside a
decode loop where a cudaMalloc (which can synchronise the whole device) is not
allowed.  k3moe_route_noalloc serves them by keeping its scratch in a
library-owned static device array.  These tests call it through the C ABI
(ctypes, raw pointers) and check that it returns what k3moe_route returns on
the same inputs - indices exactly, weights and logits within the router
tests' fp32 tolerance - on two calls in a row, so that the shared scratch the
first call leaves behind does not change the second.
"""
import ctypes

import numpy as np
import pytest

import synth
from gpu_util import to_dev

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


def _inputs(name, T=None):
    cfg = synth.CONFIGS[name] if T is None else synth.custom(name, T=T)
    d = synth.dense_inputs(cfg)
    return cfg, to_dev(d["hidden"], "cuda"), to_dev(d["router_w"], "cuda"), to_dev(d["router_b"], "cuda")


def _noalloc(k3, x, w, b, k, with_logits):
    import torch

    T, d_r = x.shape
    E = w.shape[0]
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    logits = torch.zeros((T, E), dtype=torch.float32, device="cuda") if with_logits else None
    vp = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    st = k3.lib().k3moe_route_noalloc(vp(x), T, d_r, vp(w), vp(b), E, k, vp(idx), vp(wts),
                                      vp(logits),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, k3.lib().k3moe_status_string(st)
    return idx, wts, logits


def _check(k3, cfg, x, w, b, with_logits):
    idx_n, w_n, l_n = _noalloc(k3, x, w, b, cfg.k, with_logits)
    idx_r, w_r, l_r = k3.k3moe_route(x, w, b, cfg.k)
    assert np.array_equal(idx_n.cpu().numpy(), idx_r.cpu().numpy())
    assert np.allclose(w_n.cpu().numpy(), w_r.cpu().numpy(), rtol=2e-6, atol=1e-7)
    if with_logits:
        assert np.allclose(l_n.cpu().numpy(), l_r.cpu().numpy(), rtol=1e-6, atol=1e-6)


def test_noalloc_matches_route_two_calls(k3):
    cfg1, x1, w1, b1 = _inputs("verify_t8")
    cfg2, x2, w2, b2 = _inputs("decode_t1")
    _check(k3, cfg1, x1, w1, b1, with_logits=False)  # logits in the static scratch
    _check(k3, cfg2, x2, w2, b2, with_logits=True)
    _check(k3, cfg1, x1, w1, b1, with_logits=False)


def test_noalloc_tiny_two_calls(k3):
    cfg, x, w, b = _inputs("tiny")
    _check(k3, cfg, x, w, b, with_logits=True)
    _check(k3, cfg, x, w, b, with_logits=False)


def test_noalloc_rejects_sizes_beyond_its_scratch(k3):
    import torch

    cfg, x, w, b = _inputs("decode_t1", T=9)
    idx = torch.empty((9, 16), dtype=torch.int32, device="cuda")
    wts = torch.empty((9, 16), dtype=torch.float32, device="cuda")
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    L = k3.lib()
    assert L.k3moe_route_noalloc(vp(x), 9, x.shape[1], vp(w), vp(b), 896, 16, vp(idx), vp(wts),
                                 None, None) == 2  # K3MOE_ERR_SHAPE
    assert L.k3moe_route_noalloc(vp(x), 1, x.shape[1], vp(w), vp(b), 2048, 16, vp(idx), vp(wts),
                                 None, None) == 2
