"""Python binding of libk3moe: the latent routed-expert MoE layer over MXFP4
weights (Kimi-K3 style) for GB300 (sm_103a).

This module only marshals arguments: every step of the layer runs in the CUDA
kernels of ``lib/libk3moe.so`` (built in-tree by ``_build.py``).  PyTorch
provides device memory and streams.  The functions carry the C ABI's names
(``include/k3moe.h``); tensors go in and out.  If the library is missing the
import of a function fails loudly: there is no other implementation.

bf16 tensors are ``torch.bfloat16`` (int16/uint16 tensors holding bf16 bits
are accepted and viewed).  All device tensors must be contiguous and 16-byte
aligned.  Workspaces are uint8 device tensors; a fresh workspace must be
zero-filled (the helpers here allocate with ``torch.zeros``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libk3moe.so")

ACT_SILU_GATED = 0
PATH_AUTO, PATH_BLOCK_SCALED, PATH_BF16_DEQUANT = 0, 1, 2
PATH_DECODE, PATH_GROUPED = PATH_BLOCK_SCALED, PATH_BF16_DEQUANT  # ABI version 3 names
FORMAT_SPLIT, FORMAT_GGML = 0, 1

STATUS = {
    0: "K3MOE_OK", 1: "K3MOE_ERR_INVALID_ARG", 2: "K3MOE_ERR_SHAPE", 3: "K3MOE_ERR_ALIGN",
    4: "K3MOE_ERR_WORKSPACE", 5: "K3MOE_ERR_CUDA", 6: "K3MOE_ERR_NONFINITE",
    7: "K3MOE_ERR_TIMEOUT", 8: "K3MOE_ERR_UNSUPPORTED",
}

#: every symbol the C header declares (checked by the CPU test suite)
EXPORTS = (
    "k3moe_abi_version", "k3moe_inject_fault", "k3moe_status_string", "k3moe_repack_mxfp4",
    "k3moe_unpack_mxfp4",
    "k3moe_route_workspace_size", "k3moe_route", "k3moe_route_noalloc", "k3moe_permute",
    "k3moe_rmsnorm",
    "k3moe_gemm_bf16", "k3moe_workspace_size", "k3moe_forward", "k3moe_forward_routed",
    "k3moe_host_staging_size",
    "k3moe_forward_host", "k3moe_forward_routing", "k3moe_forward_intermediates",
    "k3moe_get_status", "k3moe_trace",
    "k3moe_graph_create", "k3moe_graph_launch", "k3moe_graph_destroy",
    "k3moe_trace_read", "k3moe_trace_read_stamps", "k3moe_prepared_scales_size",
    "k3moe_prepare_scales",
    "k3moe_unprepare_scales",
    "k3moe_cache_state_size", "k3moe_cache_init", "k3moe_forward_cached",
    "k3moe_cache_read_stats", "k3moe_graph_create_cached",
)


class K3MoEError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {what}")


class LayerDesc(ctypes.Structure):
    """Mirror of ``k3moe_layer_desc``."""
    _fields_ = [
        ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("d", ctypes.c_int32),
        ("f", ctypes.c_int32), ("d_router", ctypes.c_int32), ("act", ctypes.c_int32),
        ("path", ctypes.c_int32), ("D", ctypes.c_int32), ("eps", ctypes.c_float),
        ("format", ctypes.c_int32),
        ("w1_q", ctypes.c_void_p), ("w3_q", ctypes.c_void_p), ("w2_q", ctypes.c_void_p),
        ("w1_s", ctypes.c_void_p), ("w3_s", ctypes.c_void_p), ("w2_s", ctypes.c_void_p),
        ("w1_sf", ctypes.c_void_p), ("w3_sf", ctypes.c_void_p), ("w2_sf", ctypes.c_void_p),
        ("router_w", ctypes.c_void_p), ("router_b", ctypes.c_void_p),
        ("norm_gamma", ctypes.c_void_p), ("w_down", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
    ]


class CacheDesc(ctypes.Structure):
    """Mirror of ``k3moe_expert_cache``."""
    _fields_ = [
        ("slots", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("w1_q", ctypes.c_void_p), ("w3_q", ctypes.c_void_p), ("w2_q", ctypes.c_void_p),
        ("w1_s", ctypes.c_void_p), ("w3_s", ctypes.c_void_p), ("w2_s", ctypes.c_void_p),
        ("state", ctypes.c_void_p),
    ]


class CacheStats(ctypes.Structure):
    """Mirror of ``k3moe_cache_stats``."""
    _fields_ = [
        ("calls", ctypes.c_uint64), ("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64),
        ("bytes", ctypes.c_uint64), ("last_hits", ctypes.c_int32), ("last_misses", ctypes.c_int32),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libk3moe.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    f32 = ctypes.c_float
    sigs = {
        "k3moe_abi_version": ([], ctypes.c_int),
        "k3moe_inject_fault": ([ctypes.c_int], ctypes.c_int),
        "k3moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "k3moe_repack_mxfp4": ([vp, vp, i64, i64, vp, vp], ctypes.c_int),
        "k3moe_unpack_mxfp4": ([vp, i64, i64, vp, vp, vp], ctypes.c_int),
        "k3moe_route_workspace_size": ([i32, i32], sz),
        "k3moe_route": ([vp, i32, i32, vp, vp, i32, i32, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "k3moe_route_noalloc": ([vp, i32, i32, vp, vp, i32, i32, vp, vp, vp, vp], ctypes.c_int),
        "k3moe_permute": ([vp, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "k3moe_rmsnorm": ([vp, i32, i32, vp, f32, vp, vp], ctypes.c_int),
        "k3moe_gemm_bf16": ([vp, vp, i32, i32, i32, vp, i32, vp], ctypes.c_int),
        "k3moe_workspace_size": ([ctypes.POINTER(LayerDesc), i32], sz),
        "k3moe_forward": ([ctypes.POINTER(LayerDesc), vp, i32, vp, vp, sz, vp], ctypes.c_int),
        "k3moe_forward_routed": ([ctypes.POINTER(LayerDesc), vp, i32, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "k3moe_host_staging_size": ([ctypes.POINTER(LayerDesc), i32], sz),
        "k3moe_forward_host": ([ctypes.POINTER(LayerDesc), vp, i32, vp, vp, sz, vp], ctypes.c_int),
        "k3moe_forward_routing": ([ctypes.POINTER(LayerDesc), vp, i32, vp, vp, vp, vp],
                                  ctypes.c_int),
        "k3moe_forward_intermediates": ([ctypes.POINTER(LayerDesc), vp, i32, vp, vp, vp, vp],
                                        ctypes.c_int),
        "k3moe_get_status": ([vp, vp, ctypes.POINTER(i32)], ctypes.c_int),
        "k3moe_trace": ([ctypes.c_int], ctypes.c_int),
        "k3moe_graph_create": ([ctypes.POINTER(LayerDesc), vp, i32, vp, vp, sz,
                                ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
        "k3moe_graph_launch": ([vp, vp], ctypes.c_int),
        "k3moe_graph_destroy": ([vp], ctypes.c_int),
        "k3moe_trace_read": ([ctypes.c_int, ctypes.POINTER(ctypes.c_char_p),
                              ctypes.POINTER(ctypes.c_float)], ctypes.c_int),
        "k3moe_trace_read_stamps": ([ctypes.c_int, ctypes.POINTER(ctypes.c_char_p),
                                     ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)],
                                    ctypes.c_int),
        "k3moe_prepared_scales_size": ([i64, i64, i64], sz),
        "k3moe_prepare_scales": ([vp, i64, i64, i64, vp, vp], ctypes.c_int),
        "k3moe_cache_state_size": ([i32, i32], sz),
        "k3moe_cache_init": ([vp, i32, i32, vp], ctypes.c_int),
        "k3moe_forward_cached": ([ctypes.POINTER(LayerDesc), ctypes.POINTER(CacheDesc), vp, i32,
                                  vp, vp, sz, vp], ctypes.c_int),
        "k3moe_cache_read_stats": ([vp, vp, ctypes.POINTER(CacheStats)], ctypes.c_int),
        "k3moe_graph_create_cached": ([ctypes.POINTER(LayerDesc), ctypes.POINTER(CacheDesc), vp,
                                       i32, vp, vp, sz, ctypes.POINTER(ctypes.c_void_p)],
                                      ctypes.c_int),
        "k3moe_unprepare_scales": ([vp, i64, i64, i64, vp, vp], ctypes.c_int),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def _check(st: int):
    if st != 0:
        raise K3MoEError(st, lib().k3moe_status_string(st).decode())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _bf16(t: torch.Tensor, name: str):
    _dev(t, name)
    if t.dtype in (torch.int16, torch.uint16):
        t = t.view(torch.bfloat16)
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bf16")
    return t


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled uint8 device workspace of nbytes."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def k3moe_abi_version() -> int:
    return lib().k3moe_abi_version()


FAULT_DROP_SIGNAL = 1


def k3moe_inject_fault(code: int) -> int:
    """Testing aid: arm a device-side fault for the next k3moe_forward of this
    thread (FAULT_DROP_SIGNAL: a pipeline stage is never signalled and the
    bounded wait for it runs out after 1 ms); 0 disarms."""
    return int(lib().k3moe_inject_fault(int(code)))


def k3moe_repack_mxfp4(packed: torch.Tensor, scale: torch.Tensor, out=None, stream=None):
    """compressed-tensors (packed [rows, cols/2], scale [rows, cols/32]) -> ggml blocks [rows, cols/32, 17]."""
    _dev(packed, "packed"), _dev(scale, "scale")
    rows, cols = packed.shape[0], packed.shape[-1] * 2
    if out is None:
        out = torch.empty((rows, cols // 32, 17), dtype=torch.uint8, device=packed.device)
    _check(lib().k3moe_repack_mxfp4(_p(packed), _p(scale), rows, cols, _p(_dev(out, "out")),
                                    _stream(stream)))
    return out


def k3moe_unpack_mxfp4(blocks: torch.Tensor, packed_out=None, scale_out=None, stream=None):
    """ggml blocks [rows, cols/32, 17] -> (packed [rows, cols/2], scale [rows, cols/32])."""
    _dev(blocks, "blocks")
    rows, nb = blocks.shape[0], blocks.shape[1]
    cols = nb * 32
    if packed_out is None:
        packed_out = torch.empty((rows, cols // 2), dtype=torch.uint8, device=blocks.device)
    if scale_out is None:
        scale_out = torch.empty((rows, nb), dtype=torch.uint8, device=blocks.device)
    _check(lib().k3moe_unpack_mxfp4(_p(blocks), rows, cols, _p(packed_out), _p(scale_out),
                                    _stream(stream)))
    return packed_out, scale_out


def k3moe_route_workspace_size(T: int, E: int) -> int:
    return lib().k3moe_route_workspace_size(T, E)


def k3moe_route(x, router_w, bias, k: int, with_logits: bool = True, ws=None, stream=None):
    """Router: returns (idx [T,k] int32, w [T,k] fp32, logits [T,E] fp32 or None)."""
    x, router_w = _bf16(x, "x"), _bf16(router_w, "router_w")
    _dev(bias, "bias")
    T, d_r = x.shape
    E = router_w.shape[0]
    dev = x.device
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev) if with_logits else None
    if ws is None:
        ws = workspace(k3moe_route_workspace_size(T, E), dev)
    _check(lib().k3moe_route(_p(x), T, d_r, _p(router_w), _p(bias), E, k, _p(idx), _p(w),
                             _p(logits), _p(ws), ws.numel(), _stream(stream)))
    return idx, w, logits


def k3moe_permute(idx, E: int, ws=None, stream=None):
    """Histogram, scan and permutation: dict counts, offsets, perm, inv (int32)."""
    _dev(idx, "idx")
    T, k = idx.shape
    dev = idx.device
    out = {
        "counts": torch.empty(E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "perm": torch.empty(T * k, dtype=torch.int32, device=dev),
        "inv": torch.empty(T * k, dtype=torch.int32, device=dev),
    }
    if ws is None:
        ws = workspace(k3moe_route_workspace_size(T, E), dev)
    _check(lib().k3moe_permute(_p(idx), T, k, E, _p(out["counts"]), _p(out["offsets"]),
                               _p(out["perm"]), _p(out["inv"]), _p(ws), ws.numel(),
                               _stream(stream)))
    return out


def k3moe_rmsnorm(h, gamma, eps: float, out=None, stream=None):
    h, gamma = _bf16(h, "h"), _bf16(gamma, "gamma")
    T, D = h.shape
    if out is None:
        out = torch.empty_like(h)
    _check(lib().k3moe_rmsnorm(_p(h), T, D, _p(gamma), float(eps), _p(out), _stream(stream)))
    return out


def k3moe_gemm_bf16(x, w, out_fp32: bool = False, out=None, stream=None):
    """out[t, n] = sum_c x[t, c] w[n, c] on tcgen05 (bf16 in, fp32 accumulate)."""
    x, w = _bf16(x, "x"), _bf16(w, "w")
    T, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((T, N), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=x.device)
    _check(lib().k3moe_gemm_bf16(_p(x), _p(w), T, N, K, _p(out), 1 if out_fp32 else 0,
                                 _stream(stream)))
    return out


def k3moe_prepared_scales_size(E: int, rows: int, cols: int) -> int:
    return lib().k3moe_prepared_scales_size(E, rows, cols)


def k3moe_prepare_scales(scale, stream=None):
    """Canonical E8M0 scales [E, rows, cols/32] (or [rows, cols/32], one
    expert) -> the prepared atoms the kernels can read instead, a flat uint8
    tensor of k3moe_prepared_scales_size(E, rows, cols) bytes."""
    _dev(scale, "scale")
    E = scale.shape[0] if scale.dim() == 3 else 1
    rows, cols = scale.shape[-2], 32 * scale.shape[-1]
    sf = torch.empty(k3moe_prepared_scales_size(E, rows, cols), dtype=torch.uint8, device=scale.device)
    _check(lib().k3moe_prepare_scales(_p(scale), E, rows, cols, _p(sf), _stream(stream)))
    return sf


def k3moe_unprepare_scales(sf, shape, stream=None):
    """Inverse of k3moe_prepare_scales: the canonical array of ``shape``
    ([E, rows, cols/32] or [rows, cols/32])."""
    scale = torch.empty(shape, dtype=torch.uint8, device=sf.device)
    E = scale.shape[0] if scale.dim() == 3 else 1
    _check(lib().k3moe_unprepare_scales(_p(sf), E, scale.shape[-2], 32 * scale.shape[-1], _p(scale),
                                        _stream(stream)))
    return scale


class MoELayer:
    """Device tensors of one layer plus the ``k3moe_layer_desc`` that points at them.

    Takes the expert weights as the checkpoint stores them: codes (w*_q) and
    canonical E8M0 scales (w*_s, one byte per row and 32 inputs).  With
    ``prepared=True`` it also keeps the scales in the prepared atom layout
    (k3moe_prepare_scales, run once here on the current stream), which the
    kernels then read instead."""

    def __init__(self, *, w1_q, w1_s, w3_q, w3_s, w2_q, w2_s, router_w, router_b, k: int,
                 norm_gamma=None, w_down=None, w_up=None, eps: float = 1e-5,
                 path: int = PATH_AUTO, act: int = ACT_SILU_GATED, prepared: bool = False):
        self.tensors = dict(w1_q=w1_q, w3_q=w3_q, w2_q=w2_q, w1_s=w1_s, w3_s=w3_s, w2_s=w2_s,
                            router_w=_bf16(router_w, "router_w"), router_b=router_b)
        if prepared:
            self.tensors.update(w1_sf=k3moe_prepare_scales(w1_s), w3_sf=k3moe_prepare_scales(w3_s),
                                w2_sf=k3moe_prepare_scales(w2_s))
        E, f, half_d = w1_q.shape
        d = 2 * half_d
        block = w_down is not None
        if block:
            self.tensors.update(norm_gamma=_bf16(norm_gamma, "norm_gamma"),
                                w_down=_bf16(w_down, "w_down"), w_up=_bf16(w_up, "w_up"))
        D = w_down.shape[1] if block else 0
        desc = LayerDesc()
        desc.E, desc.k, desc.d, desc.f = E, k, d, f
        desc.d_router = D if block else d
        desc.act, desc.path, desc.D, desc.eps, desc.format = act, path, D, eps, FORMAT_SPLIT
        for name, t in self.tensors.items():
            setattr(desc, name, t.data_ptr())
        self.desc = desc
        self.E, self.k, self.d, self.f, self.D = E, k, d, f, D
        self.prepared = prepared

    def with_path(self, path: int) -> "MoELayer":
        other = object.__new__(MoELayer)
        other.__dict__.update(self.__dict__)
        desc = LayerDesc.from_buffer_copy(self.desc)
        desc.path = path
        other.desc = desc
        return other

    @property
    def width(self) -> int:
        return self.D if self.D else self.d


def k3moe_workspace_size(layer: MoELayer, T: int) -> int:
    return lib().k3moe_workspace_size(ctypes.byref(layer.desc), T)


def k3moe_host_staging_size(layer: MoELayer, T: int) -> int:
    return lib().k3moe_host_staging_size(ctypes.byref(layer.desc), T)


def k3moe_forward(layer: MoELayer, hidden, out=None, ws=None, stream=None):
    """The layer (or block) on device tensors: hidden [T, width] bf16 -> out [T, width] bf16."""
    hidden = _bf16(hidden, "hidden")
    T = hidden.shape[0]
    if out is None:
        out = torch.empty_like(hidden)
    if ws is None:
        ws = workspace(k3moe_workspace_size(layer, T), hidden.device)
    _check(lib().k3moe_forward(ctypes.byref(layer.desc), _p(hidden), T, _p(out), _p(ws),
                               ws.numel(), _stream(stream)))
    return out


def k3moe_forward_routed(layer: MoELayer, hidden, idx, wts, out=None, ws=None, stream=None):
    """The layer's experts and combine on the caller's selection: hidden [T, d]
    bf16, idx [T, k] int32, wts [T, k] fp32 (device) -> out [T, d] bf16."""
    hidden = _bf16(hidden, "hidden")
    _dev(idx, "idx"), _dev(wts, "wts")
    if idx.dtype != torch.int32 or wts.dtype != torch.float32:
        raise TypeError("idx must be int32 and wts float32")
    T = hidden.shape[0]
    if out is None:
        out = torch.empty_like(hidden)
    if ws is None:
        ws = workspace(k3moe_workspace_size(layer, T), hidden.device)
    _check(lib().k3moe_forward_routed(ctypes.byref(layer.desc), _p(hidden), T, _p(idx), _p(wts), _p(out),
                                      _p(ws), ws.numel(), _stream(stream)))
    return out


def k3moe_forward_host(layer: MoELayer, hidden_host: torch.Tensor, out_host=None, ws=None,
                       stream=None):
    """The layer on HOST tensors (bf16, ideally pinned); copies happen inside the call."""
    if hidden_host.is_cuda or not hidden_host.is_contiguous():
        raise ValueError("hidden_host must be a contiguous host tensor")
    if hidden_host.dtype in (torch.int16, torch.uint16):
        hidden_host = hidden_host.view(torch.bfloat16)
    T = hidden_host.shape[0]
    if out_host is None:
        out_host = torch.empty_like(hidden_host, pin_memory=hidden_host.is_pinned())
    if ws is None:
        ws = workspace(k3moe_workspace_size(layer, T) + k3moe_host_staging_size(layer, T))
    _check(lib().k3moe_forward_host(ctypes.byref(layer.desc), _p(hidden_host), T, _p(out_host),
                                    _p(ws), ws.numel(), _stream(stream)))
    return out_host


def k3moe_forward_routing(layer: MoELayer, ws, T: int, with_logits: bool = True, stream=None):
    dev = ws.device
    idx = torch.empty((T, layer.k), dtype=torch.int32, device=dev)
    w = torch.empty((T, layer.k), dtype=torch.float32, device=dev)
    logits = torch.empty((T, layer.E), dtype=torch.float32, device=dev) if with_logits else None
    _check(lib().k3moe_forward_routing(ctypes.byref(layer.desc), _p(ws), T, _p(idx), _p(w),
                                       _p(logits), _stream(stream)))
    return idx, w, logits


def k3moe_forward_intermediates(layer: MoELayer, ws, T: int, stream=None):
    """Block mode: (hn [T, D], z [T, d], m [T, d]) bf16 of the last forward on ``ws``."""
    dev = ws.device
    hn = torch.empty((T, layer.D), dtype=torch.bfloat16, device=dev)
    z = torch.empty((T, layer.d), dtype=torch.bfloat16, device=dev)
    m = torch.empty((T, layer.d), dtype=torch.bfloat16, device=dev)
    _check(lib().k3moe_forward_intermediates(ctypes.byref(layer.desc), _p(ws), T, _p(hn), _p(z), _p(m),
                                             _stream(stream)))
    return hn, z, m


def k3moe_get_status(ws, stream=None) -> int:
    """Synchronise and return (and clear) the workspace's device status word."""
    st = ctypes.c_int32(0)
    _check(lib().k3moe_get_status(_p(ws), _stream(stream), ctypes.byref(st)))
    return st.value


def k3moe_trace(mode) -> int:
    """Set kernel tracing of k3moe_forward: 0 off, 1 events between launches,
    2 device stamps (start / end of each kernel inside the forward), 3 both.
    True / False are 1 / 0.  Returns the previous mode."""
    return int(lib().k3moe_trace(int(mode)))


def k3moe_trace_read(max_entries: int = 32):
    """[(kernel name, ms)] of the most recent event-traced forward (waits for its events)."""
    names = (ctypes.c_char_p * max_entries)()
    ms = (ctypes.c_float * max_entries)()
    n = lib().k3moe_trace_read(max_entries, names, ms)
    return [(names[i].decode(), float(ms[i])) for i in range(n)]


def k3moe_trace_read_stamps(max_entries: int = 48):
    """[(kernel name, start us, end us)] of the most recent stamped forward
    (device times after the earliest start; synchronises the device)."""
    names = (ctypes.c_char_p * max_entries)()
    st = (ctypes.c_double * max_entries)()
    en = (ctypes.c_double * max_entries)()
    n = lib().k3moe_trace_read_stamps(max_entries, names, st, en)
    return [(names[i].decode(), float(st[i]), float(en[i])) for i in range(n)]


def expert_arrays(layer: MoELayer):
    """Names of the six expert arrays the kernels read: the codes and either
    the prepared or the canonical scales."""
    sc = ("w1_sf", "w3_sf", "w2_sf") if layer.prepared else ("w1_s", "w3_s", "w2_s")
    return ("w1_q", "w3_q", "w2_q") + sc


def ggml_layer(layer: MoELayer, stream=None) -> MoELayer:
    """A copy of ``layer`` whose expert matrices are llama.cpp's MXFP4 blocks
    ([E, rows, K/32, 17], written by k3moe_repack_mxfp4 from the codes and the
    canonical scales), descriptor format K3MOE_FORMAT_GGML.  Router and
    block-mode tensors stay shared with ``layer``."""
    other = object.__new__(MoELayer)
    other.__dict__.update(layer.__dict__)
    other.tensors = dict(layer.tensors)
    desc = LayerDesc.from_buffer_copy(layer.desc)
    for m in ("w1", "w3", "w2"):
        codes, canon = layer.tensors[m + "_q"], layer.tensors[m + "_s"]
        E, rows, half = codes.shape
        K = 2 * half
        blocks = k3moe_repack_mxfp4(codes.view(E * rows, half), canon.view(E * rows, K // 32),
                                    stream=stream)
        other.tensors[m + "_q"] = blocks.view(E, rows, K // 32, 17)
        for sc in (m + "_s", m + "_sf"):
            other.tensors.pop(sc, None)
            setattr(desc, sc, None)
        setattr(desc, m + "_q", blocks.data_ptr())
    desc.format = FORMAT_GGML
    other.desc = desc
    other.prepared = False
    return other


def host_resident(layer: MoELayer) -> MoELayer:
    """A copy of ``layer`` whose six expert arrays (codes and the scales the
    kernels read) live in one page-locked host buffer, for
    k3moe_forward_cached.  The router and block-mode tensors stay shared with
    ``layer``; the device expert arrays are referenced only by ``layer``
    (drop it to free them)."""
    align = 256
    names = expert_arrays(layer)
    offs, total = [], 0
    for n in names:
        offs.append(total)
        total += (layer.tensors[n].numel() + align - 1) // align * align
    buf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    other = object.__new__(MoELayer)
    other.__dict__.update(layer.__dict__)
    other.tensors = dict(layer.tensors)
    desc = LayerDesc.from_buffer_copy(layer.desc)
    for n in ("w1_s", "w3_s", "w2_s", "w1_sf", "w3_sf", "w2_sf"):
        if n not in names:  # the other scale layout is not kept on the host
            other.tensors.pop(n, None)
            setattr(desc, n, None)
    for n, off in zip(names, offs):
        src = layer.tensors[n]
        view = buf[off:off + src.numel()].view(src.shape)
        view.copy_(src)
        other.tensors[n] = view
        setattr(desc, n, view.data_ptr())
    other.desc = desc
    other.host_buffer = buf
    return other


class ExpertCache:
    """Device slots and bookkeeping of a ``k3moe_expert_cache`` (initialised
    here with k3moe_cache_init on the current stream)."""

    def __init__(self, layer: MoELayer, slots: int, device=None, stream=None):
        dev = device or "cuda"
        E, d, f = layer.E, layer.d, layer.f
        u8 = torch.uint8
        # the slots' scales in the layer's layout: prepared atoms or canonical rows
        nsc = k3moe_prepared_scales_size(slots, f, d) if layer.prepared else slots * f * d // 32
        self.tensors = dict(
            w1_q=torch.empty((slots, f, d // 2), dtype=u8, device=dev),
            w3_q=torch.empty((slots, f, d // 2), dtype=u8, device=dev),
            w2_q=torch.empty((slots, d, f // 2), dtype=u8, device=dev),
            w1_s=torch.empty(nsc, dtype=u8, device=dev),
            w3_s=torch.empty(nsc, dtype=u8, device=dev),
            w2_s=torch.empty(nsc, dtype=u8, device=dev),
            state=torch.zeros(max(int(lib().k3moe_cache_state_size(E, slots)), 256), dtype=u8,
                              device=dev),
        )
        desc = CacheDesc()
        desc.slots, desc.reserved = slots, 0
        for name, t in self.tensors.items():
            setattr(desc, name, t.data_ptr())
        self.desc = desc
        self.E, self.slots = E, slots
        _check(lib().k3moe_cache_init(_p(self.tensors["state"]), E, slots, _stream(stream)))

    def reset(self, stream=None):
        _check(lib().k3moe_cache_init(_p(self.tensors["state"]), self.E, self.slots,
                                      _stream(stream)))

    def stats(self, stream=None) -> dict:
        """k3moe_cache_read_stats (synchronises the stream)."""
        st = CacheStats()
        _check(lib().k3moe_cache_read_stats(_p(self.tensors["state"]), _stream(stream),
                                            ctypes.byref(st)))
        return {name: int(getattr(st, name)) for name, _ in CacheStats._fields_}

    def maps(self):
        """(slot_of [E], expert_of [S], stamp [S]) as device int tensors (views of the state)."""
        st = self.tensors["state"]
        E, S = self.E, self.slots
        al = lambda n: (n * 4 + 255) // 256 * 256  # noqa: E731
        o1 = 256
        o2 = o1 + al(E)
        o3 = o2 + al(S)
        slot_of = st[o1:o1 + 4 * E].view(torch.int32)
        expert_of = st[o2:o2 + 4 * S].view(torch.int32)
        stamp = st[o3:o3 + 4 * S].view(torch.int32)
        return slot_of, expert_of, stamp


def k3moe_cache_state_size(E: int, slots: int) -> int:
    return lib().k3moe_cache_state_size(E, slots)


def k3moe_forward_cached(layer: MoELayer, cache: ExpertCache, hidden, out=None, ws=None,
                         stream=None):
    """k3moe_forward with host-resident expert arrays (``host_resident``) behind ``cache``."""
    hidden = _bf16(hidden, "hidden")
    T = hidden.shape[0]
    if out is None:
        out = torch.empty_like(hidden)
    if ws is None:
        ws = workspace(k3moe_workspace_size(layer, T), hidden.device)
    _check(lib().k3moe_forward_cached(ctypes.byref(layer.desc), ctypes.byref(cache.desc),
                                      _p(hidden), T, _p(out), _p(ws), ws.numel(),
                                      _stream(stream)))
    return out


class ForwardGraph:
    """A CUDA graph of one k3moe_forward (or, with ``cache``, one
    k3moe_forward_cached) with fixed buffers (k3moe_graph_create[_cached])."""

    def __init__(self, layer: MoELayer, hidden, out, ws, cache: "ExpertCache | None" = None):
        hidden = _bf16(hidden, "hidden")
        self._keep = (layer, hidden, out, ws, cache)
        h = ctypes.c_void_p(None)
        if cache is None:
            _check(lib().k3moe_graph_create(ctypes.byref(layer.desc), _p(hidden), hidden.shape[0],
                                            _p(out), _p(ws), ws.numel(), ctypes.byref(h)))
        else:
            _check(lib().k3moe_graph_create_cached(ctypes.byref(layer.desc),
                                                   ctypes.byref(cache.desc), _p(hidden),
                                                   hidden.shape[0], _p(out), _p(ws), ws.numel(),
                                                   ctypes.byref(h)))
        self.handle = h

    def launch(self, stream=None):
        _check(lib().k3moe_graph_launch(self.handle, _stream(stream)))

    def close(self):
        if self.handle:
            lib().k3moe_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def k3moe_graph_create(layer: MoELayer, hidden, out, ws) -> ForwardGraph:
    return ForwardGraph(layer, hidden, out, ws)


def k3moe_graph_launch(graph: ForwardGraph, stream=None):
    graph.launch(stream)


def k3moe_graph_destroy(graph: ForwardGraph):
    graph.close()
