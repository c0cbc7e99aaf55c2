"""The C ABI: library loads, exports what include/k3moe.h declares, the ctypes
struct matches the C layout, and host-side validation rejects bad calls
before anything reaches a GPU (CPU only)."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "k3moe.h")


@pytest.fixture(scope="module")
def k3():
    import __graft_entry__

    __graft_entry__.build()
    import mxfp4_routed_expert_sigmoid_gb300 as k3mod

    return k3mod


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(k3moe_\w+)\s*\(", text)))


def test_exports_match_header(k3):
    declared = header_functions()
    assert declared == sorted(k3.EXPORTS)
    L = k3.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert k3.k3moe_abi_version() == 4


def test_status_strings(k3):
    L = k3.lib()
    for code in range(9):
        assert L.k3moe_status_string(code)
    assert L.k3moe_status_string(99) == b"unknown status"


@pytest.mark.parametrize("py,c", [("LayerDesc", "k3moe_layer_desc"),
                                  ("CacheDesc", "k3moe_expert_cache"),
                                  ("CacheStats", "k3moe_cache_stats")])
def test_desc_layout_matches_c(k3, py, c):
    struct = getattr(k3, py)
    fields = [f for f, _ in struct._fields_]
    prog = "#include <stdio.h>\n#include <stddef.h>\n#include \"k3moe.h\"\nint main(void){\n"
    prog += f'printf("%zu\\n", sizeof({c}));\n'
    for f in fields:
        prog += f'printf("%zu\\n", offsetof({c}, {f}));\n'
    prog += "return 0;}\n"
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(src, "w").write(prog)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        vals = [int(v) for v in subprocess.run([exe], capture_output=True, text=True,
                                               check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(struct)
    for f, off in zip(fields, vals[1:]):
        assert getattr(struct, f).offset == off, f


A16 = 0x10000  # a fake 16-byte aligned address: validation rejects before any use
A1 = 0x10001


def desc(k3, **over):
    d = k3.LayerDesc()
    d.E, d.k, d.d, d.f, d.d_router = 896, 16, 3584, 3072, 3584
    d.act, d.path, d.D, d.eps, d.format = 0, 0, 0, 0.0, 0
    for name in ("w1_q", "w3_q", "w2_q", "w1_s", "w3_s", "w2_s", "router_w", "router_b"):
        setattr(d, name, A16)
    for k_, v in over.items():
        setattr(d, k_, v)
    return d


def test_repack_validation(k3):
    L = k3.lib()
    assert L.k3moe_repack_mxfp4(None, A16, 4, 64, A16, None) == 1
    assert L.k3moe_repack_mxfp4(A16, A16, 0, 64, A16, None) == 1
    assert L.k3moe_repack_mxfp4(A16, A16, 4, 48, A16, None) == 2
    assert L.k3moe_repack_mxfp4(A1, A16, 4, 64, A16, None) == 3
    assert L.k3moe_unpack_mxfp4(A16, 4, 40, A16, A16, None) == 2
    assert L.k3moe_unpack_mxfp4(A16, 4, 64, A1, A16, None) == 3


def test_prepare_scales_validation(k3):
    L = k3.lib()
    assert L.k3moe_prepare_scales(None, 1, 128, 256, A16, None) == 1
    assert L.k3moe_prepare_scales(A16, 0, 128, 256, A16, None) == 1
    assert L.k3moe_prepare_scales(A16, 1, 0, 256, A16, None) == 1
    assert L.k3moe_prepare_scales(A16, 1, 96, 256, A16, None) == 2
    assert L.k3moe_prepare_scales(A16, 1, 128, 352, A16, None) == 2
    assert L.k3moe_prepare_scales(A1, 1, 128, 256, A16, None) == 3
    assert L.k3moe_unprepare_scales(A16, 1, 128, 32, A16, None) == 2
    assert L.k3moe_unprepare_scales(A16, 1, 128, 256, None, None) == 1
    # per expert: ceil(rows / 128) tiles x ceil(cols / 128) groups x 512 bytes
    assert L.k3moe_prepared_scales_size(896, 3072, 3584) == 896 * 3072 * 3584 // 32
    assert L.k3moe_prepared_scales_size(8, 64, 64) == 8 * 512
    assert L.k3moe_prepared_scales_size(3, 192, 320) == 3 * 2 * 3 * 512
    assert L.k3moe_prepared_scales_size(0, 64, 64) == 0


def test_route_validation(k3):
    L = k3.lib()
    ws = L.k3moe_route_workspace_size(8, 896)
    assert ws > 8 * 896 * 4
    call = lambda **kw: L.k3moe_route(
        kw.get("x", A16), kw.get("T", 8), kw.get("d_r", 3584), A16, A16, kw.get("E", 896),
        kw.get("k", 16), A16, A16, None, kw.get("ws", A16), kw.get("ws_bytes", ws), None)
    assert call(x=None) == 1
    assert call(k=17, E=16) == 2
    assert call(k=33) == 2
    assert call(E=2048) == 2
    assert call(d_r=100) == 2
    assert call(x=A1) == 3
    assert call(ws_bytes=ws - 1) == 4
    assert L.k3moe_permute(A16, 8, 16, 896, A16, A16, A16, A16, A16, 0, None) == 4
    assert L.k3moe_permute(A16, 8, 40, 896, A16, A16, A16, A16, A16, 1 << 20, None) == 2


def test_forward_validation(k3):
    # every case fails validation before anything is launched (the pointers are fake)
    L = k3.lib()
    fwd = lambda dsc, **kw: L.k3moe_forward(ctypes.byref(dsc), kw.get("h", A16), kw.get("T", 1),
                                            A16, A16, kw.get("ws", 1 << 40), None)
    assert fwd(desc(k3, d=96, d_router=96)) == 2     # the MMAs take 64 inputs at a time
    assert fwd(desc(k3, f=3072 + 32)) == 2
    assert fwd(desc(k3, k=40)) == 2
    assert fwd(desc(k3, k=17, E=16)) == 2
    assert fwd(desc(k3, E=2000)) == 2
    assert fwd(desc(k3, act=1)) == 8
    assert fwd(desc(k3, format=2)) == 1
    # ggml blocks: no separate scales; rows of whole 16-byte units; streaming path only
    gg = dict(format=1, w1_s=None, w3_s=None, w2_s=None)
    assert fwd(desc(k3, w1_q=A16 + 16, **gg), ws=16) == 4
    assert fwd(desc(k3, d=3584 - 256, d_router=3584 - 256, **gg)) == 2
    assert fwd(desc(k3, f=3072 + 256, **gg)) == 2
    assert fwd(desc(k3, path=2, **gg)) == 8
    assert fwd(desc(k3, **gg), T=1025) == 8
    assert fwd(desc(k3, w2_q=A1, **gg)) == 3
    assert fwd(desc(k3, path=7)) == 1
    # scales: the canonical arrays, or all three prepared arrays
    assert fwd(desc(k3, w2_s=None)) == 1
    assert fwd(desc(k3, w1_s=None, w3_s=None, w2_s=None)) == 1
    assert fwd(desc(k3, w1_sf=A16)) == 1                # one prepared array without the others
    assert fwd(desc(k3, w1_sf=A16, w3_sf=A16, w2_sf=A1)) == 3
    assert fwd(desc(k3, w1_sf=A16, w3_sf=A16, w2_sf=A16, w1_s=None, w3_s=None, w2_s=None), ws=16) == 4
    assert fwd(desc(k3, w3_s=A1)) == 3
    assert fwd(desc(k3, w3_q=A1)) == 3
    assert fwd(desc(k3, w2_q=A16 + 16)) == 3  # E2M1 codes: 32-byte aligned for TMA
    assert fwd(desc(k3, d_router=7168)) == 2
    assert fwd(desc(k3, D=7168, d_router=7168)) == 1  # block mode without its tensors
    assert fwd(desc(k3), h=A1) == 3
    assert fwd(desc(k3), ws=16) == 4
    assert fwd(desc(k3, path=1), T=1025) == 8  # the streaming kernels take at most 1024 tokens
    # a workspace one byte short of the plan, for widths whose scales are
    # prepared per call (d, f not multiples of 512) and for the K3 widths
    for over in (dict(d=64, f=64, d_router=64, E=8, k=2), dict()):
        dd = desc(k3, **over)
        need = L.k3moe_workspace_size(ctypes.byref(dd), 4)
        assert fwd(dd, T=4, ws=need - 1) == 4
    small = desc(k3, d=64, f=64, d_router=64, E=8, k=2)
    prep = desc(k3, d=64, f=64, d_router=64, E=8, k=2, w1_sf=A16, w3_sf=A16, w2_sf=A16)
    # the per-call preparation takes workspace room that prepared scales do not
    assert L.k3moe_workspace_size(ctypes.byref(small), 4) > L.k3moe_workspace_size(ctypes.byref(prep), 4)


def cache_desc(k3, **over):
    c = k3.CacheDesc()
    c.slots, c.reserved = 64, 0
    for name in ("w1_q", "w3_q", "w2_q", "w1_s", "w3_s", "w2_s", "state"):
        setattr(c, name, A16)
    for k_, v in over.items():
        setattr(c, k_, v)
    return c


def test_cache_validation(k3):
    """Host checks of the cached forward and the cache set-up (no launch)."""
    L = k3.lib()

    def fwd(dsc, c, T=1):
        return L.k3moe_forward_cached(ctypes.byref(dsc), None if c is None else ctypes.byref(c),
                                      A16, T, A16, A16, 1 << 40, None)

    assert fwd(desc(k3), None) == 1
    assert fwd(desc(k3), cache_desc(k3, reserved=1)) == 1
    assert fwd(desc(k3), cache_desc(k3, state=None)) == 1
    assert fwd(desc(k3), cache_desc(k3, slots=15)) == 2   # fewer slots than one token's experts
    assert fwd(desc(k3), cache_desc(k3, slots=897)) == 2  # more slots than experts
    assert fwd(desc(k3), cache_desc(k3), T=8) == 2        # 8 tokens may use 128 experts
    assert fwd(desc(k3), cache_desc(k3, w2_q=A16 + 16)) == 3
    assert fwd(desc(k3), cache_desc(k3, w3_s=A1)) == 3
    # canonical scales whose rows are not whole 512-input stages: no cache
    assert fwd(desc(k3, d=768, d_router=768), cache_desc(k3)) == 8
    assert fwd(desc(k3), cache_desc(k3, w1_q=None)) == 1
    assert fwd(desc(k3, path=2), cache_desc(k3)) == 8     # the grouped path has no cache
    assert fwd(desc(k3), cache_desc(k3), T=2000) == 8
    assert fwd(desc(k3, k=40), cache_desc(k3)) == 2       # the layer checks come first
    assert L.k3moe_cache_state_size(896, 0) == 0
    st = L.k3moe_cache_state_size(896, 160)
    assert st >= 256 + 896 * 4 + 4 * 160 * 4
    assert L.k3moe_cache_init(None, 896, 160, None) == 1
    assert L.k3moe_cache_init(A16, 896, 900, None) == 2
    assert L.k3moe_cache_init(A16, 2000, 160, None) == 2
    assert L.k3moe_cache_init(A1, 896, 160, None) == 3
    assert L.k3moe_cache_read_stats(None, None, None) == 1


def test_workspace_sizes(k3):
    L = k3.lib()
    d = desc(k3)
    sizes = [L.k3moe_workspace_size(ctypes.byref(d), T) for T in (1, 8, 512, 8192)]
    assert all(b > a for a, b in zip(sizes, sizes[1:]))
    # at least the fp32 staging of every (token, expert) output row
    assert sizes[-1] >= 8192 * 16 * 3584 * 4
    assert L.k3moe_workspace_size(None, 1) == 0
    blk = desc(k3, D=7168, d_router=7168)
    assert L.k3moe_workspace_size(ctypes.byref(blk), 64) > L.k3moe_workspace_size(ctypes.byref(d), 64)
    assert L.k3moe_host_staging_size(ctypes.byref(blk), 64) == 2 * 64 * 7168 * 2


def test_binding_fails_loudly_without_library(k3, monkeypatch):
    monkeypatch.setattr(k3, "_lib", None)
    monkeypatch.setattr(k3, "LIB_PATH", "/nonexistent/libk3moe.so")
    with pytest.raises(ImportError):
        k3.lib()
