"""Host-side checks of the C ABI: the library loads, exports every entry
point the header declares, sizes workspaces, and rejects bad arguments
before anything is enqueued (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moeq4k.h")


@pytest.fixture(scope="module")
def lib():
    from quantized_routed_expert_02_gb300 import build
    build.build()
    return ctypes.CDLL(build.LIB)


@pytest.fixture(scope="module")
def m(lib):
    from quantized_routed_expert_02_gb300 import moeq4k
    return moeq4k


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("moe_router", "moe_ffn", "moe_layer", "moe_permute", "moe_workspace_bytes",
                 "moe_read_device_status", "moe_status_str"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in moeq4k.h but not exported"


def test_binding_covers_every_symbol(m):
    assert sorted(m.EXPORTS) == declared_functions()


def test_status_strings(m):
    assert m.status_str(0) == "MOE_OK"
    assert m.status_str(5) == "MOE_ERR_EXPERT_RANGE"
    assert m.status_str(99) == "MOE_ERR_UNKNOWN"


def test_workspace_bytes(m):
    T, H, E, k, I = 4096, 2048, 128, 8, 768
    n = m.moe_workspace_bytes(T, H, E, k, I)
    # h [T*k, I] and per-slot outputs [T*k, H] in fp32, the fp16 copies of
    # x [T*k, H] (expert-sorted rows) and h [T*k, I] used by the tensor-core
    # path, and the normalised FFN input [T, H] in fp32 dominate
    big = 4 * T * k * (I + H) + 2 * T * k * H + 2 * T * k * I + 4 * T * H
    assert n >= big
    assert n < big + (8 << 20)
    assert m.moe_workspace_bytes_host(T, H, E, k, I) >= n + 2 * 4 * T * H
    assert m.moe_workspace_bytes(0, H, E, k, I) == 0
    assert m.moe_workspace_bytes(1, 2000, E, k, I) == 0      # H not a multiple of 256
    assert m.moe_workspace_bytes(1, H, 8, 9, I) == 0          # k > E
    assert m.moe_workspace_bytes(1, H, 300, 8, I) == 0        # E above the limit


ALIGNED = 1 << 20     # any 256-aligned non-null value: never dereferenced on these paths


@pytest.mark.parametrize("args,code", [
    ((1, 2048, 128, 8, 768), 0),
    ((0, 2048, 128, 8, 768), 1),
    ((1, 2048, 128, 0, 768), 1),
    ((1, 2048, 4, 8, 768), 1),
    ((1, 2048, 128, 8, 700), 1),
    ((1, 300, 128, 8, 768), 1),
])
def test_ffn_shape_errors(lib, args, code):
    T, H, E, k, I = args
    if code == 0:
        return
    P = ctypes.c_void_p
    f = lib.moe_ffn
    f.restype = ctypes.c_int
    r = f(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), T, H, E, k, I,
          P(ALIGNED), P(ALIGNED), ctypes.c_size_t(1 << 40), P(None))
    assert r == code


def _ffn(lib, x=ALIGNED, idx=ALIGNED, w=ALIGNED, g=ALIGNED, u=ALIGNED, d=ALIGNED, y=ALIGNED,
         ws=ALIGNED, ws_bytes=1 << 40, dims=(1, 2048, 128, 8, 768)):
    P = ctypes.c_void_p
    f = lib.moe_ffn
    f.restype = ctypes.c_int
    return f(P(x), P(idx), P(w), P(g), P(u), P(d), *dims, P(y), P(ws), ctypes.c_size_t(ws_bytes),
             P(None))


def test_ffn_null_pointers(lib):
    assert _ffn(lib, x=0) == 2
    assert _ffn(lib, d=0) == 2
    assert _ffn(lib, ws=0) == 2


def test_ffn_misaligned(lib):
    assert _ffn(lib, x=ALIGNED + 4) == 3
    assert _ffn(lib, g=ALIGNED + 8) == 3
    assert _ffn(lib, ws=ALIGNED + 16) == 3


def test_ffn_workspace_too_small(lib, m):
    need = m.moe_workspace_bytes(1, 2048, 128, 8, 768)
    assert _ffn(lib, ws_bytes=need - 1) == 4


def test_router_errors(lib):
    P = ctypes.c_void_p
    f = lib.moe_router
    f.restype = ctypes.c_int
    args = lambda x=ALIGNED, k=8, E=128: (P(x), P(ALIGNED), P(None), 1, 2048, E, k, P(ALIGNED),
                                          P(ALIGNED), P(ALIGNED), ctypes.c_size_t(1 << 30), P(None))
    assert f(*args(x=0)) == 2
    assert f(*args(k=129)) == 1
    assert f(*args(k=33, E=64)) == 1
    assert f(*args(x=ALIGNED + 4)) == 3


def test_layer_host_null(lib):
    P = ctypes.c_void_p
    f = lib.moe_layer_host
    f.restype = ctypes.c_int
    r = f(P(None), P(ALIGNED), P(None), P(ALIGNED), P(ALIGNED), P(ALIGNED), 1, 2048, 128, 8, 768,
          P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), ctypes.c_size_t(1 << 40), P(None))
    assert r == 2


def _fn(lib, name):
    f = getattr(lib, name)
    f.restype = ctypes.c_int
    return f


def test_layer_errors(lib):
    """moe_layer: shape, null, alignment and workspace errors, in that order."""
    P, S = ctypes.c_void_p, ctypes.c_size_t
    f = _fn(lib, "moe_layer")

    def call(x=ALIGNED, bias=None, y=ALIGNED, T=1, k=8, ws=ALIGNED, ws_bytes=1 << 40):
        return f(P(x), P(ALIGNED), P(bias), P(ALIGNED), P(ALIGNED), P(ALIGNED), T, 2048, 128, k,
                 768, P(ALIGNED), P(ALIGNED), P(y), P(ws), S(ws_bytes), P(None))
    assert call(T=0) == 1
    assert call(k=0) == 1
    assert call(x=0) == 2
    assert call(y=0) == 2
    assert call(x=ALIGNED + 8) == 3
    assert call(bias=ALIGNED + 4) == 3
    assert call(ws=0) == 2
    assert call(ws=ALIGNED + 16) == 3          # the workspace is 256-byte aligned
    assert call(ws_bytes=1024) == 4


def test_layer_block_errors(lib):
    """moe_layer_block: eps must be finite and >= 0, capture_token in [-1, T),
    the capture buffers aligned."""
    P, S = ctypes.c_void_p, ctypes.c_size_t
    f = _fn(lib, "moe_layer_block")

    def call(eps=1e-6, cap=-1, cap_idx=None, cap_ffn=None, norm_w=None, T=2):
        return f(P(ALIGNED), P(norm_w), ctypes.c_float(eps), P(ALIGNED), P(None), P(ALIGNED),
                 P(ALIGNED), P(ALIGNED), T, 2048, 128, 8, 768, P(ALIGNED), P(ALIGNED), P(ALIGNED),
                 1, cap, P(cap_idx), P(None), P(cap_ffn), P(ALIGNED), S(1024), P(None))
    assert call(eps=-1.0) == 1
    assert call(eps=float("nan")) == 1
    assert call(eps=float("inf")) == 1
    assert call(cap=-2) == 1
    assert call(cap=2) == 1                     # T = 2: tokens 0 and 1
    assert call(norm_w=ALIGNED + 4) == 3
    assert call(cap=0, cap_idx=ALIGNED + 2) == 3
    assert call(cap=0, cap_ffn=ALIGNED + 4) == 3
    assert call(cap=1) == 4                     # valid so far; the 1 KB workspace is too small


def test_permute_errors(lib):
    P, S = ctypes.c_void_p, ctypes.c_size_t
    f = _fn(lib, "moe_permute")

    def call(idx=ALIGNED, T=5, k=4, E=16, perm=ALIGNED, ws_bytes=1 << 40):
        return f(P(idx), T, k, E, P(ALIGNED), P(ALIGNED), P(perm), P(ALIGNED), S(ws_bytes), P(None))
    assert call(T=0) == 1
    assert call(k=17) == 1                      # k > E
    assert call(idx=0) == 2
    assert call(perm=ALIGNED + 4) == 3
    assert call(ws_bytes=16) == 4


def test_workspace_init_errors(lib):
    P, S = ctypes.c_void_p, ctypes.c_size_t
    f = _fn(lib, "moe_workspace_init")
    assert f(P(None), S(1 << 20), P(None)) == 2
    assert f(P(ALIGNED + 128), S(1 << 20), P(None)) == 3
    assert f(P(ALIGNED), S(8), P(None)) == 4


def test_q8k_errors(lib):
    P, S = ctypes.c_void_p, ctypes.c_size_t
    q = _fn(lib, "moe_quantize_q8k")
    assert q(P(ALIGNED), 0, 256, P(ALIGNED), P(ALIGNED), P(ALIGNED), P(None)) == 1
    assert q(P(ALIGNED), 2, 300, P(ALIGNED), P(ALIGNED), P(ALIGNED), P(None)) == 1  # n % 256
    assert q(P(None), 2, 256, P(ALIGNED), P(ALIGNED), P(ALIGNED), P(None)) == 2
    assert q(P(ALIGNED + 4), 2, 256, P(ALIGNED), P(ALIGNED), P(ALIGNED), P(None)) == 3
    for name in ("moe_ffn_q8k", "moe_layer_q8k"):
        f = _fn(lib, name)
        if name == "moe_ffn_q8k":
            call = lambda x=ALIGNED, T=1, ws_bytes=1 << 40: f(  # noqa: E731
                P(x), P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), T, 2048, 128, 8,
                768, P(ALIGNED), P(ALIGNED), S(ws_bytes), P(None))
        else:
            call = lambda x=ALIGNED, T=1, ws_bytes=1 << 40: f(  # noqa: E731
                P(x), P(ALIGNED), P(None), P(ALIGNED), P(ALIGNED), P(ALIGNED), T, 2048, 128, 8,
                768, P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), S(ws_bytes), P(None))
        assert call(T=0) == 1, name
        assert call(x=0) == 2, name
        assert call(x=ALIGNED + 4) == 3, name
        assert call(ws_bytes=1024) == 4, name


def test_noalloc_errors(lib):
    """moe_layer_noalloc: one token only, k*I within the fixed scratch."""
    P = ctypes.c_void_p
    f = _fn(lib, "moe_layer_noalloc")

    def call(T=1, k=8, I=768, E=128, x=ALIGNED):
        return f(P(x), P(ALIGNED), P(None), P(ALIGNED), P(ALIGNED), P(ALIGNED), T, 2048, E, k, I,
                 P(ALIGNED), P(ALIGNED), P(ALIGNED), P(None))
    assert call(T=2) == 1
    assert call(k=32, I=4096) == 9               # k*I above the scratch limit
    assert call(x=0) == 2
    assert call(x=ALIGNED + 4) == 3
