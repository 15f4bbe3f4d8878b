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
