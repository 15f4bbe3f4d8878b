"""Python binding of the moeq4k C ABI (``libmoeq4k.so``).

Argument marshalling only: tensors become raw device pointers, the stream
defaults to PyTorch's current stream, and a non-OK status raises
``MoeError``.  Every step of the layer runs in the library's CUDA kernels;
there is no Python or CPU fallback.  Importing this module without the
built library raises immediately.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoeq4k.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m quantized_routed_expert_02_gb300.build` "
        "(or __graft_entry__.build()); the moeq4k layer has no fallback path")

_lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_S = ctypes.c_size_t

_SIGS = {
    "moe_status_str": ([ctypes.c_int], ctypes.c_char_p),
    "moe_version": ([], ctypes.c_int),
    "moe_workspace_bytes": ([_I, _I, _I, _I, _I], _S),
    "moe_workspace_bytes_host": ([_I, _I, _I, _I, _I], _S),
    "moe_layer_launch_count": ([_I, _I, _I, _I, _I], ctypes.c_int),
    "moe_workspace_init": ([_P, _S, _P], ctypes.c_int),
    "moe_router": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _S, _P], ctypes.c_int),
    "moe_permute": ([_P, _I, _I, _I, _P, _P, _P, _P, _S, _P], ctypes.c_int),
    "moe_ffn": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _S, _P], ctypes.c_int),
    "moe_layer": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _S, _P],
                  ctypes.c_int),
    "moe_layer_host": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _S, _P],
                       ctypes.c_int),
    "moe_layer_block": ([_P, _P, ctypes.c_float, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P,
                         _P, _I, _I, _P, _P, _P, _P, _S, _P], ctypes.c_int),
    "moe_quantize_q8k": ([_P, _I, _I, _P, _P, _P, _P], ctypes.c_int),
    "moe_ffn_q8k": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _S, _P], ctypes.c_int),
    "moe_layer_q8k": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _S, _P],
                      ctypes.c_int),
    "moe_layer_q8k_launch_count": ([_I, _I, _I, _I, _I], ctypes.c_int),
    "moe_read_device_status": ([_P, _P, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
    "moe_layer_noalloc": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P],
                          ctypes.c_int),
    "moe_debug_set_wait_limit": ([ctypes.c_ulonglong], None),
    "moe_debug_withhold_arrivals": ([_I], None),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTS = tuple(_SIGS)

MOE_OK = 0
STATUS_NAMES = {i: _lib.moe_status_str(i).decode() for i in range(10)}


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")


def _check(code: int, where: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def status_str(code: int) -> str:
    return _lib.moe_status_str(int(code)).decode()


def version() -> int:
    return _lib.moe_version()


def moe_workspace_bytes(T, H, E, k, I) -> int:
    return _lib.moe_workspace_bytes(T, H, E, k, I)


def moe_workspace_bytes_host(T, H, E, k, I) -> int:
    return _lib.moe_workspace_bytes_host(T, H, E, k, I)


def moe_layer_launch_count(T, H, E, k, I) -> int:
    return _lib.moe_layer_launch_count(T, H, E, k, I)


def moe_layer_q8k_launch_count(T, H, E, k, I) -> int:
    return _lib.moe_layer_q8k_launch_count(T, H, E, k, I)


def alloc_workspace(T, H, E, k, I, device="cuda", host_staging=False) -> torch.Tensor:
    """A uint8 device workspace of the right size, initialised with
    moe_workspace_init (header and tag region zeroed)."""
    n = (moe_workspace_bytes_host if host_staging else moe_workspace_bytes)(T, H, E, k, I)
    if n == 0:
        raise MoeError(1, "moe_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws)
    return ws


def moe_workspace_init(ws, stream=None) -> None:
    _check(_lib.moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "moe_workspace_init")


def moe_router(x, Wr, bias, k, idx, w, ws, stream=None) -> None:
    T, H = x.shape
    E = Wr.shape[0]
    _check(_lib.moe_router(_ptr(x), _ptr(Wr), _ptr(bias), T, H, E, k, _ptr(idx), _ptr(w),
                           _ptr(ws), ws.numel(), _stream(stream)), "moe_router")


def moe_permute(idx, E, counts, offs, perm, ws, stream=None) -> None:
    T, k = idx.shape
    _check(_lib.moe_permute(_ptr(idx), T, k, E, _ptr(counts), _ptr(offs), _ptr(perm),
                            _ptr(ws), ws.numel(), _stream(stream)), "moe_permute")


def moe_ffn(x, idx, w, gate, up, down, E, I, y, ws, stream=None) -> None:
    T, H = x.shape
    k = idx.shape[1]
    _check(_lib.moe_ffn(_ptr(x), _ptr(idx), _ptr(w), _ptr(gate), _ptr(up), _ptr(down),
                        T, H, E, k, I, _ptr(y), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_ffn")


def moe_layer(x, Wr, bias, gate, up, down, k, I, idx, w, y, ws, stream=None) -> None:
    T, H = x.shape
    E = Wr.shape[0]
    _check(_lib.moe_layer(_ptr(x), _ptr(Wr), _ptr(bias), _ptr(gate), _ptr(up), _ptr(down),
                          T, H, E, k, I, _ptr(idx), _ptr(w), _ptr(y), _ptr(ws), ws.numel(),
                          _stream(stream)), "moe_layer")


def moe_layer_block(hidden, norm_w, eps, Wr, bias, gate, up, down, k, I, idx, w, out, ws,
                    add_residual=True, capture_token=-1, cap_idx=None, cap_w=None, cap_ffn=None,
                    stream=None) -> None:
    """RMSNorm (``norm_w`` None: none) -> router -> expert FFN -> residual
    add; optional capture of one token's routing and pre-residual output."""
    T, H = hidden.shape
    E = Wr.shape[0]
    _check(_lib.moe_layer_block(_ptr(hidden), _ptr(norm_w), float(eps), _ptr(Wr), _ptr(bias),
                                _ptr(gate), _ptr(up), _ptr(down), T, H, E, k, I, _ptr(idx),
                                _ptr(w), _ptr(out), 1 if add_residual else 0, int(capture_token),
                                _ptr(cap_idx), _ptr(cap_w), _ptr(cap_ffn), _ptr(ws), ws.numel(),
                                _stream(stream)), "moe_layer_block")


def moe_layer_host(x_host, Wr, bias, gate, up, down, k, I, idx, w, y_host, ws,
                   stream=None) -> None:
    """``x_host`` / ``y_host``: CPU float32 tensors (pinned for async DMA)."""
    T, H = x_host.shape
    E = Wr.shape[0]
    _check(_lib.moe_layer_host(_ptr(x_host), _ptr(Wr), _ptr(bias), _ptr(gate), _ptr(up),
                               _ptr(down), T, H, E, k, I, _ptr(idx), _ptr(w), _ptr(y_host),
                               _ptr(ws), ws.numel(), _stream(stream)), "moe_layer_host")


def moe_layer_noalloc(x, Wr, bias, gate, up, down, k, I, idx, w, y, stream=None) -> None:
    """Single-token layer without a workspace (the library's fixed scratch)."""
    T, H = x.shape
    E = Wr.shape[0]
    _check(_lib.moe_layer_noalloc(_ptr(x), _ptr(Wr), _ptr(bias), _ptr(gate), _ptr(up), _ptr(down),
                                  T, H, E, k, I, _ptr(idx), _ptr(w), _ptr(y), _stream(stream)),
           "moe_layer_noalloc")


def moe_quantize_q8k(v, q, d, sums, stream=None) -> None:
    """Q8_K blocks of the fp32 rows ``v`` [rows, n]: int8 codes ``q`` [rows, n],
    fp32 scales ``d`` [rows, n/256], int32 sub-block sums ``sums`` [rows, n/32]."""
    rows, n = v.shape
    _check(_lib.moe_quantize_q8k(_ptr(v), rows, n, _ptr(q), _ptr(d), _ptr(sums), _stream(stream)),
           "moe_quantize_q8k")


def moe_ffn_q8k(x, idx, w, gate, up, down, E, I, y, ws, stream=None) -> None:
    T, H = x.shape
    k = idx.shape[1]
    _check(_lib.moe_ffn_q8k(_ptr(x), _ptr(idx), _ptr(w), _ptr(gate), _ptr(up), _ptr(down),
                            T, H, E, k, I, _ptr(y), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_ffn_q8k")


def moe_layer_q8k(x, Wr, bias, gate, up, down, k, I, idx, w, y, ws, stream=None) -> None:
    T, H = x.shape
    E = Wr.shape[0]
    _check(_lib.moe_layer_q8k(_ptr(x), _ptr(Wr), _ptr(bias), _ptr(gate), _ptr(up), _ptr(down),
                              T, H, E, k, I, _ptr(idx), _ptr(w), _ptr(y), _ptr(ws), ws.numel(),
                              _stream(stream)), "moe_layer_q8k")


def moe_read_device_status(ws, stream=None):
    """(status code, detail) of the workspace's sticky device status; syncs the stream."""
    detail = ctypes.c_int32(0)
    code = _lib.moe_read_device_status(_ptr(ws), _stream(stream), ctypes.byref(detail))
    return int(code), int(detail.value)


def moe_debug_set_wait_limit(ns: int) -> None:
    _lib.moe_debug_set_wait_limit(int(ns))


def moe_debug_withhold_arrivals(n: int) -> None:
    _lib.moe_debug_withhold_arrivals(int(n))
