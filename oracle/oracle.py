"""ctypes front of the fp64 CPU oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the benchmark's
CPU-baseline leg use it.  The product path (the CUDA library and its Python
binding) never imports this module.

``build()`` compiles the C file with gcc (no fast-math, no FMA contraction,
OpenMP on).  Every function here only marshals NumPy arrays to the C entry
points; the arithmetic is all in ``moe_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _SO) -> str:
    """Compile the oracle into a shared library (skipped when up to date)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(path: str = _SO):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i, l = ctypes.c_int, ctypes.c_long
    lib.moq_decode_block.argtypes = [P, P]
    lib.moq_decode_rows.argtypes = [P, l, i, P]
    lib.moq_router.argtypes = [P, P, P, i, i, i, i, P, P, P, P]
    lib.moq_expert.argtypes = [P, P, P, P, i, i, P, P]
    lib.moq_ffn.argtypes = [P, P, P, P, P, P, i, i, i, i, i, P, i, P]
    lib.moq_ffn.restype = l
    lib.moq_permutation.argtypes = [P, i, i, i, P, P, P]
    lib.moq_rmsnorm.argtypes = [P, P, ctypes.c_double, i, i, P]
    lib.moq_add_residual.argtypes = [P, P, l, P]
    lib.moq_q8k_quantize.argtypes = [P, l, P, P, P]
    lib.moq_row_dot_q8k.argtypes = [P, i, P, P, P]
    lib.moq_row_dot_q8k.restype = ctypes.c_double
    lib.moq_ffn_q8k.argtypes = [P, P, P, P, P, P, i, i, i, i, i, P, i, P]
    lib.moq_ffn_q8k.restype = l
    lib.moq_set_threads.argtypes = [i]
    lib.moq_max_threads.restype = i
    return lib


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(build())
        return _lib


def load_variant(path: str):
    """Load another build of the oracle source (used by the mutation tests)."""
    return _load(path)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """Thin wrapper over one loaded oracle library."""

    def __init__(self, handle=None):
        self.L = handle if handle is not None else lib()

    def set_threads(self, n: int):
        self.L.moq_set_threads(int(n))

    def max_threads(self) -> int:
        return int(self.L.moq_max_threads())

    def decode_block(self, blk: np.ndarray) -> np.ndarray:
        blk = _c(blk, np.uint8).reshape(-1)
        assert blk.size == 144
        out = np.empty(256, dtype=np.float64)
        self.L.moq_decode_block(_p(blk), _p(out))
        return out

    def decode_rows(self, blob: np.ndarray, nrows: int, ncols: int) -> np.ndarray:
        blob = _c(blob, np.uint8).reshape(-1)
        assert blob.size == nrows * (ncols // 256) * 144
        out = np.empty((nrows, ncols), dtype=np.float64)
        self.L.moq_decode_rows(_p(blob), nrows, ncols, _p(out))
        return out

    def router(self, x, Wr, bias, k):
        x = _c(x, np.float32)
        Wr = _c(Wr, np.float32)
        T, H = x.shape
        E = Wr.shape[0]
        b = None if bias is None else _c(bias, np.float32)
        logits = np.empty((T, E), dtype=np.float64)
        p = np.empty((T, E), dtype=np.float64)
        idx = np.empty((T, k), dtype=np.int32)
        w = np.empty((T, k), dtype=np.float64)
        self.L.moq_router(_p(x), _p(Wr), None if b is None else _p(b), T, H, E, k,
                          _p(logits), _p(p), _p(idx), _p(w))
        return dict(logits=logits, p=p, idx=idx, w=w)

    def expert(self, xv, gate_e, up_e, down_e, H, I):
        xv = _c(xv, np.float64)
        h = np.empty(I, dtype=np.float64)
        o = np.empty(H, dtype=np.float64)
        self.L.moq_expert(_p(xv), _p(_c(gate_e, np.uint8)), _p(_c(up_e, np.uint8)),
                          _p(_c(down_e, np.uint8)), H, I, _p(h), _p(o))
        return h, o

    def ffn(self, x, idx, w, gate, up, down, E, I, tokens=None):
        """y [T,H] fp64 (rows not in ``tokens`` are left NaN) and the skip count."""
        x = _c(x, np.float32)
        T, H = x.shape
        idx = _c(idx, np.int32)
        k = idx.shape[1]
        w = _c(w, np.float64)
        y = np.full((T, H), np.nan, dtype=np.float64)
        tok = None if tokens is None else _c(tokens, np.int32)
        skipped = self.L.moq_ffn(_p(x), _p(idx), _p(w), _p(_c(gate, np.uint8)),
                                 _p(_c(up, np.uint8)), _p(_c(down, np.uint8)),
                                 T, H, E, k, I, None if tok is None else _p(tok),
                                 0 if tok is None else tok.size, _p(y))
        return y, int(skipped)

    def permutation(self, idx, E):
        idx = _c(idx, np.int32)
        T, k = idx.shape
        counts = np.empty(E, dtype=np.int32)
        offs = np.empty(E + 1, dtype=np.int32)
        perm = np.full(T * k, -1, dtype=np.int32)
        self.L.moq_permutation(_p(idx), T, k, E, _p(counts), _p(offs), _p(perm))
        return counts, offs, perm[:offs[E]]

    def layer(self, x, Wr, bias, k, gate, up, down, E, I, tokens=None):
        r = self.router(x, Wr, bias, k)
        y, skipped = self.ffn(x, r["idx"], r["w"], gate, up, down, E, I, tokens)
        r["y"] = y
        return r

    # ---- Q8_K activations (the integer-dot variant of the layer)

    def q8k_quantize(self, v):
        """Q8_K blocks of fp32 rows v [rows, n] (n a multiple of 256): codes
        int8 [rows, n], scales fp32 [rows, n/256], sub-block code sums int32
        [rows, n/32]."""
        v = _c(v, np.float32)
        if v.ndim == 1:
            v = v.reshape(1, -1)
        rows, n = v.shape
        assert n % 256 == 0
        q = np.empty((rows, n), dtype=np.int8)
        d = np.empty((rows, n // 256), dtype=np.float32)
        sums = np.empty((rows, n // 32), dtype=np.int32)
        self.L.moq_q8k_quantize(_p(v), rows * (n // 256), _p(q), _p(d), _p(sums))
        return q, d, sums

    def row_dot_q8k(self, row, ncols, q, d, sums):
        """fp64 dot of one Q4_K row (bytes) with one Q8_K vector."""
        return float(self.L.moq_row_dot_q8k(_p(_c(row, np.uint8)), ncols // 256,
                                            _p(_c(q, np.int8)), _p(_c(d, np.float32)),
                                            _p(_c(sums, np.int32))))

    def ffn_q8k(self, x, idx, w, gate, up, down, E, I, tokens=None):
        """y [T,H] fp64 with Q8_K activations (rows not in ``tokens`` NaN)
        and the skip count."""
        x = _c(x, np.float32)
        T, H = x.shape
        idx = _c(idx, np.int32)
        k = idx.shape[1]
        w = _c(w, np.float64)
        y = np.full((T, H), np.nan, dtype=np.float64)
        tok = None if tokens is None else _c(tokens, np.int32)
        skipped = self.L.moq_ffn_q8k(_p(x), _p(idx), _p(w), _p(_c(gate, np.uint8)),
                                     _p(_c(up, np.uint8)), _p(_c(down, np.uint8)),
                                     T, H, E, k, I, None if tok is None else _p(tok),
                                     0 if tok is None else tok.size, _p(y))
        return y, int(skipped)

    def layer_q8k(self, x, Wr, bias, k, gate, up, down, E, I, tokens=None):
        """The fp32 router, then the FFN with Q8_K activations."""
        r = self.router(x, Wr, bias, k)
        y, skipped = self.ffn_q8k(x, r["idx"], r["w"], gate, up, down, E, I, tokens)
        r["y"] = y
        return r

    def rmsnorm(self, x, gamma, eps):
        """fp32 [T,H]: x / sqrt(mean(x^2) + eps) * gamma per row (fp64 inside)."""
        x = _c(x, np.float32)
        T, H = x.shape
        g = _c(gamma, np.float32).reshape(-1)
        assert g.size == H
        out = np.empty((T, H), dtype=np.float32)
        self.L.moq_rmsnorm(_p(x), _p(g), float(eps), T, H, _p(out))
        return out

    def add_residual(self, hidden, y):
        hidden = _c(hidden, np.float32)
        y = _c(y, np.float64)
        assert hidden.shape == y.shape
        out = np.empty(y.shape, dtype=np.float64)
        self.L.moq_add_residual(_p(hidden), _p(y), y.size, _p(out))
        return out

    def block(self, hidden, norm_w, eps, Wr, bias, k, gate, up, down, E, I, residual=True,
              tokens=None):
        """The layer with the steps on each side of it: ffn_in = RMSNorm(hidden)
        (skipped when ``norm_w`` is None), the router and FFN on ffn_in, and
        out = hidden + y (``residual``) or y.  Returns the layer's dict plus
        ``ffn_in`` and ``out``."""
        ffn_in = _c(hidden, np.float32) if norm_w is None else self.rmsnorm(hidden, norm_w, eps)
        r = self.layer(ffn_in, Wr, bias, k, gate, up, down, E, I, tokens)
        r["ffn_in"] = ffn_in
        r["out"] = self.add_residual(hidden, r["y"]) if residual else r["y"].copy()
        return r


def near_tie_free(logits_row: np.ndarray, k: int, gap: float = 1e-5) -> bool:
    """True when the k+1 largest biased logits are pairwise >= ``gap`` apart
    (adjacent in sorted order), so the selection and its order do not hinge
    on rounding."""
    n = min(k + 1, logits_row.size)
    top = np.sort(logits_row)[::-1][:n]
    return bool(np.all(top[:-1] - top[1:] >= gap))
