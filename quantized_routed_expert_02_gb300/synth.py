"""Seeded synthetic inputs for the routed-expert Q4_K FFN layer.

This module draws the inputs that both the CUDA path and the CPU oracle
consume: activations ``x``, router weights ``Wr`` (and the optional logit
bias), and the per-expert gate/up/down weight blobs in the GGUF Q4_K block
format.  It holds none of the layer's arithmetic (no dequantisation, no
matvec, no softmax): the only "encoding" here is the byte placement of the
Q4_K fields, which is the input file format itself.

Q4_K block format (256 weights in 144 bytes), the format the expert tensors
of a ``Q4_K_M`` model file use (forward_qwen3_moe.rs, aprender-serve 0.35.0,
doc of ``forward_single_qwen3_moe_with_cache``, "Contract"):

* bytes 0..1    ``d``     IEEE binary16, little-endian
* bytes 2..3    ``dmin``  IEEE binary16, little-endian
* bytes 4..15   ``scales[12]``: eight 6-bit scales ``sc[j]`` and eight 6-bit
  mins ``m[j]``, one pair per 32-weight sub-block ``j``.  For ``j < 4`` the
  low six bits of ``scales[j]`` / ``scales[j+4]`` hold ``sc[j]`` / ``m[j]``;
  for ``j >= 4`` the low / high nibble of ``scales[j+4]`` hold the low four
  bits of ``sc[j]`` / ``m[j]`` and the top two bits of ``scales[j-4]`` /
  ``scales[j]`` hold their high two bits.
* bytes 16..143 ``qs[128]``: byte ``qs[32c + l]`` (c = 0..3, l = 0..31)
  holds weight ``64c + l`` in its low nibble and weight ``64c + 32 + l`` in
  its high nibble.

Weight ``i`` of sub-block ``j = i // 32`` decodes to ``d*sc[j]*q - dmin*m[j]``.

Random streams: every (layer, expert, matrix) blob and every activation row
has its own NumPy PCG64 stream keyed by a seed tuple, so any single expert or
row can be regenerated alone.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Optional

import numpy as np

QK_K = 256            # weights per Q4_K superblock
BLOCK_BYTES = 144     # bytes per Q4_K superblock

# stream tags for the seed tuples
_GATE, _UP, _DOWN, _ROUTER, _X = 0, 1, 2, 3, 4


@dataclass(frozen=True)
class LayerShape:
    """Shape of one routed-expert FFN layer and of the batch it processes."""
    name: str
    T: int            # tokens in the batch
    H: int            # hidden size
    E: int            # experts
    k: int            # experts selected per token
    I: int            # expert intermediate size
    wr_std: float     # std of the router weight entries
    zipf_bias: bool = False   # add b_e = 2*ln(1/(e+1)^0.8) to the logits
    layers: int = 1   # independently seeded layers in the timing rotation
    cfg_id: int = 0   # seed namespace

    @property
    def nsb_h(self) -> int:
        return self.H // QK_K

    @property
    def nsb_i(self) -> int:
        return self.I // QK_K

    @property
    def gate_bytes(self) -> int:
        """Bytes of one expert's gate (or up) matrix, [I rows x H]."""
        return self.I * self.nsb_h * BLOCK_BYTES

    @property
    def down_bytes(self) -> int:
        """Bytes of one expert's down matrix, [H rows x I]."""
        return self.H * self.nsb_i * BLOCK_BYTES

    @property
    def expert_bytes(self) -> int:
        return 2 * self.gate_bytes + self.down_bytes


# The five workloads: a tiny layer, a Qwen3-30B-A3B-shaped layer at decode
# (T=1), batched decode with a Zipf-skewed router (T=64) and prefill
# (T=4096), and a Qwen3-235B-A22B-shaped layer at T=1 and T=32.
SHAPES = {
    "tiny": LayerShape("tiny", 1, 256, 8, 2, 256, 0.05, cfg_id=0),
    "a3b_decode": LayerShape("a3b_decode", 1, 2048, 128, 8, 768, 0.02, layers=48, cfg_id=1),
    "a3b_batch64_zipf": LayerShape("a3b_batch64_zipf", 64, 2048, 128, 8, 768, 0.02,
                                   zipf_bias=True, layers=48, cfg_id=2),
    "a3b_prefill": LayerShape("a3b_prefill", 4096, 2048, 128, 8, 768, 0.02, layers=48, cfg_id=3),
    "a22b_decode": LayerShape("a22b_decode", 1, 4096, 128, 8, 1536, 0.015, layers=8, cfg_id=4),
    "a22b_batch32": LayerShape("a22b_batch32", 32, 4096, 128, 8, 1536, 0.015, layers=8, cfg_id=4),
}


def custom_shape(T, H, E, k, I, wr_std=0.05, zipf_bias=False, cfg_id=9, name="custom") -> LayerShape:
    return LayerShape(name, T, H, E, k, I, wr_std, zipf_bias=zipf_bias, cfg_id=cfg_id)


def layer_seed(shape: LayerShape, layer: int) -> int:
    return 1000 * shape.cfg_id + layer


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(list(key))


# ---------------------------------------------------------------------------
# Q4_K byte placement
# ---------------------------------------------------------------------------

def pack_scales(sc: np.ndarray, m: np.ndarray) -> np.ndarray:
    """Place eight 6-bit scales and eight 6-bit mins per block into 12 bytes.

    ``sc``, ``m``: integer arrays [..., 8] with values 0..63.  Returns uint8
    [..., 12] laid out as described in the module docstring.
    """
    sc = np.asarray(sc, dtype=np.uint16)
    m = np.asarray(m, dtype=np.uint16)
    out = np.empty(sc.shape[:-1] + (12,), dtype=np.uint16)
    out[..., 0:4] = (sc[..., 0:4] & 63) | ((sc[..., 4:8] >> 4) << 6)
    out[..., 4:8] = (m[..., 0:4] & 63) | ((m[..., 4:8] >> 4) << 6)
    out[..., 8:12] = (sc[..., 4:8] & 15) | ((m[..., 4:8] & 15) << 4)
    return out.astype(np.uint8)


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """Place 256 4-bit codes per block (in weight order) into 128 bytes."""
    q = np.asarray(q, dtype=np.uint8).reshape(q.shape[:-1] + (4, 2, 32))
    lo = q[..., 0, :] & 15          # weights 64c + l
    hi = q[..., 1, :] & 15          # weights 64c + 32 + l
    return (lo | (hi << 4)).reshape(q.shape[:-3] + (128,)).astype(np.uint8)


def pack_blocks(d: np.ndarray, dmin: np.ndarray, sc: np.ndarray, m: np.ndarray,
                qs: np.ndarray) -> np.ndarray:
    """Assemble [n,144] Q4_K blocks from fp16 d/dmin, scales/mins and packed qs bytes."""
    d = np.asarray(d, dtype=np.float16).reshape(-1)
    dmin = np.asarray(dmin, dtype=np.float16).reshape(-1)
    n = d.shape[0]
    out = np.empty((n, BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:2] = d.view(np.uint8).reshape(n, 2)
    out[:, 2:4] = dmin.view(np.uint8).reshape(n, 2)
    out[:, 4:16] = pack_scales(np.asarray(sc).reshape(n, 8), np.asarray(m).reshape(n, 8))
    out[:, 16:144] = np.asarray(qs, dtype=np.uint8).reshape(n, 128)
    return out


def random_blocks(rng: np.random.Generator, n: int) -> np.ndarray:
    """n random Q4_K blocks with the workload's distributions.

    Nibbles uniform 0..15 (uniform random bytes), sc uniform 1..63, m uniform
    0..63, d = fp16(|N(0,1e-3)|), dmin = fp16(|N(0,5e-4)|); fp16 rounding is
    NumPy's round-to-nearest-even.  The qs bytes come straight from the raw
    64-bit output of the generator; the 16 header bytes are then written over.
    """
    out = rng.bit_generator.random_raw(n * (BLOCK_BYTES // 8)).view(np.uint8).reshape(n, BLOCK_BYTES)
    d = np.abs(rng.normal(0.0, 1e-3, n)).astype(np.float16)
    dmin = np.abs(rng.normal(0.0, 5e-4, n)).astype(np.float16)
    sc = rng.integers(1, 64, size=(n, 8), dtype=np.uint8)
    m = rng.integers(0, 64, size=(n, 8), dtype=np.uint8)
    out[:, 0:2] = d.view(np.uint8).reshape(n, 2)
    out[:, 2:4] = dmin.view(np.uint8).reshape(n, 2)
    out[:, 4:16] = pack_scales(sc, m)
    return out


# ---------------------------------------------------------------------------
# per-layer inputs
# ---------------------------------------------------------------------------

def expert_matrix(shape: LayerShape, layer: int, expert: int, which: str) -> np.ndarray:
    """One expert's Q4_K matrix as a flat uint8 array.

    ``which`` is ``"gate"`` / ``"up"`` ([I rows x H/256 blocks]) or
    ``"down"`` ([H rows x I/256 blocks]); blocks run contiguously along the
    reduction dimension, rows follow one another.
    """
    tag = {"gate": _GATE, "up": _UP, "down": _DOWN}[which]
    rows, nsb = (shape.I, shape.nsb_h) if which != "down" else (shape.H, shape.nsb_i)
    blk = random_blocks(_rng(layer_seed(shape, layer), tag, expert), rows * nsb)
    return blk.reshape(-1)


def expert_blobs(shape: LayerShape, layer: int, experts=None) -> dict:
    """Gate/up/down blobs of a layer, expert-major: gate/up [E][I][H/256]x144 B,
    down [E][H][I/256]x144 B.  ``experts``: optional subset (others left zero)."""
    E = shape.E
    out = {}
    for which, per in (("gate", shape.gate_bytes), ("up", shape.gate_bytes),
                       ("down", shape.down_bytes)):
        buf = np.zeros(E * per, dtype=np.uint8)
        for e in (range(E) if experts is None else experts):
            buf[e * per:(e + 1) * per] = expert_matrix(shape, layer, e, which)
        out[which] = buf
    return out


def router_weights(shape: LayerShape, layer: int) -> np.ndarray:
    """Wr [E, H] fp32 ~ N(0, wr_std)."""
    r = _rng(layer_seed(shape, layer), _ROUTER)
    return r.normal(0.0, shape.wr_std, (shape.E, shape.H)).astype(np.float32)


def router_bias(shape: LayerShape) -> Optional[np.ndarray]:
    """The synthetic Zipf-like skew b_e = 2*ln(1/(e+1)^0.8), or None."""
    if not shape.zipf_bias:
        return None
    return np.array([2.0 * math.log(1.0 / (e + 1) ** 0.8) for e in range(shape.E)],
                    dtype=np.float32)


def x_row(shape: LayerShape, layer: int, row: int, attempt: int = 0) -> np.ndarray:
    return _rng(layer_seed(shape, layer), _X, row, attempt).normal(
        0.0, 1.0, shape.H).astype(np.float32)


@dataclass
class Activations:
    x: np.ndarray                        # [T, H] fp32
    attempts: np.ndarray = field(default=None)   # redraws per row


def activations(shape: LayerShape, layer: int,
                accept: Optional[Callable[[int, np.ndarray], bool]] = None,
                max_attempts: int = 64) -> Activations:
    """x [T, H] fp32 ~ N(0,1), one stream per (row, attempt).

    ``accept(row, x_row)`` may reject a row (the near-tie rule); the row is
    then redrawn from its next attempt stream while every other row stays
    as it is.
    """
    T, H = shape.T, shape.H
    x = np.empty((T, H), dtype=np.float32)
    att = np.zeros(T, dtype=np.int32)
    for t in range(T):
        a = 0
        r = x_row(shape, layer, t, a)
        while accept is not None and not accept(t, r):
            a += 1
            if a >= max_attempts:
                raise RuntimeError(f"row {t}: no acceptable draw in {max_attempts} attempts")
            r = x_row(shape, layer, t, a)
        x[t] = r
        att[t] = a
    return Activations(x, att)


def activations_fast(shape: LayerShape, layer: int) -> np.ndarray:
    """x [T, H] from one stream per layer (no per-row redraw); timing use only."""
    return _rng(layer_seed(shape, layer), _X, 1 << 30).normal(
        0.0, 1.0, (shape.T, shape.H)).astype(np.float32)
