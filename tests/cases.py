"""Seeded parity cases: synthetic inputs plus the oracle's results.

Rows of x whose biased top-(k+1) logits (fp64, oracle) have an adjacent gap
below 1e-5 are redrawn from the row's next stream, so the expert selection
and its order do not hinge on rounding.
"""
from __future__ import annotations

import functools

import numpy as np

from oracle.oracle import Oracle, near_tie_free
from quantized_routed_expert_02_gb300 import synth

GAP = 1e-5


def exact_ties_only(logits_row: np.ndarray, k: int, gap: float = GAP, depth: int = 1) -> bool:
    """True when every adjacent pair among the k + depth largest logits is
    either exactly equal (a deliberate tie: identical router rows give
    identical logits on both sides) or at least ``gap`` apart."""
    top = np.sort(logits_row)[::-1][:min(k + depth, logits_row.size)]
    d = top[:-1] - top[1:]
    return bool(np.all((d == 0.0) | (d >= gap)))


def tie_free_x(o: Oracle, shape, layer, Wr, bias, max_rounds=32, accept=None):
    """x rows redrawn until ``accept(logits_row)`` holds for every row
    (default: no adjacent gap below GAP among the top k+1 logits)."""
    if accept is None:
        def accept(row):
            return near_tie_free(row, shape.k, GAP)
    x = np.stack([synth.x_row(shape, layer, t, 0) for t in range(shape.T)])
    attempt = np.zeros(shape.T, dtype=np.int32)
    for _ in range(max_rounds):
        lg = o.router(x, Wr, bias, shape.k)["logits"]
        bad = [t for t in range(shape.T) if not accept(lg[t])]
        if not bad:
            return x, attempt
        for t in bad:
            attempt[t] += 1
            x[t] = synth.x_row(shape, layer, t, int(attempt[t]))
    raise RuntimeError("could not draw tie-free activations")


@functools.lru_cache(maxsize=8)
def layer_case(shape, layer=0, sample=None):
    """Inputs and oracle outputs of one layer.  ``sample``: a tuple of token
    ids to run the oracle's FFN on (None = every token)."""
    o = Oracle()
    Wr = synth.router_weights(shape, layer)
    bias = synth.router_bias(shape)
    x, attempts = tie_free_x(o, shape, layer, Wr, bias)
    blobs = synth.expert_blobs(shape, layer)
    r = o.router(x, Wr, bias, shape.k)
    tokens = None if sample is None else np.array(sample, dtype=np.int32)
    y, skipped = o.ffn(x, r["idx"], r["w"], blobs["gate"], blobs["up"], blobs["down"],
                       shape.E, shape.I, tokens=tokens)
    return dict(shape=shape, x=x, Wr=Wr, bias=bias, blobs=blobs, idx=r["idx"], w=r["w"],
                logits=r["logits"], y=y, attempts=attempts, tokens=tokens)


def y_tolerance(y_ref: np.ndarray) -> float:
    """max|y_gpu - y_oracle| <= 2e-3 * max|y_oracle| + 1e-5."""
    finite = y_ref[np.isfinite(y_ref)]
    return 2e-3 * float(np.max(np.abs(finite))) + 1e-5


W_TOL = 1e-6
