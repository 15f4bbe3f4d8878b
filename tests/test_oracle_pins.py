"""Pins of the fp64 oracle against facts fixed outside it.

Each test checks the oracle against something it does not compute itself:
hand-built Q4_K blocks, closed forms, special cases that reduce to a dense
NumPy computation, brute force on tiny inputs, and NumPy's stable sort.
"""
import json
import math
import os

import numpy as np
import pytest

from quantized_routed_expert_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4k_blocks.json")


def _silu(z):
    # exp(-z) overflows to inf for very negative z, and z / inf is the limit 0
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


# ---------------------------------------------------------------- Q4_K decode

def _golden_blocks():
    with open(GOLDEN) as f:
        return json.load(f)["blocks"]


@pytest.mark.parametrize("blk", _golden_blocks(), ids=lambda b: b["name"])
def test_hand_built_block(oracle, blk):
    raw = np.frombuffer(bytes.fromhex(blk["hex"]), dtype=np.uint8)
    assert raw.size == 144
    got = oracle.decode_block(raw)
    if "expect_runs16" in blk:
        want = np.repeat(np.array(blk["expect_runs16"], dtype=np.float64), 16)
    else:
        want = np.tile(np.array(blk["expect_pattern64"], dtype=np.float64), 4)
    np.testing.assert_array_equal(got, want)


def test_pack_decode_round_trip(oracle):
    """Random fields -> synth's byte placement -> oracle decode recovers
    d*sc*q - dmin*m exactly for every weight (pins the packer to the decoder)."""
    rng = np.random.default_rng(7)
    n = 64
    d = rng.normal(0, 1e-2, n).astype(np.float16)
    dmin = np.abs(rng.normal(0, 1e-2, n)).astype(np.float16)
    sc = rng.integers(0, 64, (n, 8))
    m = rng.integers(0, 64, (n, 8))
    q = rng.integers(0, 16, (n, 256))
    blocks = synth.pack_blocks(d, dmin, sc, m, synth.pack_nibbles(q))
    for b in range(n):
        got = oracle.decode_block(blocks[b])
        j = np.arange(256) // 32
        want = (float(d[b]) * sc[b][j].astype(np.float64) * q[b]
                - float(dmin[b]) * m[b][j].astype(np.float64))
        np.testing.assert_array_equal(got, want)


def test_decode_rows_matches_blockwise(oracle):
    rng = np.random.default_rng(3)
    rows, ncols = 3, 512
    blob = synth.random_blocks(rng, rows * 2).reshape(-1)
    dense = oracle.decode_rows(blob, rows, ncols)
    for r in range(rows):
        for s in range(2):
            np.testing.assert_array_equal(
                dense[r, 256 * s:256 * (s + 1)],
                oracle.decode_block(blob[(r * 2 + s) * 144:(r * 2 + s + 1) * 144]))


def test_generated_fields_in_range(oracle):
    """Generated blocks have sc in 1..63 (never 0): every weight of a block
    with all codes forced to 0 must be -dmin*m, and with codes 15 the spread
    d*sc*15 must be positive."""
    rng = np.random.default_rng(11)
    blk = synth.random_blocks(rng, 32).copy()
    blk[:, 16:] = 0xFF
    for b in range(32):
        w15 = oracle.decode_block(blk[b])
        blk0 = blk[b].copy()
        blk0[16:] = 0
        w0 = oracle.decode_block(blk0)
        spread = (w15 - w0).reshape(8, 32)
        assert np.all(spread > 0)
        assert np.all(w0 <= 0)


# ---------------------------------------------------------------- router

def test_router_closed_form(oracle):
    # logits 0, ln2, ln3 -> p = 1/6, 2/6, 3/6; top-2 = [2, 1]; w = [3/5, 2/5]
    x = np.ones((1, 1), np.float32)
    Wr = np.array([[0.0], [math.log(2)], [math.log(3)]], np.float32)
    r = oracle.router(x, Wr, None, 2)
    assert r["idx"].tolist() == [[2, 1]]
    np.testing.assert_allclose(r["w"], [[0.6, 0.4]], atol=1e-7)
    np.testing.assert_allclose(r["p"], [[1 / 6, 2 / 6, 3 / 6]], atol=1e-7)


def test_router_ties_lowest_index(oracle):
    x = np.ones((1, 4), np.float32)
    Wr = np.zeros((6, 4), np.float32)
    Wr[3] = 1.0
    r = oracle.router(x, Wr, None, 3)
    # expert 3 first, then the tied zeros by lowest index
    assert r["idx"].tolist() == [[3, 0, 1]]
    e4 = math.exp(4.0)
    np.testing.assert_allclose(r["w"], [[e4 / (e4 + 2), 1 / (e4 + 2), 1 / (e4 + 2)]], rtol=1e-12)


def test_router_weights_sum_to_one_and_sorted(oracle):
    rng = np.random.default_rng(5)
    T, H, E, k = 33, 256, 16, 4
    x = rng.normal(0, 1, (T, H)).astype(np.float32)
    Wr = rng.normal(0, 0.05, (E, H)).astype(np.float32)
    r = oracle.router(x, Wr, None, k)
    np.testing.assert_allclose(r["w"].sum(1), 1.0, atol=1e-12)
    assert np.all(np.diff(r["w"], axis=1) <= 0)


def test_router_topk_matches_brute_force(oracle):
    rng = np.random.default_rng(9)
    T, H, E, k = 40, 512, 32, 6
    x = rng.normal(0, 1, (T, H)).astype(np.float32)
    Wr = rng.normal(0, 0.05, (E, H)).astype(np.float32)
    b = rng.normal(0, 0.5, E).astype(np.float32)
    r = oracle.router(x, Wr, b, k)
    logits = x.astype(np.float64) @ Wr.astype(np.float64).T + b.astype(np.float64)
    np.testing.assert_allclose(r["logits"], logits, rtol=1e-12, atol=1e-12)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t]))   # value desc, index asc
        assert r["idx"][t].tolist() == order[:k].tolist()
        p = np.exp(logits[t] - logits[t].max())
        p /= p.sum()
        sel = p[order[:k]]
        np.testing.assert_allclose(r["w"][t], sel / sel.sum(), rtol=1e-12)


def test_router_k_equals_E_is_dense_softmax(oracle):
    rng = np.random.default_rng(12)
    x = rng.normal(0, 1, (5, 256)).astype(np.float32)
    Wr = rng.normal(0, 0.1, (8, 256)).astype(np.float32)
    r = oracle.router(x, Wr, None, 8)
    logits = x.astype(np.float64) @ Wr.astype(np.float64).T
    sm = np.exp(logits - logits.max(1, keepdims=True))
    sm /= sm.sum(1, keepdims=True)
    for t in range(5):
        np.testing.assert_allclose(r["w"][t], sm[t][r["idx"][t]], rtol=1e-12)
        assert sorted(r["idx"][t].tolist()) == list(range(8))


# ---------------------------------------------------------------- FFN

def _tiny_layer(H=256, I=256, E=8, seed=21):
    shape = synth.custom_shape(1, H, E, 2, I, cfg_id=90 + seed % 7)
    blobs = synth.expert_blobs(shape, 0)
    return shape, blobs


def _dense(oracle, shape, blobs, e):
    H, I = shape.H, shape.I
    g = oracle.decode_rows(blobs["gate"][e * shape.gate_bytes:(e + 1) * shape.gate_bytes], I, H)
    u = oracle.decode_rows(blobs["up"][e * shape.gate_bytes:(e + 1) * shape.gate_bytes], I, H)
    d = oracle.decode_rows(blobs["down"][e * shape.down_bytes:(e + 1) * shape.down_bytes], H, I)
    return g, u, d


def _dense_ffn(gud, xv):
    g, u, d = gud
    return d @ (_silu(g @ xv) * (u @ xv))


def test_ffn_brute_force_tiny(oracle):
    shape, blobs = _tiny_layer()
    rng = np.random.default_rng(1)
    T, k = 3, 2
    x = rng.normal(0, 1, (T, shape.H)).astype(np.float32)
    idx = np.array([[1, 6], [3, 3], [7, 0]], np.int32)
    w = np.array([[0.7, 0.3], [0.25, 0.75], [0.5, 0.5]])
    y, skipped = oracle.ffn(x, idx, w, blobs["gate"], blobs["up"], blobs["down"], shape.E, shape.I)
    assert skipped == 0
    dense = {e: _dense(oracle, shape, blobs, e) for e in set(idx.ravel().tolist())}
    for t in range(T):
        want = sum(w[t, j] * _dense_ffn(dense[idx[t, j]], x[t].astype(np.float64)) for j in range(k))
        np.testing.assert_allclose(y[t], want, rtol=1e-10, atol=1e-12 * np.abs(want).max())


def test_ffn_k_equals_E_is_dense_mixture(oracle):
    shape, blobs = _tiny_layer(E=4, seed=2)
    rng = np.random.default_rng(2)
    x = rng.normal(0, 1, (2, shape.H)).astype(np.float32)
    Wr = rng.normal(0, 0.05, (4, shape.H)).astype(np.float32)
    r = oracle.layer(x, Wr, None, 4, blobs["gate"], blobs["up"], blobs["down"], 4, shape.I)
    logits = x.astype(np.float64) @ Wr.astype(np.float64).T
    for t in range(2):
        p = np.exp(logits[t] - logits[t].max())
        p /= p.sum()
        want = sum(p[e] * _dense_ffn(_dense(oracle, shape, blobs, e), x[t].astype(np.float64))
                   for e in range(4))
        np.testing.assert_allclose(r["y"][t], want, rtol=1e-10, atol=1e-12 * np.abs(want).max())


def test_ffn_k1_is_single_expert(oracle):
    shape, blobs = _tiny_layer(seed=3)
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, (2, shape.H)).astype(np.float32)
    Wr = rng.normal(0, 0.05, (shape.E, shape.H)).astype(np.float32)
    r = oracle.layer(x, Wr, None, 1, blobs["gate"], blobs["up"], blobs["down"], shape.E, shape.I)
    assert np.all(r["w"] == 1.0)
    logits = x.astype(np.float64) @ Wr.astype(np.float64).T
    for t in range(2):
        e = int(np.argmax(logits[t]))
        assert r["idx"][t, 0] == e
        want = _dense_ffn(_dense(oracle, shape, blobs, e), x[t].astype(np.float64))
        np.testing.assert_allclose(r["y"][t], want, rtol=1e-10, atol=1e-12 * np.abs(want).max())


def test_ffn_one_hot_router(oracle):
    """A logit gap of 1000 makes every other probability underflow to 0, so
    k=2 reduces to one dense SwiGLU FFN of the favoured expert."""
    shape, blobs = _tiny_layer(seed=4)
    rng = np.random.default_rng(4)
    x = rng.normal(0, 1, (1, shape.H)).astype(np.float32)
    Wr = rng.normal(0, 0.05, (shape.E, shape.H)).astype(np.float32)
    bias = np.zeros(shape.E, np.float32)
    bias[5] = 1000.0
    r = oracle.layer(x, Wr, bias, 2, blobs["gate"], blobs["up"], blobs["down"], shape.E, shape.I)
    assert r["idx"][0, 0] == 5
    assert r["w"][0, 0] == 1.0 and r["w"][0, 1] == 0.0
    want = _dense_ffn(_dense(oracle, shape, blobs, 5), x[0].astype(np.float64))
    np.testing.assert_allclose(r["y"][0], want, rtol=1e-10, atol=1e-12 * np.abs(want).max())


def test_ffn_out_of_range_slot_contributes_nothing(oracle):
    shape, blobs = _tiny_layer(seed=5)
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, (1, shape.H)).astype(np.float32)
    idx = np.array([[2, 99]], np.int32)
    y, skipped = oracle.ffn(x, idx, np.array([[0.5, 0.5]]), blobs["gate"], blobs["up"],
                            blobs["down"], shape.E, shape.I)
    assert skipped == 1
    want = 0.5 * _dense_ffn(_dense(oracle, shape, blobs, 2), x[0].astype(np.float64))
    np.testing.assert_allclose(y[0], want, rtol=1e-10, atol=1e-12 * np.abs(want).max())


def test_ffn_token_subset_matches_full(oracle):
    shape, blobs = _tiny_layer(seed=6)
    rng = np.random.default_rng(6)
    x = rng.normal(0, 1, (5, shape.H)).astype(np.float32)
    idx = rng.integers(0, shape.E, (5, 2)).astype(np.int32)
    w = rng.random((5, 2))
    full, _ = oracle.ffn(x, idx, w, blobs["gate"], blobs["up"], blobs["down"], shape.E, shape.I)
    part, _ = oracle.ffn(x, idx, w, blobs["gate"], blobs["up"], blobs["down"], shape.E, shape.I,
                         tokens=np.array([4, 1]))
    np.testing.assert_array_equal(part[[4, 1]], full[[4, 1]])
    assert np.isnan(part[0]).all()


def test_silu_closed_form(oracle):
    """One weight row per matrix: with H = I = 256 and an expert whose gate,
    up and down rows are known, h = SiLU(g)*u and y = w * down . h."""
    H = I = 256
    # every gate/up weight = 1/128 (d=2^-7, sc=1, q=1, dmin=0); down weight = 2 (d=2, sc=1, q=1)
    def block(d_bits):
        b = np.zeros(144, np.uint8)
        b[0], b[1] = d_bits & 0xFF, d_bits >> 8
        b[4:8] = 1
        b[12:16] = 1
        b[16:] = 0x11
        return b
    g_blk = block(0x2000)   # 2^-7
    d_blk = block(0x4000)   # 2.0
    gate = np.tile(g_blk, I)
    down = np.tile(d_blk, H)
    xv = np.full(H, 0.5, np.float32)
    h, o = oracle.expert(xv, gate, gate, down, H, I)
    g = 256 * 0.5 / 128.0     # = 1.0
    want_h = g / (1 + math.exp(-g)) * g
    np.testing.assert_allclose(h, want_h, rtol=1e-15)
    np.testing.assert_allclose(o, 2.0 * 256 * want_h, rtol=1e-14)


# ---------------------------------------------------------------- permutation

def test_permutation_invariants(oracle):
    rng = np.random.default_rng(8)
    T, k, E = 300, 4, 16
    idx = rng.integers(0, E, (T, k)).astype(np.int32)
    counts, offs, perm = oracle.permutation(idx, E)
    flat = idx.ravel()
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    assert offs[0] == 0 and np.all(np.diff(offs) == counts) and offs[-1] == T * k
    np.testing.assert_array_equal(perm, np.argsort(flat, kind="stable"))
    assert sorted(perm.tolist()) == list(range(T * k))


def test_permutation_skips_out_of_range(oracle):
    idx = np.array([[0, 5], [9, 0], [-1, 2]], np.int32)
    counts, offs, perm = oracle.permutation(idx, 6)
    assert counts.tolist() == [2, 0, 1, 0, 0, 1]
    assert perm.tolist() == [0, 3, 5, 1]


@pytest.mark.parametrize("H,I", [(512, 256), (256, 512)])
def test_ffn_brute_force_rectangular(oracle, H, I):
    shape = synth.custom_shape(1, H, 4, 2, I, cfg_id=97)
    blobs = synth.expert_blobs(shape, 0)
    rng = np.random.default_rng(H + I)
    x = rng.normal(0, 1, (2, H)).astype(np.float32)
    idx = np.array([[3, 1], [0, 2]], np.int32)
    w = np.array([[0.9, 0.1], [0.4, 0.6]])
    y, _ = oracle.ffn(x, idx, w, blobs["gate"], blobs["up"], blobs["down"], 4, I)
    for t in range(2):
        want = sum(w[t, j] * _dense_ffn(_dense(oracle, shape, blobs, idx[t, j]),
                                        x[t].astype(np.float64)) for j in range(2))
        np.testing.assert_allclose(y[t], want, rtol=1e-10, atol=1e-12 * np.abs(want).max())


# ---------------------------------------------------------------- pre-FFN RMSNorm and residual
# forward_qwen3_moe.rs (aprender-serve 0.35.0), steps 2f-2h of
# forward_qwen3_moe: ffn_input = rms_norm(hidden, ffn_norm_weight, eps), the
# MoE FFN on it, hidden += ffn_output.

def test_rmsnorm_constant_row(oracle):
    """A constant row c has root-mean-square |c|: with eps = 0 the norm is
    sign(c) * gamma exactly; with eps > 0 it is c / sqrt(c^2 + eps) * gamma."""
    H = 256
    gamma = np.linspace(-2.0, 3.0, H).astype(np.float32)
    for c in (0.75, -3.0, 1024.0):
        x = np.full((1, H), c, dtype=np.float32)
        np.testing.assert_array_equal(oracle.rmsnorm(x, gamma, 0.0)[0],
                                      (np.sign(c) * gamma).astype(np.float32))
        eps = 0.5
        want = (c / math.sqrt(c * c + eps)) * gamma.astype(np.float64)
        got = oracle.rmsnorm(x, gamma, eps)[0].astype(np.float64)
        assert np.max(np.abs(got - want)) <= 1e-6 * np.max(np.abs(want))


def test_rmsnorm_hand_example(oracle):
    """x = (1, 2, 3, 4): mean of squares 30/4 = 7.5, 1/sqrt(7.5) =
    0.36514837167011..., gamma = (1, 0.5, 2, -1)."""
    x = np.array([[1.0, 2.0, 3.0, 4.0]], dtype=np.float32)
    gamma = np.array([1.0, 0.5, 2.0, -1.0], dtype=np.float32)
    want = np.array([0.3651483716701107, 0.3651483716701107, 2.1908902300206643,
                     -1.4605934866804429])
    got = oracle.rmsnorm(x, gamma, 0.0)[0].astype(np.float64)
    assert np.max(np.abs(got - want)) <= 1e-7


def test_rmsnorm_scale_invariance_and_unit_rms(oracle):
    """With eps = 0 the norm ignores a positive scale of its row (bitwise
    for a power of two) and, with gamma = 1, has root-mean-square 1."""
    rng = np.random.default_rng(11)
    x = rng.normal(0.0, 1.0, (3, 512)).astype(np.float32)
    ones = np.ones(512, dtype=np.float32)
    a = oracle.rmsnorm(x, ones, 0.0)
    np.testing.assert_array_equal(oracle.rmsnorm(4.0 * x, ones, 0.0), a)
    assert np.max(np.abs(oracle.rmsnorm(3.0 * x, ones, 0.0) - a)) <= 1e-6
    rms = np.sqrt(np.mean(a.astype(np.float64) ** 2, axis=1))
    assert np.max(np.abs(rms - 1.0)) <= 1e-6


def _block_inputs(T=3, H=256, E=8, k=2, I=256, cfg=93):
    shape = synth.custom_shape(T, H, E, k, I, wr_std=0.05, cfg_id=cfg)
    blobs = synth.expert_blobs(shape, 0)
    Wr = synth.router_weights(shape, 0)
    hidden = (3.0 * synth.activations_fast(shape, 0)).astype(np.float32)
    return shape, blobs, Wr, hidden


def test_block_zero_norm_weight_returns_hidden(oracle):
    """gamma = 0 makes the FFN input zero: every logit is 0, so the top k
    are experts 0..k-1 (lowest indices) with weight 1/k, every expert maps 0
    to 0, and the block's output is the residual stream itself."""
    shape, blobs, Wr, hidden = _block_inputs()
    r = oracle.block(hidden, np.zeros(shape.H, np.float32), 1e-6, Wr, None, shape.k,
                     blobs["gate"], blobs["up"], blobs["down"], shape.E, shape.I)
    np.testing.assert_array_equal(r["idx"], np.tile(np.arange(shape.k), (shape.T, 1)))
    np.testing.assert_array_equal(r["y"], 0.0)
    np.testing.assert_array_equal(r["out"], hidden.astype(np.float64))


def test_block_output_is_hidden_plus_ffn_of_normed(oracle):
    """With eps = 0, scaling the residual stream by 4 leaves the normed FFN
    input, the routing and the FFN output bit-identical; the output is
    hidden + y (so the two outputs differ by exactly 3 * hidden)."""
    shape, blobs, Wr, hidden = _block_inputs()
    gamma = np.linspace(0.5, 1.5, shape.H).astype(np.float32)
    args = (Wr, None, shape.k, blobs["gate"], blobs["up"], blobs["down"], shape.E, shape.I)
    r1 = oracle.block(hidden, gamma, 0.0, *args)
    r4 = oracle.block(4.0 * hidden, gamma, 0.0, *args)
    np.testing.assert_array_equal(r1["ffn_in"], r4["ffn_in"])
    np.testing.assert_array_equal(r1["idx"], r4["idx"])
    np.testing.assert_array_equal(r1["y"], r4["y"])
    assert np.max(np.abs(r1["y"])) > 1.0
    h64 = hidden.astype(np.float64)
    assert np.max(np.abs(r1["out"] - (h64 + r1["y"]))) == 0.0
    assert np.max(np.abs((r4["out"] - r1["out"]) - 3.0 * h64)) <= 1e-9 * np.max(np.abs(r1["out"]))
    # without the norm the FFN sees the residual stream itself
    r0 = oracle.block(hidden, None, 0.0, *args)
    np.testing.assert_array_equal(r0["ffn_in"], hidden)
    ref = oracle.layer(hidden, *args)
    np.testing.assert_array_equal(r0["y"], ref["y"])


# ---------------------------------------------------------------- Q8_K activations
#
# The Q8_K-activation variant (qwen3_moe_dispatch.rs, aprender-serve 0.70.2,
# doc of cpu_reference: the production CPU path's activations are Q8_K).
# Reading pinned here: per 256-element block, d = amax / 127 and codes
# q = round-half-even(v * (127 / amax)) in fp32, with sub-block code sums.

def test_q8k_hand_block(oracle):
    """v_i = i - 128: amax = 128, the scale 127/128 = 0.9921875 is exact and
    so is every product (i - 128) * 0.9921875, so the codes are the rounded
    exact values: -128 -> -127, -65 -> -64.49 -> -64, -64 -> -63.5 -> -64
    (half to even), 63 -> 62.51 -> 63, 64 -> 63.5 -> 64 (half to even),
    127 -> 126.01 -> 126."""
    v = (np.arange(256) - 128).astype(np.float32)
    q, d, sums = oracle.q8k_quantize(v)
    assert d[0, 0] == np.float32(128.0) / np.float32(127.0)
    hand = {0: -127, 63: -64, 64: -64, 65: -63, 128: 0, 191: 63, 192: 64, 255: 126}
    for i, want in hand.items():
        assert q[0, i] == want, (i, q[0, i], want)
    # every code: the exact product rounded half to even (Python's round on a Fraction)
    from fractions import Fraction
    exact = [round(Fraction(i - 128) * Fraction(127, 128)) for i in range(256)]
    np.testing.assert_array_equal(q[0].astype(int), exact)
    np.testing.assert_array_equal(sums[0], [sum(exact[32 * j:32 * j + 32]) for j in range(8)])


def test_q8k_zero_and_single_value_blocks(oracle):
    v = np.zeros((2, 256), np.float32)
    v[1, 7] = -3.0
    q, d, sums = oracle.q8k_quantize(v)
    assert d[0, 0] == 0.0 and not q[0].any() and not sums[0].any()
    assert d[1, 0] == np.float32(3.0) / np.float32(127.0)
    assert q[1, 7] == -127 and np.count_nonzero(q[1]) == 1
    assert sums[1, 0] == -127 and not sums[1, 1:].any()


def test_q8k_reconstruction_bound(oracle):
    """Every code reconstructs its value to within half a step, the block's
    largest magnitude lands on +-127, and the sums are the sub-block sums."""
    rng = np.random.default_rng(31)
    v = rng.normal(0, 1, (6, 512)).astype(np.float32)
    v[1] *= 1e-3
    v[2, :256] *= 1e4
    v[3, 256:] = 0.0
    q, d, sums = oracle.q8k_quantize(v)
    for r in range(6):
        for b in range(2):
            vb = v[r, 256 * b:256 * b + 256].astype(np.float64)
            qb = q[r, 256 * b:256 * b + 256].astype(np.float64)
            db = float(d[r, b])
            if not np.any(vb):
                assert db == 0.0 and not np.any(qb)
                continue
            assert np.max(np.abs(qb * db - vb)) <= 0.5 * db * (1 + 1e-5)
            assert np.max(np.abs(qb)) == 127
    np.testing.assert_array_equal(sums, q.astype(np.int32).reshape(6, -1, 32).sum(axis=2))


def test_q8k_row_dot_is_dense_dot_of_dequantised(oracle):
    """The integer form (P, S sums with the block scales) equals the fp64 dot
    of the dequantised Q4_K row with the dequantised vector d * q."""
    rng = np.random.default_rng(32)
    row = synth.random_blocks(rng, 3)
    v = rng.normal(0, 1, 768).astype(np.float32)
    q, d, sums = oracle.q8k_quantize(v)
    dense_row = oracle.decode_rows(row, 1, 768)[0]
    vdq = q[0].astype(np.float64) * np.repeat(d[0].astype(np.float64), 256)
    want = float(dense_row @ vdq)
    got = oracle.row_dot_q8k(row, 768, q[0], d[0], sums[0])
    assert abs(got - want) <= 1e-12 * max(1.0, float(np.abs(dense_row).sum() * np.abs(vdq).max()))


def test_q8k_ffn_is_dense_composition(oracle):
    """The Q8_K FFN against dense NumPy matrices: x quantised (the pinned
    quantiser), g and u dense products with the dequantised x, h = SiLU(g) u
    rounded to fp32 and quantised, o = W_down times the dequantised h,
    y = sum_j w_j o_j."""
    shape, blobs = _tiny_layer(E=4, seed=6)
    rng = np.random.default_rng(33)
    T = 3
    x = rng.normal(0, 1, (T, shape.H)).astype(np.float32)
    idx = np.array([[1, 3], [2, 2], [0, 1]], np.int32)
    w = np.array([[0.6, 0.4], [0.5, 0.5], [0.9, 0.1]])
    y, skipped = oracle.ffn_q8k(x, idx, w, blobs["gate"], blobs["up"], blobs["down"], shape.E,
                                shape.I)
    assert skipped == 0

    def deq(v):
        q, d, _ = oracle.q8k_quantize(v)
        return q[0].astype(np.float64) * np.repeat(d[0].astype(np.float64), 256)

    dense = {e: _dense(oracle, shape, blobs, e) for e in range(4)}
    for t in range(T):
        xv = deq(x[t])
        want = np.zeros(shape.H)
        for j in range(2):
            g, u, dn = dense[idx[t, j]]
            h = (_silu(g @ xv) * (u @ xv)).astype(np.float32)
            want += w[t, j] * (dn @ deq(h))
        np.testing.assert_allclose(y[t], want, rtol=1e-9, atol=1e-12 * np.abs(want).max())


def test_q8k_ffn_close_to_fp32_ffn(oracle):
    """Eight-bit activations cost little accuracy on one layer: the output's
    cosine with the fp32-activation FFN stays above 0.99 on every token (the
    pages measure 0.985 for a whole model's logits, after every layer)."""
    shape, blobs = _tiny_layer(E=8, seed=7)
    rng = np.random.default_rng(34)
    x = rng.normal(0, 1, (4, shape.H)).astype(np.float32)
    idx = np.array([[0, 5], [1, 2], [7, 3], [4, 6]], np.int32)
    w = np.full((4, 2), 0.5)
    args = (blobs["gate"], blobs["up"], blobs["down"], shape.E, shape.I)
    yq, _ = oracle.ffn_q8k(x, idx, w, *args)
    yf, _ = oracle.ffn(x, idx, w, *args)
    for t in range(4):
        cos = float(yq[t] @ yf[t] / (np.linalg.norm(yq[t]) * np.linalg.norm(yf[t])))
        assert 0.99 < cos < 1.0
