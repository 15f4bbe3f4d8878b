"""The Q8_K-activation variant of the layer against the oracle, through the
C ABI.

qwen3_moe_dispatch.rs (aprender-serve 0.70.2), doc of cpu_reference: the
production CPU path runs the layer on Q8_K activations.  Here every
activation vector that meets a Q4_K matrix (x before gate/up, h before
down) is quantised per 256 values to int8 codes with one fp32 scale and the
products are integer dots.

Bars:
- quantisation (moe_quantize_q8k): codes, scales and sub-block sums
  bit-exact (both sides take every step in fp32);
- the layer (moe_layer_q8k / moe_ffn_q8k): expert indices bit-exact,
  |w - w_oracle| <= 1e-6, y within 2e-3 * max|y_oracle| + 1e-5.  The codes of
  h are decided in fp32 on each side from that side's own h, so a code can
  differ by one where h * 127 / amax lies within rounding of a half; one
  such code moves y by at most d8 * max|W_down|, far inside the tolerance.
"""
import numpy as np
import pytest

from oracle.oracle import Oracle
from quantized_routed_expert_02_gb300 import synth
from tests.cases import W_TOL, tie_free_x, y_tolerance
from tests.test_gpu_parity import DEV, m  # noqa: F401

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def quantize_gpu(m, v):
    rows, n = v.shape
    vd = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(DEV)
    q = torch.empty(rows, n, dtype=torch.int8, device=DEV)
    d = torch.empty(rows, n // 256, dtype=torch.float32, device=DEV)
    s = torch.empty(rows, n // 32, dtype=torch.int32, device=DEV)
    m.moe_quantize_q8k(vd, q, d, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), d.cpu().numpy(), s.cpu().numpy()


def test_quantize_bit_exact(m, oracle):
    rng = np.random.default_rng(41)
    v = rng.normal(0, 1, (9, 1024)).astype(np.float32)
    v[1] *= 1e-4                                   # small magnitudes
    v[2] *= 3e4                                    # large magnitudes
    v[3, :256] = 0.0                               # an all-zero block
    v[4, :] = 0.0
    v[4, 300] = -7.25                              # one value in its block
    v[5, :256] = np.arange(256) - 128              # exact half-integer products
    v[6] = np.round(v[6] * 64) / 64                # coarse grid: many ties of magnitude
    v[7, 512:768] = np.linspace(-1, 1, 256)
    v[8] = rng.standard_cauchy(1024).astype(np.float32)  # heavy tails
    qg, dg, sg = quantize_gpu(m, v)
    qo, do, so = oracle.q8k_quantize(v)
    np.testing.assert_array_equal(qg, qo)
    np.testing.assert_array_equal(dg, do)
    np.testing.assert_array_equal(sg, so)


def test_quantize_many_rows(m, oracle):
    rng = np.random.default_rng(42)
    v = (rng.normal(0, 1, (300, 768)) * rng.uniform(0.01, 100, (300, 1))).astype(np.float32)
    qg, dg, sg = quantize_gpu(m, v)
    qo, do, so = oracle.q8k_quantize(v)
    np.testing.assert_array_equal(qg, qo)
    np.testing.assert_array_equal(dg, do)
    np.testing.assert_array_equal(sg, so)


def test_quantize_rejects_bad_shapes(m):
    v = torch.zeros(2, 300, device=DEV)
    q = torch.zeros(2, 300, dtype=torch.int8, device=DEV)
    with pytest.raises(m.MoeError):
        m.moe_quantize_q8k(v, q, torch.zeros(2, 2, device=DEV),
                           torch.zeros(2, 10, dtype=torch.int32, device=DEV))


def q8k_case(shape, layer=0, experts_only=False, tokens=None):
    o = Oracle()
    Wr = synth.router_weights(shape, layer)
    bias = synth.router_bias(shape)
    x, _ = tie_free_x(o, shape, layer, Wr, bias)
    r0 = o.router(x, Wr, bias, shape.k)
    experts = sorted(set(r0["idx"].ravel().tolist())) if experts_only else None
    blobs = synth.expert_blobs(shape, layer, experts=experts)
    r = o.layer_q8k(x, Wr, bias, shape.k, blobs["gate"], blobs["up"], blobs["down"], shape.E,
                    shape.I, tokens=tokens)
    return dict(shape=shape, x=x, Wr=Wr, bias=bias, blobs=blobs, r=r, tokens=tokens)


def run_q8k(m, case):
    s = case["shape"]
    dev = lambda a: None if a is None else torch.from_numpy(a).to(DEV)  # noqa: E731
    b = case["blobs"]
    idx = torch.empty(s.T, s.k, dtype=torch.int32, device=DEV)
    w = torch.empty(s.T, s.k, dtype=torch.float32, device=DEV)
    y = torch.full((s.T, s.H), float("nan"), device=DEV)
    ws = m.alloc_workspace(s.T, s.H, s.E, s.k, s.I, device=DEV)
    m.moe_layer_q8k(dev(case["x"]), dev(case["Wr"]), dev(case["bias"]), dev(b["gate"]),
                    dev(b["up"]), dev(b["down"]), s.k, s.I, idx, w, y, ws)
    code, detail = m.moe_read_device_status(ws)
    assert code == 0, (m.status_str(code), detail)
    return idx.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()


def check_q8k(case, idx, w, y):
    r = case["r"]
    np.testing.assert_array_equal(idx, r["idx"])
    assert np.max(np.abs(w.astype(np.float64) - r["w"])) <= W_TOL
    rows = slice(None) if case["tokens"] is None else case["tokens"]
    yo = r["y"][rows]
    yg = y[rows].astype(np.float64)
    assert np.all(np.isfinite(yg))
    err = float(np.max(np.abs(yg - yo)))
    tol = y_tolerance(yo)
    assert err <= tol, f"max|dy| = {err:.3e} > {tol:.3e}"


Q8K_SHAPES = [
    # name, T, H, E, k, I
    ("c0", 1, 256, 8, 2, 256),
    ("a3b-token", 1, 2048, 128, 8, 768),
    ("a22b-token", 1, 4096, 128, 8, 1536),
    ("small-batch", 5, 512, 16, 4, 256),
    ("odd-sizes", 3, 768, 12, 3, 512),
    ("batch-64", 64, 2048, 128, 8, 768),
    ("batch-300", 300, 512, 32, 2, 256),
]


@pytest.mark.parametrize("name,T,H,E,k,I", Q8K_SHAPES, ids=[s[0] for s in Q8K_SHAPES])
def test_layer_q8k_matches_oracle(m, name, T, H, E, k, I):
    shape = synth.custom_shape(T, H, E, k, I, wr_std=0.02, cfg_id=61 + T % 13, name=name)
    case = q8k_case(shape, 0, experts_only=(T == 1))
    check_q8k(case, *run_q8k(m, case))
    assert m.moe_layer_q8k_launch_count(T, H, E, k, I) == 5


@pytest.mark.parametrize("name", ["a3b_batch64_zipf", "a22b_batch32"])
def test_layer_q8k_workloads(m, name):
    """The batched workloads' first layer (the Zipf bias included), every token."""
    case = q8k_case(synth.SHAPES[name], 0)
    check_q8k(case, *run_q8k(m, case))


def test_ffn_q8k_caller_routing(m, oracle):
    """Duplicate experts in a row are legal; an index outside [0, E)
    contributes nothing and is recorded."""
    shape = synth.custom_shape(3, 512, 8, 3, 256, cfg_id=67)
    blobs = synth.expert_blobs(shape, 0)
    rng = np.random.default_rng(43)
    x = rng.normal(0, 1, (3, 512)).astype(np.float32)
    idx = np.array([[1, 1, 4], [7, 0, 2], [3, 9, 5]], np.int32)
    w = np.array([[0.5, 0.3, 0.2], [0.1, 0.6, 0.3], [0.4, 0.4, 0.2]], np.float32)
    yo, skipped = oracle.ffn_q8k(x, idx, w.astype(np.float64), blobs["gate"], blobs["up"],
                                 blobs["down"], 8, 256)
    assert skipped == 1
    t = lambda a: torch.from_numpy(a).to(DEV)  # noqa: E731
    y = torch.full((3, 512), float("nan"), device=DEV)
    ws = m.alloc_workspace(3, 512, 8, 3, 256, device=DEV)
    m.moe_ffn_q8k(t(x), t(idx), t(w), t(blobs["gate"]), t(blobs["up"]), t(blobs["down"]), 8, 256,
                  y, ws)
    code, detail = m.moe_read_device_status(ws)
    assert m.status_str(code) == "MOE_ERR_EXPERT_RANGE" and detail == 9
    yg = y.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(yg - yo)) <= y_tolerance(yo)


def test_layer_q8k_repeat_is_bitwise(m):
    shape = synth.custom_shape(64, 2048, 128, 8, 768, wr_std=0.02, cfg_id=68)
    case = q8k_case(shape, 1)
    a = run_q8k(m, case)
    for _ in range(3):
        b = run_q8k(m, case)
        for u, v in zip(a, b):
            np.testing.assert_array_equal(u, v)


def test_q8k_against_fp32_activations(m):
    """The two activation paths on the same layer: the Q8_K output's cosine
    with the fp32-activation output (measured, printed) stays above 0.99 on
    every token."""
    shape = synth.SHAPES["a3b_batch64_zipf"]
    case = q8k_case(shape, 2)
    _, _, yq = run_q8k(m, case)
    s = shape
    dev = lambda a: None if a is None else torch.from_numpy(a).to(DEV)  # noqa: E731
    b = case["blobs"]
    idx = torch.empty(s.T, s.k, dtype=torch.int32, device=DEV)
    w = torch.empty(s.T, s.k, dtype=torch.float32, device=DEV)
    y = torch.empty(s.T, s.H, device=DEV)
    ws = m.alloc_workspace(s.T, s.H, s.E, s.k, s.I, device=DEV)
    m.moe_layer(dev(case["x"]), dev(case["Wr"]), dev(case["bias"]), dev(b["gate"]), dev(b["up"]),
                dev(b["down"]), s.k, s.I, idx, w, y, ws)
    yf = y.cpu().numpy().astype(np.float64)
    yq = yq.astype(np.float64)
    cos = np.sum(yq * yf, axis=1) / (np.linalg.norm(yq, axis=1) * np.linalg.norm(yf, axis=1))
    print(f"cosine(Q8_K, fp32 activations) per token: min {cos.min():.6f} mean {cos.mean():.6f}")
    assert np.all(cos > 0.99)
