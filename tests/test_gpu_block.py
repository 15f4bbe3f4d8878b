"""The layer with its neighbouring decoder-block steps (moe_layer_block)
against the oracle: pre-FFN RMSNorm, router, expert FFN, residual add, and
the capture of one token's router stage and pre-residual FFN output.

forward_qwen3_moe.rs (aprender-serve 0.35.0), steps 2f-2h of
forward_qwen3_moe: ffn_input = rms_norm(hidden, ffn_norm_weight, eps), the
MoE FFN, hidden += ffn_output.  forward_qwen3_moe_cuda_traced.rs
(aprender-serve 0.34.0), doc of forward_qwen3_moe_cuda_traced_with_plan: the
MoeRouter stage is the last token's k renormalised weights, MoeFfnOut its
[H] FFN output.

Bar: expert indices bit-exact; |w - w_oracle| <= 1e-6; the output and the
captured FFN row within 2e-3 * max|y_oracle| + 1e-5 (y the FFN output before
the residual); the captured routing equal to the call's own idx / w rows.
Rows of the residual stream are redrawn until the router input (the normed
row) has no near tie among its top k+1 logits.
"""
import numpy as np
import pytest

from oracle.oracle import Oracle, near_tie_free
from quantized_routed_expert_02_gb300 import synth
from tests.cases import GAP, W_TOL, y_tolerance
from tests.test_gpu_parity import DEV, m  # noqa: F401

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

EPS = 1e-6


def block_case(shape, layer, norm=True, experts_only=False):
    o = Oracle()
    Wr = synth.router_weights(shape, layer)
    bias = synth.router_bias(shape)
    rng = np.random.default_rng([layer, 777])
    gamma = rng.uniform(0.5, 1.5, shape.H).astype(np.float32) if norm else None
    hidden = np.stack([3.0 * synth.x_row(shape, layer, t, 0) for t in range(shape.T)])
    attempt = np.zeros(shape.T, dtype=np.int32)
    for _ in range(32):
        xin = hidden if gamma is None else o.rmsnorm(hidden, gamma, EPS)
        lg = o.router(xin, Wr, bias, shape.k)["logits"]
        bad = [t for t in range(shape.T) if not near_tie_free(lg[t], shape.k, GAP)]
        if not bad:
            break
        for t in bad:
            attempt[t] += 1
            hidden[t] = 3.0 * synth.x_row(shape, layer, t, int(attempt[t]))
    else:
        raise RuntimeError("no tie-free draw")
    hidden = hidden.astype(np.float32)
    xin = hidden if gamma is None else o.rmsnorm(hidden, gamma, EPS)
    r0 = o.router(xin, Wr, bias, shape.k)
    experts = sorted(set(r0["idx"].ravel().tolist())) if experts_only else None
    blobs = synth.expert_blobs(shape, layer, experts=experts)
    r = o.block(hidden, gamma, EPS, Wr, bias, shape.k, blobs["gate"], blobs["up"], blobs["down"],
                shape.E, shape.I, residual=True)
    return dict(shape=shape, hidden=hidden, gamma=gamma, Wr=Wr, bias=bias, blobs=blobs, r=r)


def run_block(m, case, in_place=False, capture=True, residual=True):
    s = case["shape"]
    dev = lambda a: None if a is None else torch.from_numpy(a).to(DEV)  # noqa: E731
    hidden = dev(case["hidden"])
    out = hidden if in_place else torch.full_like(hidden, float("nan"))
    idx = torch.empty(s.T, s.k, dtype=torch.int32, device=DEV)
    w = torch.empty(s.T, s.k, dtype=torch.float32, device=DEV)
    cap_idx = torch.full((s.k,), -1, dtype=torch.int32, device=DEV)
    cap_w = torch.full((s.k,), float("nan"), device=DEV)
    cap_ffn = torch.full((s.H,), float("nan"), device=DEV)
    ws = m.alloc_workspace(s.T, s.H, s.E, s.k, s.I, device=DEV)
    blobs = case["blobs"]
    m.moe_layer_block(hidden, dev(case["gamma"]), EPS, dev(case["Wr"]), dev(case["bias"]),
                      dev(blobs["gate"]), dev(blobs["up"]), dev(blobs["down"]), s.k, s.I, idx, w,
                      out, ws, add_residual=residual, capture_token=s.T - 1 if capture else -1,
                      cap_idx=cap_idx, cap_w=cap_w, cap_ffn=cap_ffn)
    code, detail = m.moe_read_device_status(ws)
    assert code == 0, (m.status_str(code), detail)
    return dict(idx=idx.cpu().numpy(), w=w.cpu().numpy(), out=out.cpu().numpy(),
                cap_idx=cap_idx.cpu().numpy(), cap_w=cap_w.cpu().numpy(),
                cap_ffn=cap_ffn.cpu().numpy())


def check_block(case, g, capture=True, residual=True):
    r = case["r"]
    np.testing.assert_array_equal(g["idx"], r["idx"])
    assert np.max(np.abs(g["w"].astype(np.float64) - r["w"])) <= W_TOL
    tol = y_tolerance(r["y"])
    want = r["out"] if residual else r["y"]
    assert np.all(np.isfinite(g["out"]))
    err = np.max(np.abs(g["out"].astype(np.float64) - want))
    assert err <= tol, f"max|d out| = {err:.3e} > {tol:.3e}"
    if capture:
        t = case["shape"].T - 1
        np.testing.assert_array_equal(g["cap_idx"], g["idx"][t])
        np.testing.assert_array_equal(g["cap_w"], g["w"][t])
        err = np.max(np.abs(g["cap_ffn"].astype(np.float64) - r["y"][t]))
        assert err <= tol, f"captured FFN row: {err:.3e} > {tol:.3e}"
    else:
        assert np.all(g["cap_idx"] == -1) and np.all(np.isnan(g["cap_ffn"]))


BLOCK_SHAPES = [
    # name, T, H, E, k, I: which path
    ("fused-a3b", 1, 2048, 128, 8, 768),     # single-token fused kernel (norm in its staging)
    ("streamed-a22b", 1, 4096, 32, 8, 1536),  # norm launch, row router, streamed launches
    ("cuda-core", 40, 512, 16, 4, 256),       # norm launch, batched CUDA-core path
    ("tensor-a3b", 64, 2048, 128, 8, 768),    # norm launch, tcgen05 grouped GEMMs
    ("tensor-split", 300, 512, 16, 2, 512),   # split-K router, GEMMs
]


@pytest.mark.parametrize("name,T,H,E,k,I", BLOCK_SHAPES, ids=[b[0] for b in BLOCK_SHAPES])
def test_block_norm_residual_capture(m, name, T, H, E, k, I):
    shape = synth.custom_shape(T, H, E, k, I, wr_std=0.02, cfg_id=55 + T % 11, name=name)
    case = block_case(shape, 0, norm=True, experts_only=(T == 1))
    check_block(case, run_block(m, case))


@pytest.mark.parametrize("name,T,H,E,k,I", [BLOCK_SHAPES[0], BLOCK_SHAPES[3]],
                         ids=[BLOCK_SHAPES[0][0], BLOCK_SHAPES[3][0]])
def test_block_in_place_residual(m, name, T, H, E, k, I):
    """out may be hidden itself: hidden += ffn(norm(hidden))."""
    shape = synth.custom_shape(T, H, E, k, I, wr_std=0.02, cfg_id=56 + T % 11, name=name)
    case = block_case(shape, 1, norm=True, experts_only=(T == 1))
    check_block(case, run_block(m, case, in_place=True))


def test_block_without_norm_or_residual_or_capture(m):
    """No norm weight: the FFN sees hidden itself; no residual: out is the
    FFN output; no capture token: the capture buffers are untouched."""
    shape = synth.custom_shape(1, 2048, 128, 8, 768, wr_std=0.02, cfg_id=58, name="plain")
    case = block_case(shape, 2, norm=False, experts_only=True)
    check_block(case, run_block(m, case, capture=False, residual=False), capture=False,
                residual=False)
    case = block_case(synth.custom_shape(40, 512, 16, 4, 256, wr_std=0.02, cfg_id=59), 0,
                      norm=False)
    check_block(case, run_block(m, case, residual=True), residual=True)


def test_block_rejects_bad_capture_token(m):
    s = synth.custom_shape(2, 256, 8, 2, 256)
    ws = m.alloc_workspace(2, 256, 8, 2, 256, device=DEV)
    z = lambda *sh: torch.zeros(*sh, device=DEV)  # noqa: E731
    gate = torch.zeros(8 * 256 * 144, dtype=torch.uint8, device=DEV)
    with pytest.raises(m.MoeError):
        m.moe_layer_block(z(2, 256), None, EPS, z(8, 256), None, gate, gate, gate, s.k, s.I,
                          torch.zeros(2, 2, dtype=torch.int32, device=DEV), z(2, 2), z(2, 256), ws,
                          capture_token=2)
