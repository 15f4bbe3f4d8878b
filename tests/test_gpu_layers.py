"""Every layer of the timing rotations against the oracle.

The benchmark runs each workload over a rotation of independently seeded
layers; here each of those layers (all 48 of the Qwen3-30B-A3B single token,
all 8 of the Qwen3-235B-A22B single token and 32-token batch, four of the
64-token Zipf batch and of the 4096-token prefill) is compared with the fp64
oracle on every token: expert indices bit-exact, |dw| <= 1e-6, y within
2e-3 * max|y| + 1e-5.

Single-token layers only need their eight routed experts, so only those
experts' matrices are generated (the other experts' bytes stay zero, which
a correct kernel never reads).
"""
import pytest

from oracle.oracle import Oracle
from quantized_routed_expert_02_gb300 import synth
from tests.cases import tie_free_x
from tests.test_gpu_parity import DEV, check_layer, m, run_layer  # noqa: F401

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def routed_case(shape, layer, o, blobs=None, experts_only=False):
    """Tie-screened inputs of one layer and the oracle's results on every
    token.  ``blobs``: reuse these expert matrices (same layer seed)."""
    Wr = synth.router_weights(shape, layer)
    bias = synth.router_bias(shape)
    x, _ = tie_free_x(o, shape, layer, Wr, bias)
    r = o.router(x, Wr, bias, shape.k)
    if blobs is None:
        experts = sorted(set(r["idx"].ravel().tolist())) if experts_only else None
        blobs = synth.expert_blobs(shape, layer, experts=experts)
    y, skipped = o.ffn(x, r["idx"], r["w"], blobs["gate"], blobs["up"], blobs["down"],
                       shape.E, shape.I)
    assert skipped == 0
    return dict(shape=shape, x=x, Wr=Wr, bias=bias, blobs=blobs, idx=r["idx"], w=r["w"],
                logits=r["logits"], y=y, tokens=None)


def test_a3b_decode_all_48_layers(m):
    shape = synth.SHAPES["a3b_decode"]
    o = Oracle()
    ws = m.alloc_workspace(1, shape.H, shape.E, shape.k, shape.I, device=DEV)
    worst = 0.0
    for layer in range(shape.layers):
        case = routed_case(shape, layer, o, experts_only=True)
        idx, w, y, _, _ = run_layer(m, case, ws=ws)
        worst = max(worst, check_layer(case, idx, w, y))
    assert worst <= 1.0


def test_a22b_all_8_layers_single_token_and_batch(m):
    """Both Qwen3-235B-A22B workloads share each layer's expert matrices."""
    dec, bat = synth.SHAPES["a22b_decode"], synth.SHAPES["a22b_batch32"]
    assert dec.cfg_id == bat.cfg_id and dec.layers == bat.layers == 8
    o = Oracle()
    for layer in range(dec.layers):
        case_b = routed_case(bat, layer, o)
        idx, w, y, _, _ = run_layer(m, case_b)
        check_layer(case_b, idx, w, y)
        case_d = routed_case(dec, layer, o, blobs=case_b["blobs"])
        idx, w, y, _, _ = run_layer(m, case_d)
        check_layer(case_d, idx, w, y)
        del case_b, case_d
        torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["a3b_batch64_zipf", "a3b_prefill"])
def test_batched_four_layers(m, name):
    shape = synth.SHAPES[name]
    o = Oracle()
    ws = m.alloc_workspace(shape.T, shape.H, shape.E, shape.k, shape.I, device=DEV)
    for layer in range(4):
        case = routed_case(shape, layer, o)
        idx, w, y, _, _ = run_layer(m, case, ws=ws)
        check_layer(case, idx, w, y)
        del case
        torch.cuda.empty_cache()
