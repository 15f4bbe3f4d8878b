"""Single-token calls whose expert rows do not fit the fused kernel (the
Qwen3-235B-A22B shape among them): router, then the streamed gate/up and
down launches (integer-digit dot products, fp32 fallbacks) with the
slot-ordered combine folded into the down pass."""
import numpy as np
import pytest

from quantized_routed_expert_02_gb300 import synth
from tests.cases import layer_case, y_tolerance
from tests.test_gpu_parity import DEV, check_layer, m, run_layer, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

STREAM_LAUNCHES = 3  # router (logits and top-k), gate/up, down + combine


def test_a22b_single_token_takes_the_streamed_path(m):
    s = synth.SHAPES["a22b_decode"]
    assert m.moe_layer_launch_count(s.T, s.H, s.E, s.k, s.I) == STREAM_LAUNCHES


# Integer-digit kernels for both launches: the A22B row lengths, many slots
# (k = 32, k*I/64 = 512 units: every thread of the CTA), long x (H = 8192:
# 128 units), odd block counts per down row (I = 1280: five blocks).  The
# fp32 fallbacks: gate/up for H = 1280 (not a power of two), down for
# k*I/64 = 768 units (more than the CTA's threads).
# The down launch's per-lane width G = ceil(k*I/64 / 32) is a template
# argument: (8192, 4, 2, 1024) has 32 units per row (G = 1), (8192, 4, 2,
# 1280) 40 (G = 2), (8192, 4, 4, 1536) 96 (G = 4), the A22B shape 192 (G = 6);
# (1024, 32, 32, 1024) and (2048, 16, 16, 2048) have 512 and take G = 4 in
# four rounds.
@pytest.mark.parametrize("H,E,k,I", [(4096, 8, 8, 1536), (1024, 32, 32, 1024),
                                     (8192, 4, 2, 1280), (2048, 16, 16, 2048),
                                     (1280, 8, 8, 2048), (1024, 16, 12, 4096),
                                     (8192, 4, 2, 1024), (8192, 4, 4, 1536)])
def test_streamed_shapes(m, H, E, k, I):
    assert m.moe_layer_launch_count(1, H, E, k, I) == STREAM_LAUNCHES
    shape = synth.custom_shape(1, H, E, k, I, wr_std=0.03, cfg_id=20 + (H + E + k + I) % 30)
    case = layer_case(shape, 0, None)
    idx, w, y, _, _ = run_layer(m, case)
    check_layer(case, idx, w, y)


def test_streamed_caller_routing(m, oracle):
    """Duplicate experts and out-of-range ids: the bad slots are skipped and
    recorded, the rest match the oracle."""
    shape = synth.custom_shape(1, 4096, 8, 8, 1536, wr_std=0.03, cfg_id=21)
    assert m.moe_layer_launch_count(1, 4096, 8, 8, 1536) == STREAM_LAUNCHES
    case = layer_case(shape, 0, None)
    d = to_dev(case)
    ws = m.alloc_workspace(1, shape.H, shape.E, shape.k, shape.I, device=DEV)
    idx_np = np.array([[1, 1, 3, 99, 0, 7, -1, 5]], dtype=np.int32)
    w_np = np.array([[0.5, 0.25, -1.0, 2.0, 0.75, 0.125, 3.0, 1.0]], dtype=np.float32)
    yo, skipped = oracle.ffn(case["x"], idx_np, w_np.astype(np.float64), case["blobs"]["gate"],
                             case["blobs"]["up"], case["blobs"]["down"], shape.E, shape.I)
    assert skipped == 2
    m.moe_ffn(d["x"], torch.from_numpy(idx_np).to(DEV), torch.from_numpy(w_np).to(DEV),
              d["gate"], d["up"], d["down"], shape.E, shape.I, d["y"], ws)
    code, detail = m.moe_read_device_status(ws)
    assert code == 5 and detail in (99, -1)
    y = d["y"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(y - yo)) <= y_tolerance(yo)


def test_streamed_repeat_is_bitwise(m):
    case = layer_case(synth.SHAPES["a22b_decode"], 0, None)
    s = case["shape"]
    _, _, y1, d, ws = run_layer(m, case)
    for _ in range(3):
        m.moe_layer(d["x"], d["Wr"], d["bias"], d["gate"], d["up"], d["down"], s.k, s.I,
                    d["idx"], d["w"], d["y"], ws)
        np.testing.assert_array_equal(d["y"].cpu().numpy(), y1)
