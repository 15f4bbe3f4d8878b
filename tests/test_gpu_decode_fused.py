"""Single-token calls (one persistent kernel) against the oracle, the
caller-routing entry at T=1, and the bounded-wait time-out."""
import numpy as np
import pytest

from quantized_routed_expert_02_gb300 import synth
from tests.cases import layer_case, y_tolerance
from tests.test_gpu_parity import DEV, check_layer, m, run_layer, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_single_token_is_one_launch(m):
    for name in ("tiny", "a3b_decode"):
        s = synth.SHAPES[name]
        assert m.moe_layer_launch_count(s.T, s.H, s.E, s.k, s.I) == 1
    s = synth.SHAPES["a3b_batch64_zipf"]
    assert m.moe_layer_launch_count(s.T, s.H, s.E, s.k, s.I) > 1


@pytest.mark.parametrize("layer", [1, 2, 3])
def test_a3b_decode_more_layers(m, layer):
    case = layer_case(synth.SHAPES["a3b_decode"], layer, None)
    idx, w, y, _, _ = run_layer(m, case)
    check_layer(case, idx, w, y)


@pytest.mark.parametrize("H,E,k,I", [(256, 8, 1, 256), (512, 16, 16, 256), (1280, 64, 6, 512),
                                     (2048, 256, 32, 256), (768, 4, 4, 1024)])
def test_single_token_shapes(m, H, E, k, I):
    shape = synth.custom_shape(1, H, E, k, I, wr_std=0.05, cfg_id=60 + (H + E + k + I) % 30)
    case = layer_case(shape, 0, None)
    idx, w, y, _, _ = run_layer(m, case)
    check_layer(case, idx, w, y)


def test_single_token_caller_routing(m, oracle):
    shape = synth.SHAPES["a3b_decode"]
    case = layer_case(shape, 0, None)
    d = to_dev(case)
    ws = m.alloc_workspace(1, shape.H, shape.E, shape.k, shape.I, device=DEV)
    idx_np = np.array([[5, 5, 127, 0, 200, 64, 3, -2]], dtype=np.int32)
    w_np = np.array([[0.5, 0.25, -1.0, 2.0, 7.0, 0.125, 0.0, 1.0]], dtype=np.float32)
    yo, skipped = oracle.ffn(case["x"], idx_np, w_np.astype(np.float64), case["blobs"]["gate"],
                             case["blobs"]["up"], case["blobs"]["down"], shape.E, shape.I)
    assert skipped == 2
    m.moe_ffn(d["x"], torch.from_numpy(idx_np).to(DEV), torch.from_numpy(w_np).to(DEV),
              d["gate"], d["up"], d["down"], shape.E, shape.I, d["y"], ws)
    code, detail = m.moe_read_device_status(ws)
    assert code == 5 and detail in (200, -2)
    y = d["y"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(y - yo)) <= y_tolerance(yo)


def test_single_token_repeat_bitwise(m):
    case = layer_case(synth.SHAPES["a3b_decode"], 0, None)
    s = case["shape"]
    _, _, y1, d, ws = run_layer(m, case)
    for _ in range(3):
        m.moe_layer(d["x"], d["Wr"], d["bias"], d["gate"], d["up"], d["down"], s.k, s.I,
                    d["idx"], d["w"], d["y"], ws)
        np.testing.assert_array_equal(d["y"].cpu().numpy(), y1)


def test_workspace_shared_with_batched_calls(m):
    """One workspace serves single-token and batched calls in turn: the
    batched path's scratch never disturbs the tagged values the single-token
    kernel keeps between calls, so each single-token result is bit-identical
    to the one from a fresh workspace."""
    dec = layer_case(synth.SHAPES["a3b_decode"], 0, None)
    bat = layer_case(synth.SHAPES["a3b_batch64_zipf"], 0, None)
    sb = bat["shape"]
    _, _, y_fresh, _, _ = run_layer(m, dec)
    ws = m.alloc_workspace(sb.T, sb.H, sb.E, sb.k, sb.I, device=DEV)
    for _ in range(2):
        idx, w, y, _, _ = run_layer(m, dec, ws=ws)
        check_layer(dec, idx, w, y)
        np.testing.assert_array_equal(y, y_fresh)
        idx, w, y, _, _ = run_layer(m, bat, ws=ws)
        check_layer(bat, idx, w, y)


def test_grid_barrier_timeout_is_reported(m):
    """A published value that never comes (CTA 0 publishes none of its router
    logits): the bounded waits run out, the call records MOE_ERR_TIMEOUT, and
    the workspace works again after re-initialisation."""
    case = layer_case(synth.SHAPES["tiny"], 0, None)
    s = case["shape"]
    d = to_dev(case)
    ws = m.alloc_workspace(1, s.H, s.E, s.k, s.I, device=DEV)
    try:
        m.moe_debug_set_wait_limit(20_000_000)      # 20 ms
        m.moe_debug_withhold_arrivals(1)
        m.moe_layer(d["x"], d["Wr"], d["bias"], d["gate"], d["up"], d["down"], s.k, s.I,
                    d["idx"], d["w"], d["y"], ws)
        code, _ = m.moe_read_device_status(ws)
        assert code == 6
    finally:
        m.moe_debug_withhold_arrivals(0)
        m.moe_debug_set_wait_limit(0)
    m.moe_workspace_init(ws)
    idx, w, y, _, _ = run_layer(m, case, ws=ws)
    check_layer(case, idx, w, y)
