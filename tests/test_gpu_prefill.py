"""Large batches run the tensor-core grouped GEMMs (tcgen05, fp16 operands,
fp32 accumulation); compared with the fp64 oracle on every token, with
ragged expert chunks (more than 256 slots for an expert, fewer than 16)."""
import numpy as np
import pytest

from quantized_routed_expert_02_gb300 import synth
from tests.cases import layer_case
from tests.test_gpu_parity import check_layer, m, run_layer  # noqa: F401

pytestmark = pytest.mark.gpu

SHAPES = [
    # T, H, E, k, I, wr_std, zipf
    (1024, 512, 16, 2, 256, 0.05, False),
    (700, 768, 8, 4, 512, 0.05, False),
    (2048, 256, 64, 1, 256, 0.05, True),
    (513, 1024, 32, 8, 768, 0.03, True),
    (512, 256, 256, 8, 256, 0.05, False),
]


def tensor_path_launches(T, k):
    """Launches of a tensor-core-path call: the router (one launch, top-k
    fused, at every batch size), the permutation with the chunk plans (one
    launch up to 4096 routed slots, else three), fp16 rows, two GEMMs,
    combine."""
    return 1 + (1 if T * k <= 4096 else 3) + 1 + 2 + 1


@pytest.mark.parametrize("T,H,E,k,I,std,zipf", SHAPES)
def test_prefill_shapes(m, T, H, E, k, I, std, zipf):
    shape = synth.custom_shape(T, H, E, k, I, wr_std=std, zipf_bias=zipf,
                               cfg_id=70 + (T + H + E + k + I) % 20)
    assert m.moe_layer_launch_count(T, H, E, k, I) == tensor_path_launches(T, k)
    case = layer_case(shape, 0, None)   # every token
    idx, w, y, _, _ = run_layer(m, case)
    check_layer(case, idx, w, y)


def test_prefill_repeat_is_bitwise(m):
    shape = synth.custom_shape(1024, 512, 16, 2, 256, cfg_id=88)
    case = layer_case(shape, 0, (0, 1, 1023))
    s = shape
    _, _, y1, d, ws = run_layer(m, case)
    for _ in range(2):
        m.moe_layer(d["x"], d["Wr"], d["bias"], d["gate"], d["up"], d["down"], s.k, s.I,
                    d["idx"], d["w"], d["y"], ws)
        np.testing.assert_array_equal(d["y"].cpu().numpy(), y1)


def test_caller_routing_beyond_chunk_capacity(m, oracle):
    """A small batch caps its chunks at the token count rounded up to 32 (64
    here); a caller's routing that repeats experts gives experts 0 and 1 about
    160 slots each, which the plan splits into several chunks."""
    import torch
    from tests.cases import y_tolerance
    from tests.test_gpu_parity import DEV, to_dev
    shape = synth.custom_shape(40, 512, 8, 8, 256, cfg_id=91)
    assert m.moe_layer_launch_count(40, 512, 8, 8, 256) == tensor_path_launches(40, 8)
    case = layer_case(shape, 0, (0, 1, 17, 39))
    rng = np.random.default_rng(91)
    idx_np = rng.integers(0, 2, (40, 8)).astype(np.int32)
    idx_np[::5, 3] = 5
    w_np = rng.uniform(-1.0, 1.0, (40, 8)).astype(np.float32)
    yo, skipped = oracle.ffn(case["x"], idx_np, w_np.astype(np.float64), case["blobs"]["gate"],
                             case["blobs"]["up"], case["blobs"]["down"], shape.E, shape.I)
    assert skipped == 0
    d = to_dev(case)
    ws = m.alloc_workspace(40, shape.H, shape.E, shape.k, shape.I, device=DEV)
    m.moe_ffn(d["x"], torch.from_numpy(idx_np).to(DEV), torch.from_numpy(w_np).to(DEV),
              d["gate"], d["up"], d["down"], shape.E, shape.I, d["y"], ws)
    assert m.moe_read_device_status(ws)[0] == 0
    y = d["y"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(y - yo)) <= y_tolerance(yo)


def test_down_readiness_timeout_is_reported(m):
    """The down GEMM waits per expert for the gate/up launch's count of
    finished h rows.  With CTA 0 of the gate/up launch counting none of its
    rows (test hook) that count never completes: the bounded wait runs out,
    the call records MOE_ERR_TIMEOUT (at the readiness wait, or at the MMA
    warp's wait for the same activation tile) instead of hanging, and the
    workspace works again after re-initialisation."""
    from tests.test_gpu_parity import DEV, to_dev
    shape = synth.custom_shape(64, 512, 16, 8, 256, cfg_id=93)
    s = shape
    assert m.moe_layer_launch_count(s.T, s.H, s.E, s.k, s.I) == tensor_path_launches(s.T, s.k)
    case = layer_case(shape, 0, (0, 31, 63))
    d = to_dev(case)
    ws = m.alloc_workspace(s.T, s.H, s.E, s.k, s.I, device=DEV)
    try:
        m.moe_debug_set_wait_limit(20_000_000)      # 20 ms
        m.moe_debug_withhold_arrivals(1)
        m.moe_layer(d["x"], d["Wr"], d["bias"], d["gate"], d["up"], d["down"], s.k, s.I,
                    d["idx"], d["w"], d["y"], ws)
        code, detail = m.moe_read_device_status(ws)
        # 21: the readiness wait; 18: the MMA warp's wait for the same
        # activation tile (both run out at the same deadline)
        assert m.status_str(code) == "MOE_ERR_TIMEOUT" and detail in (18, 21), (code, detail)
    finally:
        m.moe_debug_withhold_arrivals(0)
        m.moe_debug_set_wait_limit(0)
    m.moe_workspace_init(ws)
    idx, w, y, _, _ = run_layer(m, case, ws=ws)
    check_layer(case, idx, w, y)


def test_caller_routing_invalid_experts_tensor_path(m, oracle):
    """A caller's routing on the tensor-core path (48 tokens x 8 slots) with a
    few expert indices outside [0, E): those slots take no sorted row, count
    toward no expert's readiness and add nothing to y; the call records
    MOE_ERR_EXPERT_RANGE and y matches the oracle, which skips them too."""
    import torch
    from tests.cases import y_tolerance
    from tests.test_gpu_parity import DEV, to_dev
    shape = synth.custom_shape(48, 512, 16, 8, 256, cfg_id=94)
    assert m.moe_layer_launch_count(48, 512, 16, 8, 256) == tensor_path_launches(48, 8)
    case = layer_case(shape, 0, (0, 1, 47))
    rng = np.random.default_rng(94)
    idx_np = rng.integers(0, 16, (48, 8)).astype(np.int32)
    idx_np[3, 2] = -1
    idx_np[17, 7] = 16
    idx_np[40, 0] = 1000
    w_np = rng.uniform(-1.0, 1.0, (48, 8)).astype(np.float32)
    yo, skipped = oracle.ffn(case["x"], idx_np, w_np.astype(np.float64), case["blobs"]["gate"],
                             case["blobs"]["up"], case["blobs"]["down"], shape.E, shape.I)
    assert skipped == 3
    d = to_dev(case)
    ws = m.alloc_workspace(48, shape.H, shape.E, shape.k, shape.I, device=DEV)
    m.moe_ffn(d["x"], torch.from_numpy(idx_np).to(DEV), torch.from_numpy(w_np).to(DEV),
              d["gate"], d["up"], d["down"], shape.E, shape.I, d["y"], ws)
    code, _ = m.moe_read_device_status(ws)
    assert m.status_str(code) == "MOE_ERR_EXPERT_RANGE"
    y = d["y"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(y - yo)) <= y_tolerance(yo)
