"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Bar: expert indices bit-exact, |w_gpu - w_oracle| <= 1e-6, and
max|y_gpu - y_oracle| <= 2e-3 * max|y_oracle| + 1e-5; permutation outputs
bit-exact.
"""
import numpy as np
import pytest

from quantized_routed_expert_02_gb300 import synth
from tests.cases import W_TOL, layer_case, y_tolerance

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_02_gb300 import build
    build.build()
    from quantized_routed_expert_02_gb300 import moeq4k
    return moeq4k


DEV = "cuda"


def to_dev(case):
    s = case["shape"]
    d = dict(
        x=torch.from_numpy(case["x"]).to(DEV),
        Wr=torch.from_numpy(case["Wr"]).to(DEV),
        bias=None if case["bias"] is None else torch.from_numpy(case["bias"]).to(DEV),
        gate=torch.from_numpy(case["blobs"]["gate"]).to(DEV),
        up=torch.from_numpy(case["blobs"]["up"]).to(DEV),
        down=torch.from_numpy(case["blobs"]["down"]).to(DEV),
        idx=torch.empty(s.T, s.k, dtype=torch.int32, device=DEV),
        w=torch.empty(s.T, s.k, dtype=torch.float32, device=DEV),
        y=torch.full((s.T, s.H), float("nan"), dtype=torch.float32, device=DEV),
    )
    return d


def run_layer(m, case, ws=None):
    s = case["shape"]
    d = to_dev(case)
    if ws is None:
        ws = m.alloc_workspace(s.T, s.H, s.E, s.k, s.I, device=DEV)
    m.moe_layer(d["x"], d["Wr"], d["bias"], d["gate"], d["up"], d["down"], s.k, s.I,
                d["idx"], d["w"], d["y"], ws)
    code, detail = m.moe_read_device_status(ws)
    assert code == 0, (m.status_str(code), detail)
    return d["idx"].cpu().numpy(), d["w"].cpu().numpy(), d["y"].cpu().numpy(), d, ws


def check_layer(case, idx, w, y):
    np.testing.assert_array_equal(idx, case["idx"])
    assert np.max(np.abs(w.astype(np.float64) - case["w"])) <= W_TOL
    rows = slice(None) if case["tokens"] is None else case["tokens"]
    yo = case["y"][rows]
    yg = y[rows].astype(np.float64)
    assert np.all(np.isfinite(yg))
    err = np.max(np.abs(yg - yo))
    tol = y_tolerance(yo)
    assert err <= tol, f"max|dy| = {err:.3e} > {tol:.3e}"
    return err / tol


# ---------------------------------------------------------------- full workloads

# every token of every workload is compared (the 4096-token prefill too:
# the oracle runs its tokens on all host cores)
WORKLOADS = [
    ("tiny", None),
    ("a3b_decode", None),
    ("a3b_batch64_zipf", None),
    ("a3b_prefill", None),
    ("a22b_decode", None),
    ("a22b_batch32", None),
]


@pytest.mark.parametrize("name,sample", WORKLOADS, ids=[w[0] for w in WORKLOADS])
def test_layer_workloads(m, name, sample):
    case = layer_case(synth.SHAPES[name], 0, sample)
    idx, w, y, _, _ = run_layer(m, case)
    check_layer(case, idx, w, y)


def test_a3b_decode_second_layer(m):
    case = layer_case(synth.SHAPES["a3b_decode"], 7, None)
    idx, w, y, _, _ = run_layer(m, case)
    check_layer(case, idx, w, y)


def test_router_all_tokens_prefill(m):
    """Routing of every one of the 4096 prefill tokens is bit-exact (the
    router entry point on its own)."""
    case = layer_case(synth.SHAPES["a3b_prefill"], 0, None)
    s = case["shape"]
    d = to_dev(case)
    ws = m.alloc_workspace(s.T, s.H, s.E, s.k, s.I, device=DEV)
    m.moe_router(d["x"], d["Wr"], d["bias"], s.k, d["idx"], d["w"], ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(d["idx"].cpu().numpy(), case["idx"])
    assert np.max(np.abs(d["w"].cpu().numpy() - case["w"])) <= W_TOL


def test_permutation_matches_oracle(m, oracle):
    case = layer_case(synth.SHAPES["a3b_batch64_zipf"], 0, None)
    s = case["shape"]
    idx = torch.from_numpy(case["idx"]).to(DEV)
    counts = torch.empty(s.E, dtype=torch.int32, device=DEV)
    offs = torch.empty(s.E + 1, dtype=torch.int32, device=DEV)
    perm = torch.full((s.T * s.k,), -7, dtype=torch.int32, device=DEV)
    ws = m.alloc_workspace(s.T, s.H, s.E, s.k, s.I, device=DEV)
    m.moe_permute(idx, s.E, counts, offs, perm, ws)
    c, o, p = oracle.permutation(case["idx"], s.E)
    np.testing.assert_array_equal(counts.cpu().numpy(), c)
    np.testing.assert_array_equal(offs.cpu().numpy(), o)
    np.testing.assert_array_equal(perm.cpu().numpy(), p)


@pytest.mark.parametrize("T", [1, 5, 1000, 4096])
def test_permutation_random(m, oracle, T):
    rng = np.random.default_rng(T)
    E, k = 128, 8
    idx_np = rng.integers(0, E, (T, k)).astype(np.int32)
    idx = torch.from_numpy(idx_np).to(DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    ws = m.alloc_workspace(T, 256, E, k, 256, device=DEV)
    m.moe_permute(idx, E, counts, offs, perm, ws)
    c, o, p = oracle.permutation(idx_np, E)
    np.testing.assert_array_equal(counts.cpu().numpy(), c)
    np.testing.assert_array_equal(offs.cpu().numpy(), o)
    np.testing.assert_array_equal(perm.cpu().numpy(), p)


# ---------------------------------------------------------------- small shapes with tails

SMALL = [
    (1, 256, 4, 1, 256), (3, 256, 8, 2, 512), (17, 512, 16, 4, 256), (300, 512, 8, 2, 512),
    (17, 256, 4, 4, 256), (3, 768, 16, 16, 256), (64, 1280, 16, 3, 768), (2, 256, 256, 32, 256),
]


@pytest.mark.parametrize("T,H,E,k,I", SMALL)
def test_layer_small_shapes(m, T, H, E, k, I):
    shape = synth.custom_shape(T, H, E, k, I, wr_std=0.05, cfg_id=50 + (T + H + E + k + I) % 40)
    case = layer_case(shape, 0, None)
    idx, w, y, _, _ = run_layer(m, case)
    check_layer(case, idx, w, y)


# ---------------------------------------------------------------- caller-given routing

def test_ffn_duplicates_and_bad_index(m, oracle):
    shape = synth.custom_shape(4, 512, 8, 3, 256, cfg_id=77)
    case = layer_case(shape, 0, None)
    idx_np = np.array([[1, 1, 2], [7, 0, 7], [3, 99, 4], [-1, 5, 5]], dtype=np.int32)
    w_np = np.array([[0.5, 0.25, 0.25], [0.1, 0.2, 0.7], [0.3, 0.3, 0.4], [1.0, 2.0, -0.5]],
                    dtype=np.float32)
    yo, skipped = oracle.ffn(case["x"], idx_np, w_np.astype(np.float64), case["blobs"]["gate"],
                             case["blobs"]["up"], case["blobs"]["down"], shape.E, shape.I)
    assert skipped == 2
    d = to_dev(case)
    ws = m.alloc_workspace(shape.T, shape.H, shape.E, shape.k, shape.I, device=DEV)
    m.moe_ffn(d["x"], torch.from_numpy(idx_np).to(DEV), torch.from_numpy(w_np).to(DEV),
              d["gate"], d["up"], d["down"], shape.E, shape.I, d["y"], ws)
    code, detail = m.moe_read_device_status(ws)
    assert code == 5 and detail in (99, -1)
    y = d["y"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(y - yo)) <= y_tolerance(yo)
    # the status is sticky until the workspace header is reset
    m.moe_workspace_init(ws)
    assert m.moe_read_device_status(ws)[0] == 0


def test_deterministic_repeat(m):
    case = layer_case(synth.SHAPES["a3b_batch64_zipf"], 0, None)
    s = case["shape"]
    _, _, y1, d, ws = run_layer(m, case)
    for _ in range(2):
        m.moe_layer(d["x"], d["Wr"], d["bias"], d["gate"], d["up"], d["down"], s.k, s.I,
                    d["idx"], d["w"], d["y"], ws)
        np.testing.assert_array_equal(d["y"].cpu().numpy(), y1)


def test_layer_host_entry(m):
    case = layer_case(synth.SHAPES["a3b_decode"], 0, None)
    s = case["shape"]
    d = to_dev(case)
    ws = m.alloc_workspace(s.T, s.H, s.E, s.k, s.I, device=DEV, host_staging=True)
    xh = torch.from_numpy(case["x"]).pin_memory()
    yh = torch.empty(s.T, s.H, dtype=torch.float32).pin_memory()
    m.moe_layer_host(xh, d["Wr"], d["bias"], d["gate"], d["up"], d["down"], s.k, s.I,
                     d["idx"], d["w"], yh, ws)
    check_layer(case, d["idx"].cpu().numpy(), d["w"].cpu().numpy(), yh.numpy())
    # pinned buffers at a single token are read and written in place by the
    # fused kernel: the same numbers as the device entry point
    m.moe_layer(d["x"], d["Wr"], d["bias"], d["gate"], d["up"], d["down"], s.k, s.I, d["idx"],
                d["w"], d["y"], m.alloc_workspace(s.T, s.H, s.E, s.k, s.I, device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(d["y"].cpu(), yh)


@pytest.mark.parametrize("shape", [synth.SHAPES["a3b_decode"],
                                   synth.custom_shape(5, 512, 16, 4, 256, wr_std=0.02, cfg_id=71)],
                         ids=["single-token", "five-tokens"])
@pytest.mark.parametrize("pinned", [False, True], ids=["pageable", "pinned"])
def test_layer_host_entry_buffers(m, shape, pinned):
    """Pageable host buffers (and every batch) go through the workspace's
    staging copies, pinned single-token buffers are used in place: the
    results agree with the oracle either way."""
    case = layer_case(shape, 1, None)
    s = case["shape"]
    d = to_dev(case)
    ws = m.alloc_workspace(s.T, s.H, s.E, s.k, s.I, device=DEV, host_staging=True)
    xh = torch.from_numpy(case["x"].copy())
    yh = torch.full((s.T, s.H), float("nan"), dtype=torch.float32)
    if pinned:
        xh, yh = xh.pin_memory(), yh.pin_memory()
    m.moe_layer_host(xh, d["Wr"], d["bias"], d["gate"], d["up"], d["down"], s.k, s.I,
                     d["idx"], d["w"], yh, ws)
    check_layer(case, d["idx"].cpu().numpy(), d["w"].cpu().numpy(), yh.numpy())
    code, detail = m.moe_read_device_status(ws)
    assert code == 0, (m.status_str(code), detail)


def test_nonzero_stream(m):
    case = layer_case(synth.SHAPES["tiny"], 0, None)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        idx, w, y, _, _ = run_layer(m, case)
    check_layer(case, idx, w, y)
