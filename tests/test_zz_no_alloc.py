"""The allocation-free single-token entry point, checked against the
workspace entry point and against the oracle.

moe_layer_noalloc serves callers that cannot allocate device memory (a
plugin whose host framework owns every device allocation, or a decode loop
that must never reach an allocator on its hot path): it runs the
single-token kernel with the library's own fixed scratch array.  It runs the
same deterministic kernel as moe_layer, so its routing and output must be
bit-identical to moe_layer's, and both must match the fp64 oracle (indices
bit-exact, |dw| <= 1e-6, y within 2e-3 * max|y| + 1e-5) on tie-screened
inputs.  Two calls in a row are checked: the second sees the first call's
leftovers in the shared scratch.  Collected last, so that a failure here
comes after every other test has run; it also passes on its own in a fresh
process.
"""
import ctypes

import numpy as np
import pytest

from quantized_routed_expert_02_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _noalloc_fn(m):
    f = ctypes.CDLL(m.LIB_PATH).moe_layer_noalloc
    P, I_ = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, P, P, P, I_, I_, I_, I_, I_, P, P, P, P]
    f.restype = ctypes.c_int
    return f


def test_noalloc_matches_workspace_entry_and_oracle_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_02_gb300 import build
    build.build()
    from quantized_routed_expert_02_gb300 import moeq4k as m
    from tests.cases import W_TOL, layer_case, y_tolerance

    dev = "cuda"
    s = synth.SHAPES["a3b_decode"]
    f = _noalloc_fn(m)
    ws = m.alloc_workspace(1, s.H, s.E, s.k, s.I, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    for layer in (0, 1):   # two calls in a row through the same shared scratch
        case = layer_case(s, layer, None)
        x = torch.from_numpy(case["x"]).to(dev)
        Wr = torch.from_numpy(case["Wr"]).to(dev)
        gate, up, down = (torch.from_numpy(case["blobs"][n]).to(dev)
                          for n in ("gate", "up", "down"))
        idx_r = torch.empty(1, s.k, dtype=torch.int32, device=dev)
        w_r = torch.empty(1, s.k, device=dev)
        y_r = torch.empty(1, s.H, device=dev)
        m.moe_layer(x, Wr, None, gate, up, down, s.k, s.I, idx_r, w_r, y_r, ws)
        idx_n = torch.full((1, s.k), -1, dtype=torch.int32, device=dev)
        w_n = torch.full((1, s.k), float("nan"), device=dev)
        y_n = torch.full((1, s.H), float("nan"), device=dev)
        rc = f(x.data_ptr(), Wr.data_ptr(), None, gate.data_ptr(), up.data_ptr(),
               down.data_ptr(), 1, s.H, s.E, s.k, s.I, idx_n.data_ptr(), w_n.data_ptr(),
               y_n.data_ptr(), stream)
        assert rc == 0, m.status_str(rc)
        torch.cuda.synchronize()
        # the same kernel on the same inputs: bit-identical to the workspace entry
        np.testing.assert_array_equal(idx_n.cpu().numpy(), idx_r.cpu().numpy())
        np.testing.assert_array_equal(w_n.cpu().numpy(), w_r.cpu().numpy())
        np.testing.assert_array_equal(y_n.cpu().numpy(), y_r.cpu().numpy())
        # and within the tolerance of the oracle
        np.testing.assert_array_equal(idx_n.cpu().numpy(), case["idx"])
        assert np.max(np.abs(w_n.cpu().numpy().astype(np.float64) - case["w"])) <= W_TOL
        yn = y_n.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(yn))
        assert np.max(np.abs(yn - case["y"])) <= y_tolerance(case["y"])
    assert m.moe_read_device_status(ws)[0] == 0


def test_noalloc_rejects_oversize_and_batches():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_02_gb300 import build
    build.build()
    from quantized_routed_expert_02_gb300 import moeq4k as m
    f = _noalloc_fn(m)
    a = 1 << 20
    # k*I = 32*8192 values of h are beyond the fixed scratch
    assert f(a, a, None, a, a, a, 1, 256, 64, 32, 8192, a, a, a, None) == 9
    # more than one token is not this entry point's job
    assert f(a, a, None, a, a, a, 2, 256, 8, 2, 256, a, a, a, None) == 1
