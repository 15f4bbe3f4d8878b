"""The allocation-free single-token entry point against the workspace one.

moe_layer_noalloc serves callers that cannot allocate device memory: it
runs the single-token kernel with the library's own fixed scratch array.
It must give the same routing and, within the tolerance the other tests
use, the same output as moe_layer, on two calls in a row (the second call
sees the first call's leftovers in the shared scratch).  Collected last so
that a failure here comes after every other test has run.
"""
import ctypes

import numpy as np
import pytest

from quantized_routed_expert_02_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _inputs(shape, layer, dev):
    blobs = synth.expert_blobs(shape, layer)
    return dict(
        x=torch.from_numpy(synth.activations_fast(shape, layer)).to(dev),
        Wr=torch.from_numpy(synth.router_weights(shape, layer)).to(dev),
        gate=torch.from_numpy(blobs["gate"]).to(dev),
        up=torch.from_numpy(blobs["up"]).to(dev),
        down=torch.from_numpy(blobs["down"]).to(dev),
    )


def test_noalloc_matches_workspace_entry_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_02_gb300 import build
    build.build()
    from quantized_routed_expert_02_gb300 import moeq4k as m

    dev = "cuda"
    s = synth.SHAPES["a3b_decode"]
    lib = ctypes.CDLL(m.LIB_PATH)
    f = lib.moe_layer_noalloc
    P, I_ = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, P, P, P, I_, I_, I_, I_, I_, P, P, P, P]
    f.restype = ctypes.c_int
    ws = m.alloc_workspace(1, s.H, s.E, s.k, s.I, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    for layer in (0, 1):   # two calls in a row through the same shared scratch
        d = _inputs(s, layer, dev)
        idx_r = torch.empty(1, s.k, dtype=torch.int32, device=dev)
        w_r = torch.empty(1, s.k, device=dev)
        y_r = torch.empty(1, s.H, device=dev)
        m.moe_layer(d["x"], d["Wr"], None, d["gate"], d["up"], d["down"], s.k, s.I,
                    idx_r, w_r, y_r, ws)
        idx_n = torch.full((1, s.k), -1, dtype=torch.int32, device=dev)
        w_n = torch.full((1, s.k), float("nan"), device=dev)
        y_n = torch.full((1, s.H), float("nan"), device=dev)
        rc = f(d["x"].data_ptr(), d["Wr"].data_ptr(), None, d["gate"].data_ptr(),
               d["up"].data_ptr(), d["down"].data_ptr(), 1, s.H, s.E, s.k, s.I,
               idx_n.data_ptr(), w_n.data_ptr(), y_n.data_ptr(), stream)
        assert rc == 0, m.status_str(rc)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(idx_n.cpu().numpy(), idx_r.cpu().numpy())
        assert np.max(np.abs(w_n.cpu().numpy() - w_r.cpu().numpy())) <= 1e-6
        yr = y_r.cpu().numpy().astype(np.float64)
        yn = y_n.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(yn))
        assert np.max(np.abs(yn - yr)) <= 2e-3 * np.max(np.abs(yr)) + 1e-5
    assert m.moe_read_device_status(ws)[0] == 0


def test_noalloc_rejects_oversize_and_batches():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_02_gb300 import moeq4k as m
    lib = ctypes.CDLL(m.LIB_PATH)
    f = lib.moe_layer_noalloc
    P, I_ = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, P, P, P, I_, I_, I_, I_, I_, P, P, P, P]
    f.restype = ctypes.c_int
    a = 1 << 20
    # k*I = 32*8192 values of h are beyond the fixed scratch
    assert f(a, a, None, a, a, a, 1, 256, 64, 32, 8192, a, a, a, None) == 9
    # more than one token is not this entry point's job
    assert f(a, a, None, a, a, a, 2, 256, 8, 2, 256, a, a, a, None) == 1
