"""Exact logit ties on every router path, against the oracle.

The selection rule is "the k largest, descending, equal values by lowest
expert index".  Ties are made exact by giving several experts the same row
of Wr: both the kernels and the oracle then compute bit-identical logits for
them (the same inputs summed in the same order), so the tie is real on both
sides and only the index rule can decide it.  Every other pair of the top
logits stays at least 1e-5 apart (rows of x are redrawn until it does).

Paths: the single-token fused kernel, the one/two-token row router (also in
front of the streamed single-token launches), the 3..255-token cluster
router (1, 2, 4 or 8 tokens per cluster tile), the tensor-core cluster
router (three-pass TF32, T >= 256, E <= 128) and the large-E router
(T >= 256, E > 128).  Expert indices must match the
oracle bit for bit, the weights within 1e-6, and y within the tolerance.
"""
import numpy as np
import pytest

from oracle.oracle import Oracle
from quantized_routed_expert_02_gb300 import synth
from tests.cases import GAP, W_TOL, exact_ties_only, tie_free_x, y_tolerance
from tests.test_gpu_parity import DEV, check_layer, m, run_layer  # noqa: F401

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def grouped_rows(Wr, pattern=(2, 1, 3, 1)):
    """Copy rows so the experts fall into groups of identical rows, the group
    sizes cycling through ``pattern``: {0,1}, {2}, {3,4,5}, {6}, {7,8}, ..."""
    Wr = Wr.copy()
    E = Wr.shape[0]
    e, i = 0, 0
    while e < E:
        g = pattern[i % len(pattern)]
        i += 1
        for d in range(e + 1, min(E, e + g)):
            Wr[d] = Wr[e]
        e += g
    return Wr


def order_of(lg):
    """Expert ids by (logit descending, index ascending)."""
    return np.lexsort((np.arange(lg.size), -lg))


def make_case(shape, layer, Wr, bias, accept_depth=2, blobs="all", o=None, x=None):
    """Inputs and oracle outputs for a given (tied) router matrix.  ``blobs``:
    "all", "selected" (only the routed experts' matrices; the others stay
    zero, which no correct kernel reads) or None (router only).  ``x``: use
    these activations (they must pass the tie rule) instead of drawing."""
    o = o or Oracle()

    def accept(row):
        return exact_ties_only(row, shape.k, GAP, accept_depth)

    if x is None:
        x, _ = tie_free_x(o, shape, layer, Wr, bias, accept=accept)
    r = o.router(x, Wr, bias, shape.k)
    assert all(accept(row) for row in r["logits"])
    case = dict(shape=shape, x=x, Wr=Wr, bias=bias, idx=r["idx"], w=r["w"],
                logits=r["logits"], tokens=None, blobs=None, y=None)
    if blobs is not None:
        experts = None if blobs == "all" else sorted(set(r["idx"].ravel().tolist()))
        case["blobs"] = synth.expert_blobs(shape, layer, experts=experts)
        y, _ = o.ffn(x, r["idx"], r["w"], case["blobs"]["gate"], case["blobs"]["up"],
                     case["blobs"]["down"], shape.E, shape.I)
        case["y"] = y
    return case


def tie_stats(case):
    """(tokens with a tie inside the selection, tokens with a tie across the
    k-1 / k boundary)."""
    k = case["shape"].k
    inside = across = 0
    for lg in case["logits"]:
        s = np.sort(lg)[::-1]
        inside += int(np.any(s[:k - 1] == s[1:k]))
        across += int(s[k - 1] == s[k])
    return inside, across


# ---------------------------------------------------------------- single token, fused kernel

def boundary_tie(shape, layer, lower, o):
    """Wr and x of a single token whose rank-0 row is duplicated (a tie at
    ranks 0 / 1, which moves every later logit down one rank) and whose
    rank-(k-2) row is duplicated into an expert below (lower=True) or above
    it in index, so that two experts tie across ranks k-1 / k.  Returns None
    when this layer's draw offers no such expert."""
    Wr = synth.router_weights(shape, layer)
    k = shape.k

    def deep(row):
        return exact_ties_only(row, k, GAP, 6)

    x, _ = tie_free_x(o, shape, layer, Wr, None, accept=deep)
    lg = o.router(x, Wr, None, k)["logits"][0]
    order = order_of(lg)
    src, top = order[k - 2], order[0]
    cands = [e for e in order[k + 3:] if (e < src) == lower and e != top]
    spare = [e for e in order[k + 3:] if e not in cands[:1]]
    if not cands or not spare:
        return None
    Wr2 = Wr.copy()
    Wr2[cands[0]] = Wr[src]      # tie across ranks k-1 / k
    Wr2[spare[0]] = Wr[top]      # tie at ranks 0 / 1
    lg2 = o.router(x, Wr2, None, k)["logits"][0]
    if not exact_ties_only(lg2, k, GAP, 2):
        return None
    return Wr2, x


@pytest.mark.parametrize("lower", [True, False], ids=["dup-below", "dup-above"])
def test_fused_single_token_boundary_tie(m, lower):
    shape = synth.SHAPES["a3b_decode"]
    assert m.moe_layer_launch_count(1, shape.H, shape.E, shape.k, shape.I) == 1
    o = Oracle()
    for layer in range(8):
        made = boundary_tie(shape, layer, lower, o)
        if made is not None:
            break
    assert made is not None
    case = make_case(shape, layer, made[0], None, blobs="selected", o=o, x=made[1])
    inside, across = tie_stats(case)
    assert inside == 1 and across == 1
    idx, w, y, _, _ = run_layer(m, case)
    check_layer(case, idx, w, y)


def test_fused_single_token_grouped_rows(m):
    shape = synth.SHAPES["a3b_decode"]
    o = Oracle()
    n_inside = 0
    for layer in range(3):
        Wr = grouped_rows(synth.router_weights(shape, layer))
        case = make_case(shape, layer, Wr, None, blobs="selected", o=o)
        n_inside += tie_stats(case)[0]
        idx, w, y, _, _ = run_layer(m, case)
        check_layer(case, idx, w, y)
    assert n_inside >= 1


# ---------------------------------------------------------------- single token, streamed launches

@pytest.mark.parametrize("lower", [True, False], ids=["dup-below", "dup-above"])
def test_streamed_single_token_boundary_tie(m, lower):
    shape = synth.custom_shape(1, 4096, 32, 8, 1536, wr_std=0.015, cfg_id=31, name="a22b_e32")
    assert m.moe_layer_launch_count(1, shape.H, shape.E, shape.k, shape.I) == 3
    o = Oracle()
    for layer in range(16):
        made = boundary_tie(shape, layer, lower, o)
        if made is not None:
            break
    assert made is not None
    case = make_case(shape, layer, made[0], None, blobs="selected", o=o, x=made[1])
    assert tie_stats(case) == (1, 1)
    idx, w, y, _, _ = run_layer(m, case)
    check_layer(case, idx, w, y)


# ---------------------------------------------------------------- router kernels alone

ROUTER_PATHS = [
    # T, H, E, k: which router kernel
    (1, 2048, 128, 8),     # one/two-token row kernel (top-k in its last CTA)
    (2, 2048, 128, 7),     # the same with two tokens, odd k
    (3, 2048, 128, 8),     # cluster router, one token per tile
    (32, 4096, 128, 8),    # two tokens per tile, 16 K chunks through an 11-slot ring
    (64, 2048, 128, 8),    # four tokens per tile, the batched-decode size
    (5, 8192, 16, 3),      # two experts per group, 32 K chunks through a 16-slot ring
    (200, 1024, 256, 8),   # eight tokens per tile, four experts per warp, two CTAs per SM
    (100, 512, 256, 32),   # k = 32: the rank count's largest selection, 64 sums per lane
    (300, 2048, 128, 8),   # tensor-core cluster kernel with the top-k fused
    (256, 1024, 256, 8),   # large-E kernel (E > 128) with the top-k fused
    (260, 512, 64, 1),     # tensor-core kernel, k = 1: a tie decides the arg-max
]


@pytest.mark.parametrize("T,H,E,k", ROUTER_PATHS,
                         ids=[f"T{t}-H{h}-E{e}-k{k}" for t, h, e, k in ROUTER_PATHS])
def test_router_ties(m, T, H, E, k):
    shape = synth.custom_shape(T, H, E, k, 256, wr_std=0.02, cfg_id=32 + (T + E + k) % 17,
                               name="ties")
    o = Oracle()
    pattern = (2,) if k == 1 else (2, 1, 3, 1)
    for layer in range(8):   # a draw whose tokens meet tied experts in their selection
        Wr = grouped_rows(synth.router_weights(shape, layer), pattern)
        case = make_case(shape, layer, Wr, None, blobs=None, o=o)
        inside, across = tie_stats(case)
        if (inside >= 1 or k == 1) and (across >= 1 or T < 64):
            break
    if k > 1:
        assert inside >= 1
    assert across >= 1 or T < 64
    x = torch.from_numpy(case["x"]).to(DEV)
    Wd = torch.from_numpy(Wr).to(DEV)
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    ws = m.alloc_workspace(T, H, E, k, 256, device=DEV)
    m.moe_router(x, Wd, None, k, idx, w, ws)
    assert m.moe_read_device_status(ws)[0] == 0
    np.testing.assert_array_equal(idx.cpu().numpy(), case["idx"])
    assert np.max(np.abs(w.cpu().numpy().astype(np.float64) - case["w"])) <= W_TOL


def test_router_ties_with_bias(m):
    """A bias that is equal within each group keeps the ties exact."""
    T, H, E, k = 64, 2048, 128, 8
    shape = synth.custom_shape(T, H, E, k, 256, wr_std=0.02, cfg_id=49, name="ties")
    pattern = (2, 1, 3, 1)
    Wr = grouped_rows(synth.router_weights(shape, 0), pattern)
    b = np.array([-1.6 * np.log(e + 1) for e in range(E)], dtype=np.float32)
    e, i = 0, 0
    while e < E:
        g = pattern[i % len(pattern)]
        i += 1
        b[e:e + g] = b[e]
        e += g
    case = make_case(shape, 0, Wr, b, blobs=None)
    assert tie_stats(case)[0] >= 1
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    ws = m.alloc_workspace(T, H, E, k, 256, device=DEV)
    m.moe_router(torch.from_numpy(case["x"]).to(DEV), torch.from_numpy(Wr).to(DEV),
                 torch.from_numpy(b).to(DEV), k, idx, w, ws)
    np.testing.assert_array_equal(idx.cpu().numpy(), case["idx"])
    assert np.max(np.abs(w.cpu().numpy().astype(np.float64) - case["w"])) <= W_TOL


# ---------------------------------------------------------------- whole layer on tied routing

LAYER_TIES = [
    (64, 2048, 128, 8, 768),   # tensor-core path (512 routed slots)
    (40, 512, 16, 4, 256),     # CUDA-core batched path (160 routed slots)
    (2, 1024, 16, 5, 512),     # two tokens: row router + CUDA-core path
]


@pytest.mark.parametrize("T,H,E,k,I", LAYER_TIES, ids=[f"T{t}" for t, *_ in LAYER_TIES])
def test_layer_on_tied_routing(m, T, H, E, k, I):
    shape = synth.custom_shape(T, H, E, k, I, wr_std=0.02, cfg_id=40 + T % 7, name="ties")
    Wr = grouped_rows(synth.router_weights(shape, 0))
    case = make_case(shape, 0, Wr, None, blobs="all")
    assert tie_stats(case)[0] >= 1
    idx, w, y, _, _ = run_layer(m, case)
    check_layer(case, idx, w, y)
    assert np.max(np.abs(y.astype(np.float64) - case["y"])) <= y_tolerance(case["y"])
