"""Exact router ties on the GPU, checked bit for bit against the oracle.

The GLM-5.2 write-up ("Colibri (colibrì): GLM-5.2 local inference on 25 GB of
RAM", "How it works (validated core mechanics)") sends an exact tie to the
lower expert id; group ties follow the same rule.  Two constructions make
the ties exact on both sides:

* zero router rows with a bias on a 2^-10 grid: every affinity is 1/2 and
  every score and group sum is exact in fp32 (the selections are derived by
  hand in ``helpers.tie_design`` and pinned against the oracle on the CPU);
* duplicated router rows and bias for a whole group: the twin experts get
  bit-identical fp32 logits (the same instructions on the same operands),
  so their scores and their groups' scores tie exactly.

Each runs through the router entry point and through the whole layer, at
one position (the fused single-position kernel), a few positions, and 64+
positions (the tiled router and the tensor-core expert path)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
import quantized_expert_ffn_sigmoid_gb300 as cm  # noqa: E402
from gpu_harness import DeviceLayer, check_parity  # noqa: E402
from helpers import duplicate_group, route_margins_except_exact, tie_design  # noqa: E402


def _with_router(layer, wr, bias):
    layer.router_w = np.ascontiguousarray(wr, np.float32)
    layer.bias = np.ascontiguousarray(bias, np.float32)
    layer.wr_d = torch.from_numpy(layer.router_w).cuda()
    layer.bias_d = torch.from_numpy(layer.bias).cuda()
    return layer


def _route(layer, x):
    T, k = x.shape[0], layer.shape.top_k
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -7.0, device="cuda")
    ws = cm.new_workspace(layer.cfg, T)
    cm.coli_moe_route(layer.cfg, xd, layer.wr_d, layer.bias_d, idx, w, ws)
    assert cm.coli_moe_status(ws) == 0
    return idx.cpu().numpy(), w.cpu().numpy()


@pytest.fixture(scope="module")
def tiny_tie():
    shape = synth.TINY
    bias, expect = tie_design(shape)
    L = DeviceLayer(shape, synth.WORKLOADS["tiny_t8"][1])
    return _with_router(L, np.zeros((shape.n_experts, shape.hidden)), bias), expect


@pytest.fixture(scope="module")
def glm_tie():
    shape = synth.GLM
    bias, expect = tie_design(shape)
    L = DeviceLayer(shape, synth.WORKLOADS["glm_decode_b1"][1], device_weights=True)
    return _with_router(L, np.zeros((shape.n_experts, shape.hidden)), bias), expect


@pytest.mark.parametrize("T", [1, 3, 8, 9, 64, 96])
def test_designed_ties_router(tiny_tie, glm_tie, T):
    for L, expect in (tiny_tie, glm_tie):
        x = synth.token_batch(L.shape, 5, "ties", range(T))
        idx, w = _route(L, x)
        ridx, rw = oracle.route(oracle.router_logits(x, L.router_w), L.bias, L.shape)
        assert np.array_equal(idx, ridx)
        assert idx.tolist() == [expect] * T
        # every selected affinity is exactly 1/2: the weights are rsf / k exactly
        assert np.all(w == np.float32(L.shape.routed_scaling_factor / L.shape.top_k))


@pytest.mark.parametrize("T", [1, 4, 64])
def test_designed_ties_whole_layer_tiny(tiny_tie, T):
    L, expect = tiny_tie
    x = synth.token_batch(L.shape, 6, "ties-layer", range(T))
    g = L.run(x, layer=True)
    assert g["idx"].tolist() == [expect] * T
    check_parity(L, x, g)
    g = L.run(x)                     # route, then forward with the block-dot dump
    check_parity(L, x, g)


@pytest.mark.parametrize("T", [1, 64])
def test_designed_ties_whole_layer_glm(glm_tie, T):
    """GLM-5.2 shape: one position through the fused router-in-kernel path;
    64 positions that all pick the same 8 experts (64 pairs each) through the
    tiled router and the tensor-core expert path, every position checked."""
    L, expect = glm_tie
    x = synth.token_batch(L.shape, 7, "ties-layer", range(T))
    g = L.run(x, layer=True)
    assert g["idx"].tolist() == [expect] * T
    st = check_parity(L, x, g)
    print("glm ties", T, st)


@pytest.mark.parametrize("T", [1, 5, 33, 70])
def test_duplicated_group_ties_tiny(T):
    """Group 1's router rows and bias copied from group 0: each expert of
    group 1 ties exactly with its twin, and the two groups tie."""
    shape = synth.TINY
    L = DeviceLayer(shape, 41)
    wr, b = duplicate_group(L.router_w, L.bias, shape, 0, 1)
    _with_router(L, wr, b)
    xs = synth.token_batch(shape, 41, ("dup", T), range(4 * T + 16))
    m = route_margins_except_exact(oracle.router_logits(xs, wr), b, shape)
    x = np.ascontiguousarray(xs[m >= 1e-4][:T])
    assert x.shape[0] == T
    ridx, _ = oracle.route(oracle.router_logits(x, wr), b, shape)
    twins = sum(int(e < 4 and e + 4 in row) for row in ridx for e in row)
    idx, _ = _route(L, x)
    assert np.array_equal(idx, ridx)
    g = L.run(x, layer=True)
    check_parity(L, x, g)
    if T >= 33:
        assert twins > 0            # the tie decided some selections


@pytest.mark.parametrize("T", [1, 4, 64])
def test_duplicated_group_ties_glm(glm_tie, T):
    """GLM-5.2 router with group 6 a copy of group 2 (random positions)."""
    L0, _ = glm_tie
    shape = L0.shape
    wr, b = duplicate_group(synth.router_weight(shape, L0.seed), synth.router_bias(shape, L0.seed), shape, 2, 6)
    L = _with_router(L0, wr, b)
    try:
        xs = synth.token_batch(shape, 43, ("dup", T), range(2 * T + 8))
        m = route_margins_except_exact(oracle.router_logits(xs, wr), b, shape)
        x = np.ascontiguousarray(xs[m >= 1e-4][:T])
        assert x.shape[0] == T
        idx, _ = _route(L, x)
        ridx, _ = oracle.route(oracle.router_logits(x, wr), b, shape)
        assert np.array_equal(idx, ridx)
        g = L.run(x, layer=True)
        st = check_parity(L, x, g, tokens=None if T <= 4 else [0, T // 2, T - 1])
        print("glm duplicated group", T, st)
    finally:
        bias, _ = tie_design(shape)
        _with_router(L0, np.zeros((shape.n_experts, shape.hidden)), bias)
