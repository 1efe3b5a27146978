"""GPU parity of packed int2 weights (four codes per byte, per-row fp32
scales) against the CPU oracle, through the C ABI: routing, tables, Q8_0
codes and int32 block dots bit-exact, requantised h exact where unique,
outputs within 1e-3.  One position per call runs the fused single-position
kernel, two to four the few-position (GEMV) kernels, more the general expert
kernel."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import synth  # noqa: E402
import quantized_expert_ffn_sigmoid_gb300 as cm  # noqa: E402
from gpu_harness import DeviceLayer, check_parity  # noqa: E402
from helpers import margin_batch  # noqa: E402


def test_generator_device_twin_int2():
    import synth.gpu as sg
    shape = synth.TINY_INT2
    recs, scs = sg.expert_records(shape, 7, 0, "routed", 3)
    srec, ssc = sg.expert_records(shape, 7, 0, "shared", 1)
    for e in range(3):
        r, s = synth.expert_record(shape, 7, 0, "routed", e)
        assert np.array_equal(recs[e].cpu().numpy(), r)
        assert np.array_equal(scs[e].cpu().numpy(), s)
    r, s = synth.expert_record(shape, 7, 0, "shared", 0)
    assert np.array_equal(srec[0].cpu().numpy(), r) and np.array_equal(ssc[0].cpu().numpy(), s)


@pytest.fixture(scope="module")
def tiny2():
    return DeviceLayer(synth.TINY_INT2, 10)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 13, 33, 70])
def test_tiny_int2_parity(tiny2, T):
    x, _, _ = margin_batch(tiny2.shape, tiny2.seed, ("int2", T), T, tiny2.router_w, tiny2.bias)
    check_parity(tiny2, x, tiny2.run(x))


@pytest.mark.parametrize("T", [1, 3])
def test_tiny_int2_layer_call(tiny2, T):
    # router and experts in one coli_moe_layer call give the split calls' results
    x, _, _ = margin_batch(tiny2.shape, tiny2.seed, ("int2layer", T), T, tiny2.router_w, tiny2.bias)
    g = tiny2.run(x, layer=True)
    check_parity(tiny2, x, g)
    assert np.array_equal(g["y"], tiny2.run(x, dump=False)["y"])


def test_int2_given_routing_edge_cases(tiny2):
    """Duplicate ids, skipped slots and an all-skipped position, at five
    positions per call (general kernel), four (few-position kernels) and one
    (single-position kernel)."""
    x = synth.token_batch(tiny2.shape, 19, 0, range(5))
    idx = np.array([[0, 3, 3, 7], [15, -1, 2, -1], [1, 2, 5, 6], [-1, -1, -1, -1], [4, 4, 4, 4]])
    w = np.array([[0.5, 0.25, 0.25, 0.0], [1.0, 9.0, 0.0, 9.0], [1.0, 0.0, 0.0, 0.0],
                  [0.0, 0.0, 0.0, 0.0], [0.1, 0.2, 0.3, 0.4]], np.float32)
    g = tiny2.run(x, route=False, idx=idx, w=w)
    check_parity(tiny2, x, g, idx=idx, w=w.astype(np.float64))
    g4 = tiny2.run(x[:4], route=False, idx=idx[:4], w=w[:4])
    check_parity(tiny2, x[:4], g4, idx=idx[:4], w=w[:4].astype(np.float64))
    for p in (0, 3, 4):
        g1 = tiny2.run(x[p:p + 1], route=False, idx=idx[p:p + 1], w=w[p:p + 1])
        check_parity(tiny2, x[p:p + 1], g1, idx=idx[p:p + 1], w=w[p:p + 1].astype(np.float64))


@pytest.mark.parametrize("n_shared,shared_inter", [(0, 128), (2, 256)])
def test_int2_shared_expert_variants(n_shared, shared_inter):
    import dataclasses
    shape = dataclasses.replace(synth.TINY_INT2, n_shared=n_shared, shared_inter=shared_inter)
    L = DeviceLayer(shape, 29)
    for T in (1, 6):
        x, _, _ = margin_batch(shape, 29, ("int2sh", T), T, L.router_w, L.bias)
        check_parity(L, x, L.run(x))


def test_int2_nonfinite_and_group_scales_rejected(tiny2):
    import dataclasses
    x = synth.token_batch(tiny2.shape, 20, 0, range(2))
    x[1, 9] = np.inf
    g = tiny2.run(x, dump=False)
    assert g["status"] & cm.STATUS_NONFINITE
    assert (g["idx"][1] == -1).all() and (g["w"][1] == 0).all()
    bad = cm.Cfg.of(dataclasses.replace(tiny2.shape, group_size=64))
    assert cm.coli_moe_workspace_size(bad, 4) == 0


@pytest.fixture(scope="module")
def glm2():
    return DeviceLayer(synth.GLM_INT2, 11, device_weights=True)


@pytest.mark.parametrize("T", [1, 4])
def test_glm_int2_parity(glm2, T):
    """GLM-5.2-shaped layer with packed int2 experts: decode and MTP-verify sizes."""
    x, _, _ = margin_batch(glm2.shape, glm2.seed, ("glm_int2", T), T, glm2.router_w, glm2.bias)
    st = check_parity(glm2, x, glm2.run(x))
    print("int2 T", T, st)


@pytest.mark.parametrize("T", [32, 70])
def test_glm_int2_small_batch(glm2, T):
    """Packed int2 on the small-batch kernels (more than four positions, also
    beyond the tensor-core path's lower bound, which takes int4 and int8
    only): every table, code and output against the oracle."""
    x, _, _ = margin_batch(glm2.shape, glm2.seed, ("glm_int2_sb", T), T, glm2.router_w, glm2.bias)
    st = check_parity(glm2, x, glm2.run(x, dump=False))
    print("int2 small batch T", T, st)


def test_glm_int2_fused_decode(glm2):
    """One fused launch per position (router inside) on packed int2 experts,
    two calls in a row on one workspace; the split calls give the same y."""
    ws = cm.new_workspace(glm2.cfg, 1)
    for p in range(2):
        x, _, _ = margin_batch(glm2.shape, glm2.seed, "glm_int2_layer", 1, glm2.router_w, glm2.bias, start=p)
        g = glm2.run(x, layer=True, ws=ws)
        check_parity(glm2, x, g)
        assert np.array_equal(g["y"], glm2.run(x, dump=False, ws=ws)["y"])
