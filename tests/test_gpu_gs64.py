"""GPU parity of group-scaled int4 weights ("gs64": one fp32 scale per 64
weights of a row) against the CPU oracle, through the C ABI: routing, tables,
Q8_0 codes and int32 block dots bit-exact, requantised h exact where unique,
outputs within 1e-3."""
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


def test_generator_device_twin_gs64():
    import synth.gpu as sg
    shape = synth.TINY_GS64
    recs, scs = sg.expert_records(shape, 7, 0, "routed", 3)
    srec, ssc = sg.expert_records(shape, 7, 0, "shared", 1)
    for e in range(3):
        r, s = synth.expert_record(shape, 7, 0, "routed", e)
        assert np.array_equal(recs[e].cpu().numpy(), r)
        assert np.array_equal(scs[e].cpu().numpy(), s)
    r, s = synth.expert_record(shape, 7, 0, "shared", 0)
    assert np.array_equal(srec[0].cpu().numpy(), r) and np.array_equal(ssc[0].cpu().numpy(), s)


@pytest.fixture(scope="module")
def tiny_gs():
    return DeviceLayer(synth.TINY_GS64, 8)


@pytest.mark.parametrize("T", [1, 3, 4, 5, 8, 13, 33, 70])
def test_tiny_gs64_parity(tiny_gs, T):
    x, _, _ = margin_batch(tiny_gs.shape, tiny_gs.seed, ("gs64", T), T, tiny_gs.router_w, tiny_gs.bias)
    check_parity(tiny_gs, x, tiny_gs.run(x))


@pytest.mark.parametrize("T", [1, 3])
def test_tiny_gs64_layer_call(tiny_gs, T):
    # router and experts in one coli_moe_layer call (one fused launch at T = 1)
    # give the split calls' results
    x, _, _ = margin_batch(tiny_gs.shape, tiny_gs.seed, ("gs64layer", T), T, tiny_gs.router_w, tiny_gs.bias)
    g = tiny_gs.run(x, layer=True)
    check_parity(tiny_gs, x, g)
    assert np.array_equal(g["y"], tiny_gs.run(x, dump=False)["y"])


def test_group_size_validated(tiny_gs):
    import dataclasses
    bad = cm.Cfg.of(dataclasses.replace(tiny_gs.shape, group_size=32))
    assert cm.coli_moe_workspace_size(bad, 4) == 0


@pytest.fixture(scope="module")
def glm_gs():
    return DeviceLayer(synth.GLM_GS64, 9, device_weights=True)


@pytest.mark.parametrize("T", [1, 4])
def test_glm_gs64_parity(glm_gs, T):
    """GLM-5.2-shaped layer with group-scaled experts: decode and MTP-verify sizes."""
    x, _, _ = margin_batch(glm_gs.shape, glm_gs.seed, ("glm_gs64", T), T, glm_gs.router_w, glm_gs.bias)
    st = check_parity(glm_gs, x, glm_gs.run(x))
    print("gs64 T", T, st)


@pytest.mark.parametrize("T", [32, 70])
def test_glm_gs64_small_batch(glm_gs, T):
    """Group-scaled int4 on the small-batch kernels (every row's group scales
    of a K chunk staged beside its weights), also beyond the tensor-core
    path's lower bound (that path takes per-row scales only)."""
    x, _, _ = margin_batch(glm_gs.shape, glm_gs.seed, ("glm_gs64_sb", T), T, glm_gs.router_w, glm_gs.bias)
    st = check_parity(glm_gs, x, glm_gs.run(x, dump=False))
    print("gs64 small batch T", T, st)


@pytest.mark.parametrize("T", [2, 4, 9, 40])
def test_gs64_small_batch_block_dots(T):
    """A small layer whose K lengths (256) let the small-batch kernels take
    group scales: every int32 gate, up and down block dot dumped and compared
    bit for bit, outputs within 1e-3; a shared expert of another size."""
    import dataclasses
    shape = dataclasses.replace(synth.TINY_GS64, inter=256, shared_inter=512)
    L = DeviceLayer(shape, 12)
    x, _, _ = margin_batch(shape, 12, ("gs64sb", T), T, L.router_w, L.bias)
    check_parity(L, x, L.run(x))


def test_glm_gs64_fused_decode(glm_gs):
    """One fused launch per position (router inside) on group-scaled experts."""
    ws = cm.new_workspace(glm_gs.cfg, 1)
    for p in range(2):
        x, _, _ = margin_batch(glm_gs.shape, glm_gs.seed, "glm_gs64_layer", 1, glm_gs.router_w, glm_gs.bias,
                               start=p)
        g = glm_gs.run(x, layer=True, ws=ws)
        check_parity(glm_gs, x, g)
        assert np.array_equal(g["y"], glm_gs.run(x, dump=False, ws=ws)["y"])


def test_gs64_given_routing_edge_cases(tiny_gs):
    """Duplicate ids, skipped slots and an all-skipped position, at several
    positions per call and at one (the single-position kernel)."""
    x = synth.token_batch(tiny_gs.shape, 17, 0, range(5))
    idx = np.array([[0, 3, 3, 7], [15, -1, 2, -1], [1, 2, 5, 6], [-1, -1, -1, -1], [4, 4, 4, 4]])
    w = np.array([[0.5, 0.25, 0.25, 0.0], [1.0, 9.0, 0.0, 9.0], [1.0, 0.0, 0.0, 0.0],
                  [0.0, 0.0, 0.0, 0.0], [0.1, 0.2, 0.3, 0.4]], np.float32)
    g = tiny_gs.run(x, route=False, idx=idx, w=w)
    check_parity(tiny_gs, x, g, idx=idx, w=w.astype(np.float64))
    for p in (0, 3, 4):
        g1 = tiny_gs.run(x[p:p + 1], route=False, idx=idx[p:p + 1], w=w[p:p + 1])
        check_parity(tiny_gs, x[p:p + 1], g1, idx=idx[p:p + 1], w=w[p:p + 1].astype(np.float64))


@pytest.mark.parametrize("n_shared,shared_inter", [(0, 128), (2, 256)])
def test_gs64_shared_expert_variants(n_shared, shared_inter):
    import dataclasses
    shape = dataclasses.replace(synth.TINY_GS64, n_shared=n_shared, shared_inter=shared_inter)
    L = DeviceLayer(shape, 27)
    for T in (1, 6):
        x, _, _ = margin_batch(shape, 27, ("gs64sh", T), T, L.router_w, L.bias)
        check_parity(L, x, L.run(x))


def test_gs64_nonfinite_and_empty(tiny_gs):
    x = synth.token_batch(tiny_gs.shape, 18, 0, range(2))
    xn = x.copy()
    xn[1, 9] = np.nan
    g = tiny_gs.run(xn, dump=False)
    assert g["status"] & cm.STATUS_NONFINITE
    assert (g["idx"][1] == -1).all() and (g["w"][1] == 0).all()
    ws = cm.new_workspace(tiny_gs.cfg, 2)
    xd = torch.zeros((0, tiny_gs.shape.hidden), device="cuda")
    idx = torch.zeros((0, tiny_gs.shape.top_k), dtype=torch.int32, device="cuda")
    w = torch.zeros((0, tiny_gs.shape.top_k), device="cuda")
    y = torch.zeros((0, tiny_gs.shape.hidden), device="cuda")
    cm.coli_moe_layer(tiny_gs.cfg, tiny_gs.W, xd, tiny_gs.wr_d, tiny_gs.bias_d, idx, w, y, ws)
    assert cm.coli_moe_status(ws) == 0
