"""coli_moe_layer: router and expert layer in one call (for one position, one
fused launch).  Checked against the oracle like the two-call path, bit-for-bit
against coli_moe_route + coli_moe_forward, and with outputs fed straight back
as the next call's inputs (the kernels of a call may start while the previous
call's last kernel is finishing, so this exercises the dependency waits)."""
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


@pytest.fixture(scope="module")
def tiny():
    return DeviceLayer(synth.TINY, synth.WORKLOADS["tiny_t8"][1])


@pytest.fixture(scope="module")
def glm():
    return DeviceLayer(synth.GLM, synth.WORKLOADS["glm_decode_b1"][1], device_weights=True)


def _same(a, b):
    for key in ("idx", "w", "y", "qx", "dx", "qh", "dh", "entry_expert", "entry_count", "entry_offset", "slot"):
        assert np.array_equal(a[key], b[key]), key


@pytest.mark.parametrize("T", [1, 2, 3, 8, 13])
def test_layer_tiny_parity(tiny, T):
    x, _, _ = margin_batch(tiny.shape, tiny.seed, ("layer", T), T, tiny.router_w, tiny.bias)
    g = tiny.run(x, layer=True)
    check_parity(tiny, x, g)
    _same(g, tiny.run(x, dump=False))


def test_layer_glm_decode(glm):
    ws = cm.new_workspace(glm.cfg, 1)
    for p in range(3):
        x, _, _ = margin_batch(glm.shape, glm.seed, "layer", 1, glm.router_w, glm.bias, start=p)
        g = glm.run(x, layer=True, ws=ws)
        st = check_parity(glm, x, g)
        _same(g, glm.run(x, dump=False, ws=ws))
        print("fused decode", p, st)


def _chain(layer, T, n, fused, sync):
    """n calls, each call's y the next call's x, on one workspace."""
    shape, dev = layer.shape, "cuda"
    ws = cm.new_workspace(layer.cfg, T)
    x0 = torch.from_numpy(synth.token_batch(shape, layer.seed, ("chain", T), range(T))).to(dev)
    bufs = [x0] + [torch.empty((T, shape.hidden), device=dev) for _ in range(n)]
    idx = [torch.empty((T, shape.top_k), dtype=torch.int32, device=dev) for _ in range(n)]
    w = [torch.empty((T, shape.top_k), device=dev) for _ in range(n)]
    torch.cuda.synchronize()
    for i in range(n):
        if fused:
            cm.coli_moe_layer(layer.cfg, layer.W, bufs[i], layer.wr_d, layer.bias_d, idx[i], w[i], bufs[i + 1], ws)
        else:
            cm.coli_moe_route(layer.cfg, bufs[i], layer.wr_d, layer.bias_d, idx[i], w[i], ws)
            cm.coli_moe_forward(layer.cfg, layer.W, bufs[i], idx[i], w[i], bufs[i + 1], ws)
        if sync:
            torch.cuda.synchronize()
    st = cm.coli_moe_status(ws)
    return st, [b.cpu().numpy() for b in bufs[1:]], [t.cpu().numpy() for t in idx]


@pytest.mark.parametrize("T,fused", [(1, True), (1, False), (3, True), (3, False)])
def test_outputs_feed_next_call_directly(glm, T, fused):
    st_a, ys_a, ids_a = _chain(glm, T, 6, fused, sync=False)
    st_b, ys_b, ids_b = _chain(glm, T, 6, fused, sync=True)
    assert st_a == 0 and st_b == 0
    for i in range(6):
        assert np.all(np.isfinite(ys_b[i]))
        assert np.array_equal(ids_a[i], ids_b[i]), f"call {i}: routing differs"
        assert np.array_equal(ys_a[i], ys_b[i]), f"call {i}: output differs"


def test_layer_nonfinite_input(tiny):
    x = synth.token_batch(tiny.shape, 11, 0, range(1))
    x[0, 3] = np.nan
    g = tiny.run(x, layer=True)
    assert g["status"] & cm.STATUS_NONFINITE
    assert np.all(g["idx"] == -1) and np.all(g["w"] == 0)
    # only the shared expert contributes, so y is finite
    assert np.all(np.isfinite(g["y"]))


def test_layer_argument_errors(tiny):
    x = torch.zeros((1, tiny.shape.hidden), device="cuda")
    idx = torch.empty((1, tiny.shape.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((1, tiny.shape.top_k), device="cuda")
    y = torch.empty_like(x)
    ws = cm.new_workspace(tiny.cfg, 1)
    with pytest.raises(cm.ColiError) as e:
        cm.coli_moe_layer(tiny.cfg, tiny.W, x, tiny.wr_d[:, 1:], tiny.bias_d, idx, w, y, ws)
    assert e.value.code == cm.COLI_EALIGN
    small = ws[:64]
    with pytest.raises(cm.ColiError) as e:
        cm.coli_moe_layer(tiny.cfg, tiny.W, x, tiny.wr_d, tiny.bias_d, idx, w, y, small)
    assert e.value.code in (cm.COLI_EINVAL, cm.COLI_EWORKSPACE)
