"""coli_moe_stack_forward: a decode step through a stack of layers with the
hidden state kept on the device (JustVugg/colibri README, "Never wait for the
disk twice"), against the oracle.

The 24 + 1 layer stack at batch 32 (24 packed-int4 GLM-5.2-shaped layers and
one int8 layer, Zipf-skewed correction bias per layer, seeded residual adds
x_{l+1} = x_l + delta_l): every layer's input bit-exact against the seeded
recipe, every layer's routing bit-exact for the positions with a routing
margin, one position's output per layer within 1e-3; the step replayed from a
CUDA graph gives the same bits.  A small mixed-format stack checks the
variant that feeds each layer's output into the next input."""
import dataclasses

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
import quantized_expert_ffn_sigmoid_gb300 as cm  # noqa: E402
from gpu_harness import DeviceLayer  # noqa: E402
from helpers import normwise_err  # noqa: E402


def _run(layers, x0, residual, add_output):
    L0 = layers[0]
    n, T, H, k = len(layers), x0.shape[0], L0.shape.hidden, L0.shape.top_k
    arr = cm.stack_layers([(L.cfg, L.W, L.wr_d, L.bias_d) for L in layers])
    xs = torch.full((n + 1, T, H), float("nan"), device="cuda")
    xs[0] = torch.from_numpy(x0).cuda()
    res = None if residual is None else torch.from_numpy(np.ascontiguousarray(residual)).cuda()
    idx = torch.full((n, T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.zeros((n, T, k), device="cuda")
    y = torch.full((n, T, H), float("nan"), device="cuda")
    ws = cm.new_workspace(max((L.cfg for L in layers), key=lambda c: cm.coli_moe_workspace_size(c, T)), T)
    cm.coli_moe_stack_forward(arr, xs, res, idx, w, y, ws, add_output=add_output)
    assert cm.coli_moe_status(ws) == 0
    return arr, xs, res, idx, w, y, ws


def _check_layer(L, x, idx, w, y, positions):
    logits = oracle.router_logits(x, L.router_w)
    m = oracle.route_margins(logits, L.bias, L.shape)
    ridx, rw = oracle.route(logits, L.bias, L.shape)
    ok = m >= 1e-4
    assert np.array_equal(idx[ok], ridx[ok]), "routing indices differ"
    np.testing.assert_allclose(w[ok], rw[ok], rtol=1e-5, atol=1e-7)
    pos = [p for p in positions if ok[p]]
    ref = oracle.moe_forward(L.shape, L.get_record, x[pos], ridx[pos], rw[pos])["y"]
    assert normwise_err(y[pos], ref) <= 1e-3
    return int(ok.sum())


def test_glm_stack_step():
    seed = synth.WORKLOADS["glm_stack24_mtp1_b32"][1]
    layers = [DeviceLayer(synth.GLM_INT8 if l == 24 else synth.GLM, seed, layer=l, device_weights=True, bias="zipf")
              for l in range(25)]
    H = synth.GLM.hidden
    x0 = synth.stack_input(synth.GLM, seed, 0, 0)
    residual = np.stack([synth.residual_delta(synth.GLM, seed, 0, l)[:32 * H].reshape(32, H) for l in range(25)])
    arr, xs, res, idx, w, y, ws = _run(layers, x0, residual, False)
    xs_h, idx_h, w_h, y_h = xs.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()
    kept = []
    for l, L in enumerate(layers):
        assert np.array_equal(xs_h[l], synth.stack_input(L.shape, seed, 0, l)), f"layer {l} input"
        kept.append(_check_layer(L, xs_h[l], idx_h[l], w_h[l], y_h[l], [l % 32]))
    print("positions with a routing margin per layer", kept)
    assert min(kept) >= 16
    # the same step replayed from a CUDA graph: the same bits
    g = cm.capture_stack_step(arr, xs, res, idx, w, y, ws)
    y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert cm.coli_moe_status(ws) == 0
    assert np.array_equal(y.cpu().numpy(), y_h) and np.array_equal(idx.cpu().numpy(), idx_h)


@pytest.mark.parametrize("T", [1, 8, 70])
def test_mixed_stack_feeds_outputs_forward(T):
    """int4, int8, group-scaled int4 and packed int2 layers in one stack,
    each output added into the next layer's input on the device."""
    shapes = [synth.TINY, dataclasses.replace(synth.TINY, weight_bits=8), synth.TINY_GS64, synth.TINY_INT2]
    layers = [DeviceLayer(s, 60 + i, layer=i) for i, s in enumerate(shapes)]
    x0 = synth.token_batch(synth.TINY, 60, "mixed", range(T))
    residual = np.stack([synth.normal_f32(synth.make_key(60, "mixed-res", l), T * 256, 0.1).reshape(T, 256)
                         for l in range(len(layers))])
    _, xs, _, idx, w, y, _ = _run(layers, x0, residual, True)
    xs_h, idx_h, w_h, y_h = xs.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()
    for l, L in enumerate(layers):
        # the device's own chain: (x + y) + delta in fp32
        assert np.array_equal(xs_h[l + 1], (xs_h[l] + y_h[l]) + residual[l])
        _check_layer(L, xs_h[l], idx_h[l], w_h[l], y_h[l], list(range(T)))


def test_stack_argument_errors():
    L = DeviceLayer(synth.TINY, 61)
    other = DeviceLayer(dataclasses.replace(synth.TINY, hidden=512), 62)
    arr = cm.stack_layers([(L.cfg, L.W, L.wr_d, L.bias_d), (other.cfg, other.W, other.wr_d, other.bias_d)])
    xs = torch.zeros((3, 4, 256), device="cuda")
    idx = torch.zeros((2, 4, 4), dtype=torch.int32, device="cuda")
    w = torch.zeros((2, 4, 4), device="cuda")
    y = torch.zeros((2, 4, 256), device="cuda")
    ws = cm.new_workspace(L.cfg, 4)
    with pytest.raises(cm.ColiError) as e:   # hidden differs between layers
        cm.coli_moe_stack_forward(arr, xs, None, idx, w, y, ws)
    assert e.value.code == cm.COLI_EINVAL
    one = cm.stack_layers([(L.cfg, L.W, L.wr_d, L.bias_d)])
    small = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    cm.coli_moe_workspace_init(small)
    with pytest.raises(cm.ColiError) as e:
        cm.coli_moe_stack_forward(one, xs[:2], None, idx[:1], w[:1], y[:1], small)
    assert e.value.code == cm.COLI_EWORKSPACE
