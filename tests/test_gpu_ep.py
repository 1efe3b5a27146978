"""Expert-parallel shards of the layer on one GPU, against the oracle.

Shard r of P holds the routed experts e with e mod P == r (local record
e / P) and, on shard 0, the shared experts (colibrì v1.0 README,
"Experimental resident CUDA backend": experts placed whole per device).  Each
shard's call is checked like any other layer call -- tables bit-exact against
the oracle's for the routing with other shards' experts skipped, block dots,
h codes, output -- and the sum of the P shard outputs against the oracle's
whole layer.  All shards run here one after another on the one GPU; the
multi-device exchange (one all-reduce of y per call) is covered on the CPU
with gloo ranks and is not measured on hardware."""
import dataclasses
from types import SimpleNamespace

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
import quantized_expert_ffn_sigmoid_gb300 as cm  # noqa: E402
from quantized_expert_ffn_sigmoid_gb300 import ep  # noqa: E402
from gpu_harness import DeviceLayer, check_parity  # noqa: E402
from helpers import margin_batch, normwise_err  # noqa: E402


def _shard_view(L, r, P):
    """The oracle's view of shard r: same records by global id, shared
    experts only on shard 0."""
    shape = dataclasses.replace(L.shape, n_shared=L.shape.n_shared if r == 0 else 0)
    return SimpleNamespace(shape=shape, router_w=L.router_w, bias=L.bias, get_record=L.get_record)


def _mask(idx, E, r, P):
    own = np.zeros(E, bool)
    own[ep.owned_experts(E, r, P)] = True
    return np.where((idx >= 0) & own[np.clip(idx, 0, E - 1)], idx, -1)


def run_shards(L, x, P, layer_call=True, dump=False, tokens=None):
    """Every shard's call, each checked; returns the sum of their outputs."""
    E = L.shape.n_experts
    ridx, rw = oracle.route(oracle.router_logits(x, L.router_w), L.bias, L.shape)
    total = np.zeros((x.shape[0], L.shape.hidden))
    for r in range(P):
        parts = ep.shard_weights(L.recs, L.scs, L.srec, L.ssc, r, P)
        W = cm.make_weights(*parts)
        view = _shard_view(L, r, P)
        cfg = cm.Cfg.of(L.shape, r, P)
        if layer_call:
            g = L.run(x, layer=True, cfg=cfg, W=W, shape=view.shape)
            assert np.array_equal(g["idx"], ridx), "every shard routes the whole layer"
        else:
            g = L.run(x, route=False, idx=ridx, w=rw.astype(np.float32), dump=dump, cfg=cfg, W=W,
                      shape=view.shape)
        check_parity(view, x, g, idx=_mask(ridx, E, r, P), w=rw, tokens=tokens)
        total += g["y"]
        del parts, W
    sel = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    ref = oracle.moe_forward(L.shape, L.get_record, x[sel], ridx[sel], rw[sel])["y"]
    err = normwise_err(total[sel], ref)
    assert err <= 1e-3, f"sum over {P} shards: {err:.3e}"
    return err


@pytest.fixture(scope="module")
def tiny():
    return DeviceLayer(synth.TINY, synth.WORKLOADS["tiny_t8"][1])


@pytest.mark.parametrize("P", [2, 4])
@pytest.mark.parametrize("T", [1, 3, 8, 33, 70])
def test_tiny_shards(tiny, P, T):
    x, _, _ = margin_batch(tiny.shape, tiny.seed, ("ep", T), T, tiny.router_w, tiny.bias)
    run_shards(tiny, x, P)
    run_shards(tiny, x, P, layer_call=False, dump=True)


@pytest.mark.parametrize("shape", [synth.TINY_GS64, synth.TINY_INT2, dataclasses.replace(synth.TINY, weight_bits=8)],
                         ids=["gs64", "int2", "int8"])
@pytest.mark.parametrize("T", [1, 4, 9])
def test_tiny_shards_other_formats(shape, T):
    L = DeviceLayer(shape, 51)
    x, _, _ = margin_batch(shape, 51, ("ep", T), T, L.router_w, L.bias)
    run_shards(L, x, 2, layer_call=False, dump=True)


@pytest.mark.parametrize("shape", [synth.TINY, synth.TINY_GS64, synth.TINY_INT2], ids=["int4", "gs64", "int2"])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_shard_without_experts_outputs_zero(shape, T):
    """A shard that owns none of the call's experts and no shared expert
    computes y = 0 (every routed id here is a multiple of 4: shard 1 of 4
    owns none of them)."""
    L = DeviceLayer(shape, 52)
    x = synth.token_batch(shape, 52, "ep0", range(T))
    idx = np.tile(np.array([[0, 4, 8, 12]]), (T, 1))
    w = np.full((T, 4), 0.5, np.float32)
    parts = ep.shard_weights(L.recs, L.scs, L.srec, L.ssc, 1, 4)
    g = L.run(x, route=False, idx=idx, w=w, dump=False, cfg=cm.Cfg.of(shape, 1, 4), W=cm.make_weights(*parts),
              shape=dataclasses.replace(shape, n_shared=0))
    assert g["status"] == 0 and g["n_entries"] == 0
    assert np.all(g["y"] == 0.0)


@pytest.fixture(scope="module")
def glm():
    return DeviceLayer(synth.GLM, synth.WORKLOADS["glm_decode_b1"][1], device_weights=True)


@pytest.mark.parametrize("T,P", [(1, 2), (1, 8), (4, 2), (32, 4), (64, 4)])
def test_glm_shards(glm, T, P):
    x, _, _ = margin_batch(glm.shape, glm.seed, ("ep", T), T, glm.router_w, glm.bias)
    err = run_shards(glm, x, P, tokens=None if T <= 4 else [0, T - 1])
    print("glm shards", T, P, err)
