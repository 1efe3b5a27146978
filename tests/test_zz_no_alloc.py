"""coli_moe_forward_static: the layer for callers that cannot allocate.

Callers such as a plain C/FFI host with no device allocator of its own, or a
runtime that owns the whole device-memory budget and forbids cudaMalloc, get
the layer through this entry point, which uses the library's static 24 MiB
device scratch instead of a caller workspace.  These tests run it through the
C ABI several times in a row and compare its output with coli_moe_forward's
on a caller workspace.  Both run the same kernels on the same inputs, so the
outputs must agree bit for bit (tighter than the 1e-3 layer tolerance the
other GPU tests use against the oracle).  The calls cover the fused
single-position kernel (which keeps counters in the scratch between calls),
the few-position and small-batch kernels and the tensor-core path, in
interleaved order on one stream.  The file builds its own inputs, so it
passes in a fresh process as well as after the other tests (pytest collects
it last)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import synth  # noqa: E402
import quantized_expert_ffn_sigmoid_gb300 as cm  # noqa: E402


def _tiny_layer(shape, seed):
    recs, scs = zip(*[synth.expert_record(shape, seed, 0, "routed", e) for e in range(shape.n_experts)])
    srec, ssc = zip(*[synth.expert_record(shape, seed, 0, "shared", s) for s in range(shape.n_shared)])
    d = lambda a: torch.from_numpy(np.ascontiguousarray(np.stack(a))).cuda()
    t = [d(recs), d(scs), d(srec), d(ssc)]
    return t, cm.make_weights(*t)


def _glm_layer(shape, seed):
    import synth.gpu as sg
    recs, scs = sg.expert_records(shape, seed, 0, "routed", shape.n_experts, "cuda")
    srec, ssc = sg.expert_records(shape, seed, 0, "shared", shape.n_shared, "cuda")
    t = [recs, scs, srec, ssc]
    return t, cm.make_weights(*t)


def _routed(shape, cfg, seed, stream, T):
    x = torch.from_numpy(synth.token_batch(shape, seed, stream, range(T))).cuda()
    wr = torch.from_numpy(synth.router_weight(shape, seed)).cuda()
    bias = torch.from_numpy(synth.router_bias(shape, seed)).cuda()
    ws = cm.new_workspace(cfg, T)
    idx = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, shape.top_k), dtype=torch.float32, device="cuda")
    cm.coli_moe_route(cfg, x, wr, bias, idx, w, ws)
    assert cm.coli_moe_status(ws) == 0
    return x, idx, w


def _reference(cfg, W, x, idx, w):
    ws = cm.new_workspace(cfg, x.shape[0])
    y = torch.empty((x.shape[0], cfg.hidden), device="cuda")
    cm.coli_moe_forward(cfg, W, x, idx, w, y, ws)
    assert cm.coli_moe_status(ws) == 0
    return y


@pytest.mark.parametrize("T", [8, 33])
def test_static_scratch_matches_caller_workspace(T):
    shape = synth.TINY
    keep, W = _tiny_layer(shape, 31)
    cfg = cm.Cfg.of(shape)
    x, idx, w = _routed(shape, cfg, 31, "noalloc", T)
    ref = _reference(cfg, W, x, idx, w)
    for call in range(2):   # two calls in a row share (and must rewrite) the scratch
        y = torch.full((T, shape.hidden), float("nan"), device="cuda")
        cm.coli_moe_forward_static(cfg, W, x, idx, w, y)
        torch.cuda.synchronize()
        assert torch.equal(y, ref), f"call {call}"


def test_static_scratch_glm_interleaved_call_sizes():
    """GLM-5.2-shaped layer: one-position calls (the fused kernel, whose
    completion counters live in the scratch) back to back, then interleaved
    with 4-, 1-, 64- and 1-position calls on one stream; every output equal
    to coli_moe_forward's on a caller workspace."""
    shape = synth.GLM
    keep, W = _glm_layer(shape, 33)
    cfg = cm.Cfg.of(shape)
    cases = {T: _routed(shape, cfg, 33, ("noalloc", T), T) for T in (1, 4, 64)}
    refs = {T: _reference(cfg, W, *cases[T]) for T in cases}
    for n, T in enumerate((1, 1, 1, 4, 1, 64, 1, 4)):
        x, idx, w = cases[T]
        y = torch.full((T, shape.hidden), float("nan"), device="cuda")
        cm.coli_moe_forward_static(cfg, W, x, idx, w, y)
        torch.cuda.synchronize()
        assert torch.equal(y, refs[T]), f"call {n} (T={T})"


def test_static_scratch_rejects_too_many_positions():
    shape = synth.GLM
    cfg = cm.Cfg.of(shape)
    # 24 MiB holds the GLM-5.2-shaped layer's scratch up to 76 positions
    assert cm.coli_moe_workspace_size(cfg, 76) <= cm.STATIC_WS_BYTES < cm.coli_moe_workspace_size(cfg, 77)
    T = 77
    x = torch.zeros((T, shape.hidden), device="cuda")
    idx = torch.zeros((T, shape.top_k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, shape.top_k), device="cuda")
    y = torch.zeros((T, shape.hidden), device="cuda")
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    W = cm.make_weights(dummy, dummy, dummy, dummy)
    with pytest.raises(cm.ColiError) as e:
        cm.coli_moe_forward_static(cfg, W, x, idx, w, y)
    assert e.value.code == cm.COLI_EWORKSPACE
