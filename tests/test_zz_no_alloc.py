"""coli_moe_forward_static: the layer for callers that cannot allocate.

Callers such as a plain C/FFI host with no device allocator of its own, or a
runtime that owns the whole device-memory budget and forbids cudaMalloc, get
the layer through this entry point, which uses the library's static 24 MiB
device scratch instead of a caller workspace.  This test runs it through the
C ABI twice in a row and checks its output against coli_moe_forward's within
the layer tolerance used by the other GPU tests.  It builds its own inputs,
so it passes in a fresh process as well as after the other tests (pytest
collects this file last)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import synth  # noqa: E402
import quantized_expert_ffn_sigmoid_gb300 as cm  # noqa: E402
from helpers import normwise_err  # noqa: E402

Y_TOL = 1e-3


def _layer(shape, seed):
    recs, scs = zip(*[synth.expert_record(shape, seed, 0, "routed", e) for e in range(shape.n_experts)])
    srec, ssc = zip(*[synth.expert_record(shape, seed, 0, "shared", s) for s in range(shape.n_shared)])
    d = lambda a: torch.from_numpy(np.ascontiguousarray(np.stack(a))).cuda()
    t = [d(recs), d(scs), d(srec), d(ssc)]
    return t, cm.make_weights(*t)


@pytest.mark.parametrize("T", [8, 33])
def test_static_scratch_matches_caller_workspace(T):
    shape = synth.TINY
    keep, W = _layer(shape, 31)
    cfg = cm.Cfg.of(shape)
    x = torch.from_numpy(synth.token_batch(shape, 31, "noalloc", range(T))).cuda()
    wr = torch.from_numpy(synth.router_weight(shape, 31)).cuda()
    bias = torch.from_numpy(synth.router_bias(shape, 31)).cuda()
    ws = cm.new_workspace(cfg, T)
    idx = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, shape.top_k), dtype=torch.float32, device="cuda")
    cm.coli_moe_route(cfg, x, wr, bias, idx, w, ws)
    y_ref = torch.empty((T, shape.hidden), device="cuda")
    cm.coli_moe_forward(cfg, W, x, idx, w, y_ref, ws)
    assert cm.coli_moe_status(ws) == 0
    ref = y_ref.cpu().numpy()
    for call in range(2):   # two calls in a row share (and must rewrite) the scratch
        y = torch.full((T, shape.hidden), float("nan"), device="cuda")
        cm.coli_moe_forward_static(cfg, W, x, idx, w, y)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}"
        assert normwise_err(got, ref) <= Y_TOL, f"call {call}"


def test_static_scratch_rejects_too_many_positions():
    shape = synth.GLM
    cfg = cm.Cfg.of(shape)
    # 24 MiB holds the GLM-5.2-shaped layer's scratch up to 88 positions
    assert cm.coli_moe_workspace_size(cfg, 88) <= cm.STATIC_WS_BYTES < cm.coli_moe_workspace_size(cfg, 89)
    T = 89
    x = torch.zeros((T, shape.hidden), device="cuda")
    idx = torch.zeros((T, shape.top_k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, shape.top_k), device="cuda")
    y = torch.zeros((T, shape.hidden), device="cuda")
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    W = cm.make_weights(dummy, dummy, dummy, dummy)
    with pytest.raises(cm.ColiError) as e:
        cm.coli_moe_forward_static(cfg, W, x, idx, w, y)
    assert e.value.code == cm.COLI_EWORKSPACE
