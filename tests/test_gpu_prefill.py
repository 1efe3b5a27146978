"""Calls with many positions take the tensor-core expert path (tcgen05 MMA on
fp16-widened integer codes, one TMEM accumulator per Q8_0 block).  Same
parity bar as every other path: routing, tables and Q8_0 codes bit-exact,
gate/up and down int32 block dots bit-exact (dumped by the same kernels),
outputs within the 1e-3 / elementwise bound."""
import dataclasses

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


@pytest.mark.parametrize("T", [64, 65, 130])
def test_tiny_many_positions(tiny, T):
    x, _, _ = margin_batch(tiny.shape, tiny.seed, ("pf", T), T, tiny.router_w, tiny.bias)
    st = check_parity(tiny, x, tiny.run(x))
    print("tiny T", T, st)


def test_tiny_int8_many_positions():
    shape = dataclasses.replace(synth.TINY, weight_bits=8)
    L = DeviceLayer(shape, 31)
    x, _, _ = margin_batch(shape, 31, "pf", 70, L.router_w, L.bias)
    check_parity(L, x, L.run(x))


@pytest.mark.parametrize("n_shared,shared_inter", [(0, 128), (2, 256), (1, 384)])
def test_shared_variants_many_positions(n_shared, shared_inter):
    shape = dataclasses.replace(synth.TINY, n_shared=n_shared, shared_inter=shared_inter)
    L = DeviceLayer(shape, 32)
    x, _, _ = margin_batch(shape, 32, "pf", 64, L.router_w, L.bias)
    check_parity(L, x, L.run(x))


def test_other_router_shapes_many_positions():
    shape = dataclasses.replace(synth.TINY, n_experts=64, n_groups=8, topk_group=3, top_k=6)
    L = DeviceLayer(shape, 33)
    x, _, _ = margin_batch(shape, 33, "pf", 96, L.router_w, L.bias)
    check_parity(L, x, L.run(x))
    one = dataclasses.replace(synth.TINY, n_groups=1, topk_group=1, top_k=16)  # every expert, 64+ pairs each
    L1 = DeviceLayer(one, 34)
    x1, _, _ = margin_batch(one, 34, "pf", 80, L1.router_w, L1.bias)
    check_parity(L1, x1, L1.run(x1))


def test_given_routing_with_duplicates_and_skips(tiny):
    T = 64
    x = synth.token_batch(tiny.shape, 35, 0, range(T))
    rng = np.random.default_rng(35)
    idx = rng.integers(0, tiny.shape.n_experts, size=(T, tiny.shape.top_k)).astype(np.int32)
    idx[::5, 1] = idx[::5, 0]      # duplicate experts within a position
    idx[::7, 2] = -1               # skipped slots
    w = rng.uniform(0.1, 1.0, size=idx.shape).astype(np.float32)
    g = tiny.run(x, route=False, idx=idx, w=w)
    check_parity(tiny, x, g, idx=idx, w=w.astype(np.float64))


def test_split_entry_points_equal_forward(tiny):
    T = 96
    x, _, _ = margin_batch(tiny.shape, tiny.seed, "pf-split", T, tiny.router_w, tiny.bias)
    xd = torch.from_numpy(x).cuda()
    k = tiny.shape.top_k
    ws = cm.new_workspace(tiny.cfg, T)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), device="cuda")
    cm.coli_moe_route(tiny.cfg, xd, tiny.wr_d, tiny.bias_d, idx, w, ws)
    y1 = torch.empty((T, tiny.shape.hidden), device="cuda")
    y2 = torch.empty_like(y1)
    y3 = torch.empty_like(y1)
    cm.coli_moe_forward(tiny.cfg, tiny.W, xd, idx, w, y1, ws)
    cm.coli_moe_dispatch(tiny.cfg, xd, idx, ws)
    cm.coli_moe_experts(tiny.cfg, tiny.W, T, w, y2, ws)
    cm.coli_moe_layer(tiny.cfg, tiny.W, xd, tiny.wr_d, tiny.bias_d, idx, w, y3, ws)
    assert cm.coli_moe_status(ws) == 0
    assert torch.equal(y1, y2) and torch.equal(y1, y3)


@pytest.mark.parametrize("T", [96, 200])
def test_tiny_mixed_per_expert_dispatch(tiny, T):
    """Around 24-50 pairs per routed expert: within one call some experts run on
    the tensor cores and the others on the small-batch kernels; every block
    dot, code and output checked."""
    x, _, _ = margin_batch(tiny.shape, tiny.seed, ("mixed", T), T, tiny.router_w, tiny.bias)
    g = tiny.run(x)
    counts = g["entry_count"][:-1]
    print("tiny mixed T", T, "pairs per routed entry", sorted(counts.tolist()))
    check_parity(tiny, x, g)


@pytest.mark.parametrize("T", [64, 128, 256, 512])
def test_glm_shaped_per_expert_dispatch(T):
    """GLM-5.2 row lengths with 64 routed experts at 64-512 positions (about
    8 to 64 pairs per expert): experts below the pair threshold stream through
    the small-batch kernels, the rest and the shared expert use the tensor
    cores; block dots dumped and compared bit for bit, sampled outputs."""
    shape = dataclasses.replace(synth.GLM, n_experts=64)
    seed = synth.WORKLOADS["glm_prefill_s2048"][1]
    L = DeviceLayer(shape, seed, device_weights=True, bias="zero")
    x, _, _ = margin_batch(shape, seed, ("mixed", T), T, L.router_w, L.bias)
    g = L.run(x, dump=T <= 128)
    st = check_parity(L, x, g, tokens=None if T <= 128 else [0, T // 2, T - 1])
    counts = g["entry_count"][:-1]
    print("glm-shaped mixed T", T, "pairs per expert min/max", counts.min(), counts.max(), st)
