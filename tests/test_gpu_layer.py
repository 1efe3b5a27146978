"""GPU parity of the routed-MoE layer against the CPU oracle, through the C
ABI: routing indices, union tables, Q8_0 codes and int32 block dot products
bit-exact; requantised h exact wherever the oracle shows the code is unique;
outputs within 1e-3 (normwise per position)."""
import json
import os
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
from gpu_harness import DeviceLayer, check_parity  # noqa: E402
from helpers import margin_batch  # noqa: E402

GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def tiny():
    return DeviceLayer(synth.TINY, synth.WORKLOADS["tiny_t8"][1])


def test_generator_device_twin_matches_numpy():
    import synth.gpu as sg
    shape = synth.TINY
    recs, scs = sg.expert_records(shape, 5, 0, "routed", 3)
    for e in range(3):
        r, s = synth.expert_record(shape, 5, 0, "routed", e)
        assert np.array_equal(recs[e].cpu().numpy(), r)
        assert np.array_equal(scs[e].cpu().numpy(), s)
    key = synth.make_key(3, "x", 0, 11, 0)
    assert np.array_equal(sg.normal_f32(key, 6144, 1.0).cpu().numpy(), synth.normal_f32(key, 6144, 1.0))
    g8 = dataclasses.replace(shape, weight_bits=8)
    r8, s8 = sg.expert_records(g8, 5, 1, "shared", 1)
    rr, ss = synth.expert_record(g8, 5, 1, "shared", 0)
    assert np.array_equal(r8[0].cpu().numpy(), rr) and np.array_equal(s8[0].cpu().numpy(), ss)


def test_quantize_act_bit_exact():
    blocks = json.load(open(os.path.join(GOLD, "q8_0_blocks.json")))["blocks"]
    gold = np.array([b["x"] for b in blocks], np.float32).reshape(1, -1)
    rng = np.random.default_rng(0)
    rnd = (rng.standard_normal((37, 96 * 32)) * rng.uniform(1e-4, 1e4, (37, 1))).astype(np.float32)
    for x in (gold, rnd):
        xd = torch.from_numpy(x).cuda()
        q = torch.empty(x.shape, dtype=torch.int8, device="cuda")
        d = torch.empty((x.shape[0], x.shape[1] // 32), dtype=torch.float32, device="cuda")
        cm.coli_moe_quantize_act(xd, q, d)
        rq, rd = oracle.q8_0_quantize(x)
        assert np.array_equal(q.cpu().numpy(), rq)
        assert np.array_equal(d.cpu().numpy(), rd)


@pytest.mark.parametrize("T", [1, 3, 4, 5, 8, 13, 33])
def test_tiny_layer_parity(tiny, T):
    x, _, _ = margin_batch(tiny.shape, tiny.seed, ("tinyT", T), T, tiny.router_w, tiny.bias)
    g = tiny.run(x)
    check_parity(tiny, x, g)


def test_tiny_int8_weights():
    shape = dataclasses.replace(synth.TINY, weight_bits=8)
    L = DeviceLayer(shape, 21)
    x, _, _ = margin_batch(shape, 21, 0, 9, L.router_w, L.bias)
    check_parity(L, x, L.run(x))


@pytest.mark.parametrize("n_shared,shared_inter", [(0, 128), (2, 256), (1, 384)])
def test_shared_expert_variants(n_shared, shared_inter):
    shape = dataclasses.replace(synth.TINY, n_shared=n_shared, shared_inter=shared_inter)
    L = DeviceLayer(shape, 22)
    x, _, _ = margin_batch(shape, 22, 0, 6, L.router_w, L.bias)
    check_parity(L, x, L.run(x))


def test_other_router_shapes():
    shape = dataclasses.replace(synth.TINY, n_experts=64, n_groups=8, topk_group=3, top_k=6)
    L = DeviceLayer(shape, 23)
    x, _, _ = margin_batch(shape, 23, 0, 11, L.router_w, L.bias)
    check_parity(L, x, L.run(x))
    one = dataclasses.replace(synth.TINY, n_groups=1, topk_group=1, top_k=16)  # every expert
    L1 = DeviceLayer(one, 24)
    x1, _, _ = margin_batch(one, 24, 0, 5, L1.router_w, L1.bias)
    check_parity(L1, x1, L1.run(x1))


def test_forward_given_routing_edge_cases(tiny):
    x = synth.token_batch(tiny.shape, 7, 0, range(5))
    idx = np.array([[0, 3, 3, 7], [15, -1, 2, -1], [1, 2, 5, 6], [-1, -1, -1, -1], [4, 4, 4, 4]])
    w = np.array([[0.5, 0.25, 0.25, 0.0], [1.0, 9.0, 0.0, 9.0], [1.0, 0.0, 0.0, 0.0],
                  [0.0, 0.0, 0.0, 0.0], [0.1, 0.2, 0.3, 0.4]], np.float32)
    g = tiny.run(x, route=False, idx=idx, w=w)
    check_parity(tiny, x, g, idx=idx, w=w.astype(np.float64))


def test_bad_ids_and_nonfinite_set_status(tiny):
    x = synth.token_batch(tiny.shape, 8, 0, range(3))
    idx = np.array([[0, 1, 99, 2], [3, 4, 5, -5], [6, 7, 8, 9]])
    w = np.full((3, 4), 0.25, np.float32)
    g = tiny.run(x, route=False, idx=idx, w=w, dump=False)
    assert g["status"] == cm.STATUS_BADIDX
    xn = x.copy()
    xn[1, 17] = np.nan
    g = tiny.run(xn, dump=False)
    assert g["status"] & cm.STATUS_NONFINITE
    assert (g["idx"][1] == -1).all() and (g["w"][1] == 0).all()
    assert (g["idx"][[0, 2]] >= 0).all()


def test_abi_argument_errors(tiny):
    cfg = cm.Cfg.of(tiny.shape)
    x = torch.zeros((4, 256), device="cuda")
    idx = torch.zeros((4, 4), dtype=torch.int32, device="cuda")
    w = torch.zeros((4, 4), device="cuda")
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(cm.ColiError) as e:
        cm.coli_moe_route(cfg, x, tiny.wr_d, tiny.bias_d, idx, w, small)
    assert e.value.code == cm.COLI_EWORKSPACE
    ws = cm.new_workspace(cfg, 4)
    bad = cm.Cfg.of(tiny.shape)
    bad.topk_group = 5
    with pytest.raises(cm.ColiError) as e:
        cm.coli_moe_route(bad, x, tiny.wr_d, tiny.bias_d, idx, w, ws)
    assert e.value.code == cm.COLI_EINVAL
    xbig = torch.zeros(4 * 256 + 1, device="cuda")
    with pytest.raises(cm.ColiError) as e:
        cm.coli_moe_route(cfg, xbig[1:].view(4, 256), tiny.wr_d, tiny.bias_d, idx, w, ws)
    assert e.value.code == cm.COLI_EALIGN
    # empty input is a no-op
    cm.coli_moe_route(cfg, x[:0], tiny.wr_d, tiny.bias_d, idx, w, ws)
    assert cm.coli_moe_workspace_size(bad, 4) == 0
    assert cm.coli_moe_status(ws) == 0


def test_repeated_calls_reuse_workspace(tiny):
    ws = cm.new_workspace(tiny.cfg, 13)
    for T in (13, 2, 7):
        x, _, _ = margin_batch(tiny.shape, tiny.seed, ("reuse", T), T, tiny.router_w, tiny.bias)
        check_parity(tiny, x, tiny.run(x, ws=ws))


# --------------------------------------------------------------- GLM shapes
@pytest.fixture(scope="module")
def glm():
    return DeviceLayer(synth.GLM, synth.WORKLOADS["glm_decode_b1"][1], device_weights=True)


def test_glm_decode_b1(glm):
    """GLM-5.2 layer, one position per call (the decode workload), full check."""
    ws = cm.new_workspace(glm.cfg, 1)
    for p in range(3):
        x, _, _ = margin_batch(glm.shape, glm.seed, 0, 1, glm.router_w, glm.bias, start=p)
        st = check_parity(glm, x, glm.run(x, ws=ws))
        print("decode", p, st)


def test_glm_mtp_verify_t4():
    """4 positions per call with correlated consecutive positions."""
    shape = synth.GLM
    seed = synth.WORKLOADS["glm_mtp_verify_t4"][1]
    L = DeviceLayer(shape, seed, device_weights=True)
    for call in range(8):
        att = [0, 0, 0, 0]
        for p in range(4):
            while True:
                x = synth.mtp_chain(shape, seed, call, attempts=att)
                m = oracle.route_margins(oracle.router_logits(x[p:p + 1], L.router_w), L.bias, shape)[0]
                if m >= 1e-4:
                    break
                att[p] += 1
        g = L.run(x)
        st = check_parity(L, x, g)
        uniq = g["n_entries"] - shape.n_shared
        print("mtp call", call, "unique experts", uniq, st)
        assert uniq < 4 * shape.top_k  # positions share experts


def test_glm_prefill_s2048():
    """2048 positions: every routing index and table, and every position's
    output, requantised h codes and scales checked against the oracle."""
    shape = synth.GLM
    seed = synth.WORKLOADS["glm_prefill_s2048"][1]
    L = DeviceLayer(shape, seed, device_weights=True, bias="zero")
    x, _, rej = margin_batch(shape, seed, 0, 2048, L.router_w, L.bias)
    g = L.run(x, dump=False)
    st = check_parity(L, x, g)
    hit = g["n_entries"] - shape.n_shared
    print("prefill unique experts", hit, "rejected", rej, st)
    assert hit == shape.n_experts
    assert st["pairs"] == 2048 * (shape.top_k + shape.n_shared)


def test_glm_shaped_tensor_core_block_dots():
    """The tensor-core expert path at GLM-5.2 row lengths (hidden 6144,
    moe_inter 2048) with 16 routed experts and 128 positions, about 64 pairs
    per expert as in the 2048-position prefill: every int32 gate, up and down
    block dot product dumped and compared bit for bit."""
    shape = dataclasses.replace(synth.GLM, n_experts=16, n_groups=4, topk_group=2)
    seed = synth.WORKLOADS["glm_prefill_s2048"][1]
    L = DeviceLayer(shape, seed, device_weights=True, bias="zero")
    x, _, _ = margin_batch(shape, seed, "pf16", 128, L.router_w, L.bias)
    g = L.run(x, dump=True)
    st = check_parity(L, x, g)
    print("glm-shaped tensor-core dump", st)
    assert st["pairs"] == 128 * (shape.top_k + shape.n_shared)


@pytest.mark.parametrize("bits,layer", [(4, 0), (4, 23), (8, 24)])
def test_glm_stack_layers_b32(bits, layer):
    """Layers of the 24+1 stack at batch 32 with Zipf-skewed correction bias
    (int8 weights for the multi-token-prediction layer), every position checked."""
    shape = synth.GLM if bits == 4 else synth.GLM_INT8
    seed = synth.WORKLOADS["glm_stack24_mtp1_b32"][1]
    L = DeviceLayer(shape, seed, layer=layer, device_weights=True, bias="zipf")
    x = synth.stack_input(shape, seed, 0, layer)
    m = oracle.route_margins(oracle.router_logits(x, L.router_w), L.bias, shape)
    keep = np.flatnonzero(m >= 1e-4)
    x = np.ascontiguousarray(x[keep])
    g = L.run(x, dump=False)
    st = check_parity(L, x, g)
    counts = g["entry_count"][:-shape.n_shared]
    print("stack layer", layer, "positions", len(keep), "unique", counts.size, "max per expert",
          counts.max(), st)


def test_glm_stack_every_layer_step0():
    """Step 0 of the 24+1-layer stack at batch 32: every layer's routing
    indices and tables bit-exact for all positions with a routing margin, and
    one position's output per layer."""
    seed = synth.WORKLOADS["glm_stack24_mtp1_b32"][1]
    kept = []
    for layer in range(25):
        shape = synth.GLM_INT8 if layer == 24 else synth.GLM
        L = DeviceLayer(shape, seed, layer=layer, device_weights=True, bias="zipf")
        x = synth.stack_input(shape, seed, 0, layer)
        m = oracle.route_margins(oracle.router_logits(x, L.router_w), L.bias, shape)
        keep = np.flatnonzero(m >= 1e-4)
        xk = np.ascontiguousarray(x[keep])
        g = L.run(xk, layer=True)
        check_parity(L, xk, g, tokens=[layer % len(keep)])
        kept.append(len(keep))
        del L, g
        torch.cuda.empty_cache()
    print("stack step 0 positions with a margin per layer", kept)
    assert min(kept) >= 16


def test_single_position_edge_cases(tiny):
    """One position per call takes the fused single-position kernel: duplicate
    ids, skipped slots, bad ids and non-finite input behave as in the
    multi-position path."""
    x = synth.token_batch(tiny.shape, 9, 0, range(1))
    for idx_row, w_row in (([3, 3, -1, 7], [0.5, 0.25, 9.0, 0.25]), ([-1, -1, -1, -1], [0, 0, 0, 0]),
                           ([15, 0, 15, 15], [0.1, 0.2, 0.3, 0.4])):
        idx = np.array([idx_row])
        w = np.array([w_row], np.float32)
        g = tiny.run(x, route=False, idx=idx, w=w)
        check_parity(tiny, x, g, idx=idx, w=w.astype(np.float64))
    g = tiny.run(x, route=False, idx=np.array([[0, 99, 2, 3]]), w=np.full((1, 4), 0.25, np.float32), dump=False)
    assert g["status"] == cm.STATUS_BADIDX
    xn = x.copy()
    xn[0, 5] = np.inf
    g = tiny.run(xn, dump=False)
    assert g["status"] & cm.STATUS_NONFINITE


def test_dispatch_then_experts_equals_forward(glm):
    """The split entry points (dispatch, then experts) give the forward's output."""
    ws = cm.new_workspace(glm.cfg, 1)
    for p in range(2):
        x, _, _ = margin_batch(glm.shape, glm.seed, "split", 1, glm.router_w, glm.bias, start=p)
        xd = torch.from_numpy(x).cuda()
        idx = torch.empty((1, 8), dtype=torch.int32, device="cuda")
        w = torch.empty((1, 8), device="cuda")
        cm.coli_moe_route(glm.cfg, xd, glm.wr_d, glm.bias_d, idx, w, ws)
        y1 = torch.empty((1, glm.shape.hidden), device="cuda")
        y2 = torch.empty_like(y1)
        cm.coli_moe_forward(glm.cfg, glm.W, xd, idx, w, y1, ws)
        cm.coli_moe_dispatch(glm.cfg, xd, idx, ws)
        cm.coli_moe_experts(glm.cfg, glm.W, 1, w, y2, ws)
        assert cm.coli_moe_status(ws) == 0
        assert torch.equal(y1, y2)
