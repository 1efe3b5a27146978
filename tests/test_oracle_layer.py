"""Pins for the oracle's union tables and the whole layer (hand-worked tables,
the combine invariant against a dense every-expert evaluation)."""
from types import SimpleNamespace

import numpy as np

import oracle
import synth


def test_union_tables_hand_worked():
    idx = np.array([[3, 1], [1, 5], [5, 3]])
    t = oracle.union_tables(idx, 8, 1)
    assert t["uniq"].tolist() == [1, 3, 5]
    assert t["counts"].tolist() == [2, 2, 2, 3]
    assert t["offsets"].tolist() == [0, 2, 4, 6, 9]
    assert t["pair_token"].tolist() == [0, 1, 0, 2, 1, 2, 0, 1, 2]
    assert t["pair_j"].tolist() == [1, 0, 0, 1, 1, 0, -1, -1, -1]
    assert t["slot"].tolist() == [[2, 0], [1, 4], [5, 3]]


def test_union_tables_invalid_and_duplicate_ids():
    idx = np.array([[2, 2], [-1, 9]])
    t = oracle.union_tables(idx, 8, 0)
    assert t["uniq"].tolist() == [2]
    assert t["slot"].tolist() == [[0, 1], [-1, -1]]


def _dense_gates(idx, w, E):
    gd = np.zeros((idx.shape[0], E))
    for t in range(idx.shape[0]):
        for j in range(idx.shape[1]):
            gd[t, idx[t, j]] += w[t, j]
    return gd


def test_combine_equals_dense_every_expert(tiny_layer):
    L = tiny_layer
    shape = L["shape"]
    x = synth.token_batch(shape, L["seed"], 0, range(8))
    out = oracle.moe_layer(shape, L["get_record"], x, L["router_w"], L["bias"])
    dense = oracle.dense_reference(shape, L["get_record"], x, _dense_gates(out["idx"], out["w"], 16))
    assert np.allclose(out["y"], dense, rtol=1e-12, atol=1e-14 * np.abs(dense).max())
    assert np.allclose(out["w"].sum(1), 2.5)


def test_all_experts_selected_is_dense_weighted_sum(tiny_layer):
    L = tiny_layer
    shape = L["shape"]
    full = SimpleNamespace(**{**shape.__dict__, "n_groups": 1, "topk_group": 1, "top_k": 16})
    x = synth.token_batch(shape, L["seed"], 5, range(3))
    logits = oracle.router_logits(x, L["router_w"])
    idx, w = oracle.route(logits, L["bias"], full)
    s = oracle.sigmoid(logits)
    gd = s / s.sum(1, keepdims=True) * 2.5   # every expert, weights from all affinities
    out = oracle.moe_forward(shape, L["get_record"], x, idx, w)
    dense = oracle.dense_reference(shape, L["get_record"], x, gd)
    assert np.allclose(out["y"], dense, rtol=1e-12, atol=1e-14 * np.abs(dense).max())


def test_zero_weight_and_duplicate_slots(tiny_layer):
    L = tiny_layer
    shape = L["shape"]
    x = synth.token_batch(shape, L["seed"], 6, range(2))
    idx = np.array([[0, 3, 3, 7], [1, 2, 5, 6]])
    w = np.array([[0.5, 0.25, 0.25, 0.0], [1.0, 0.0, 0.0, 0.0]])
    out = oracle.moe_forward(shape, L["get_record"], x, idx, w)
    idx2 = np.array([[0, 3, 7, 7], [1, 2, 5, 6]])
    w2 = np.array([[0.5, 0.5, 0.0, 0.0], [1.0, 0.0, 0.0, 0.0]])
    out2 = oracle.moe_forward(shape, L["get_record"], x, idx2, w2)
    assert np.allclose(out["y"], out2["y"], rtol=1e-12)
    shared_only = oracle.moe_forward(shape, L["get_record"], x, idx, np.zeros_like(w))
    qx, dx = oracle.q8_0_quantize(x)
    rec, sc = L["get_record"]("shared", 0)
    sh = oracle.expert_ffn(rec, sc, shape.hidden, shape.shared_inter, 4, qx, dx)["o"]
    assert np.array_equal(shared_only["y"], sh)


def test_layer_matches_fp64_dequantised_path(tiny_layer):
    L = tiny_layer
    shape = L["shape"]
    x = synth.token_batch(shape, L["seed"], 0, range(8))
    out = oracle.moe_layer(shape, L["get_record"], x, L["router_w"], L["bias"])
    y = np.zeros_like(out["y"])
    for t in range(8):
        for j in range(shape.top_k):
            rec, sc = L["get_record"]("routed", int(out["idx"][t, j]))
            y[t] += out["w"][t, j] * oracle.expert_ffn_dequant_fp64(
                rec, sc, shape.hidden, shape.inter, 4, x[t:t + 1])[0]
        rec, sc = L["get_record"]("shared", 0)
        y[t] += oracle.expert_ffn_dequant_fp64(rec, sc, shape.hidden, shape.shared_inter, 4, x[t:t + 1])[0]
    assert np.allclose(out["y"], y, rtol=1e-9, atol=1e-12 * np.abs(y).max())


def test_int2_layer_combine_and_dequantised_path():
    """Packed int2 experts: the layer equals the dense every-expert evaluation
    with a dense gate matrix, and the fp64 dequantised products."""
    shape, seed = synth.TINY_INT2, 3
    routed = [synth.expert_record(shape, seed, 0, "routed", e) for e in range(shape.n_experts)]
    shared = [synth.expert_record(shape, seed, 0, "shared", 0)]
    get = lambda kind, e: routed[e] if kind == "routed" else shared[e]
    wr, bias = synth.router_weight(shape, seed), synth.router_bias(shape, seed)
    x = synth.token_batch(shape, seed, 0, range(6))
    out = oracle.moe_layer(shape, get, x, wr, bias)
    dense = oracle.dense_reference(shape, get, x, _dense_gates(out["idx"], out["w"], shape.n_experts))
    assert np.allclose(out["y"], dense, rtol=1e-12, atol=1e-14 * np.abs(dense).max())
    y = np.zeros_like(out["y"])
    for t in range(x.shape[0]):
        for j in range(shape.top_k):
            rec, sc = get("routed", int(out["idx"][t, j]))
            y[t] += out["w"][t, j] * oracle.expert_ffn_dequant_fp64(
                rec, sc, shape.hidden, shape.inter, 2, x[t:t + 1])[0]
        rec, sc = get("shared", 0)
        y[t] += oracle.expert_ffn_dequant_fp64(rec, sc, shape.hidden, shape.shared_inter, 2, x[t:t + 1])[0]
    assert np.allclose(out["y"], y, rtol=1e-9, atol=1e-12 * np.abs(y).max())


def test_runs_and_thread_pool_change_nothing(tiny_layer):
    """Splitting an expert's tokens into runs and evaluating the runs on a
    thread pool is evaluation order only: outputs, bounds, kept pairs and the
    per-run callback cover exactly the plain evaluation."""
    import concurrent.futures as cf
    L = tiny_layer
    shape = L["shape"]
    x = synth.token_batch(shape, 3, "runs", range(13))
    idx, w = oracle.route(oracle.router_logits(x, L["router_w"]), L["bias"], shape)
    idx[2, 1] = idx[2, 0]          # a duplicate id: two pairs of one token on one expert
    plain = oracle.moe_forward(shape, L["get_record"], x, idx, w, keep_pairs=True)
    seen = []
    with cf.ThreadPoolExecutor(4) as ex:
        split = oracle.moe_forward(shape, L["get_record"], x, idx, w, keep_pairs=True, max_tokens=3,
                                   map_fn=ex.map, on_entry=lambda k, e, o: seen.append((k, e, len(o["tokens"]))))
    assert np.array_equal(plain["y"], split["y"]) and np.array_equal(plain["y_err"], split["y_err"])
    assert plain["pairs"].keys() == split["pairs"].keys()
    for key, pr in plain["pairs"].items():
        for name in ("tokens", "js", "acc_g", "acc_u", "acc_d", "qh", "dh", "o"):
            assert np.array_equal(pr[name], split["pairs"][key][name]), (key, name)
    per_entry = {}
    for k, e, n in seen:
        assert n <= 3
        per_entry[(k, e)] = per_entry.get((k, e), 0) + n
    assert per_entry == {key: len(pr["tokens"]) for key, pr in plain["pairs"].items()}
