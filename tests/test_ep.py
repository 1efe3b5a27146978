"""Expert-parallel sharding on the CPU (no GPU needed).

Shard r of P owns the routed experts e with e mod P == r and, on shard 0,
the shared experts (colibrì v1.0 README, "Experimental resident CUDA
backend": each expert lives whole on one device).  The layer output is the
sum of the shards' partial outputs (the combine is linear in the experts'
contributions), which one all-reduce per layer call forms.  Pinned here with
the oracle: the shard decomposition of the package's host helpers sums to the
whole layer, also through two gloo ranks."""
import os
import socket
import sys
from types import SimpleNamespace

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _ep():
    # the helpers live in the package, whose import loads the compiled library
    try:
        from quantized_expert_ffn_sigmoid_gb300 import ep
    except (ImportError, OSError) as exc:
        pytest.skip(f"library not built: {exc}")
    return ep


def shard_routing(idx, n_experts, rank, size, owned):
    """The routing a shard computes: other shards' experts skipped (-1)."""
    own = np.zeros(n_experts, bool)
    own[owned] = True
    return np.where((idx >= 0) & own[np.clip(idx, 0, n_experts - 1)], idx, -1)


def shard_output(shape, get_record, x, idx, w, rank, size, owned):
    sh = SimpleNamespace(**{**shape.__dict__, "n_shared": shape.n_shared if rank == 0 else 0})
    return oracle.moe_forward(sh, get_record, x, shard_routing(idx, shape.n_experts, rank, size, owned), w)


def test_owned_experts_partition():
    ep = _ep()
    for E, P in ((16, 1), (16, 2), (16, 3), (256, 4), (256, 8), (5, 5)):
        parts = [ep.owned_experts(E, r, P) for r in range(P)]
        assert sorted(e for p in parts for e in p) == list(range(E))
        for r, p in enumerate(parts):
            assert all(e % P == r for e in p) and p == sorted(p)
            assert [e // P for e in p] == list(range(len(p)))   # local record index
    with pytest.raises(ValueError):
        ep.owned_experts(16, 2, 2)


def test_shard_weights_slices_records():
    ep = _ep()
    recs = torch.arange(10 * 3).reshape(10, 3)
    scs = torch.arange(10 * 2).reshape(10, 2).float()
    sh, shs = torch.zeros(1, 3), torch.zeros(1, 2)
    r, s, a, b = ep.shard_weights(recs, scs, sh, shs, 1, 3)
    assert r.tolist() == recs[[1, 4, 7]].tolist() and s.tolist() == scs[[1, 4, 7]].tolist()
    assert r.is_contiguous() and a is None and b is None
    r0 = ep.shard_weights(recs, scs, sh, shs, 0, 3)
    assert r0[2] is sh and r0[0].shape[0] == 4


@pytest.mark.parametrize("P", [2, 3, 4])
def test_shard_outputs_sum_to_the_layer(tiny_layer, P):
    ep = _ep()
    L = tiny_layer
    shape = L["shape"]
    x = synth.token_batch(shape, 9, "ep", range(11))
    whole = oracle.moe_layer(shape, L["get_record"], x, L["router_w"], L["bias"])
    total = np.zeros_like(whole["y"])
    for r in range(P):
        total += shard_output(shape, L["get_record"], x, whole["idx"], whole["w"], r, P,
                              ep.owned_experts(shape.n_experts, r, P))["y"]
    np.testing.assert_allclose(total, whole["y"], rtol=1e-12, atol=1e-12 * np.abs(whole["y"]).max())


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from quantized_expert_ffn_sigmoid_gb300 import ep
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shape = synth.TINY
        seed = synth.WORKLOADS["tiny_t8"][1]
        recs = {e: synth.expert_record(shape, seed, 0, "routed", e) for e in ep.owned_experts(16, rank, world)}
        shared = synth.expert_record(shape, seed, 0, "shared", 0)
        get = lambda kind, e: recs[e] if kind == "routed" else shared
        x = synth.token_batch(shape, seed, "ep-gloo", range(8))
        # every shard runs the router on the same input
        idx, w = oracle.route(oracle.router_logits(x, synth.router_weight(shape, seed)),
                              synth.router_bias(shape, seed), shape)
        y = torch.from_numpy(shard_output(shape, get, x, idx, w, rank, world, sorted(recs))["y"])
        ep.all_reduce_output(y)
        q.put((rank, y.numpy()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_sum_to_the_layer(tiny_layer):
    _ep()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    L = tiny_layer
    x = synth.token_batch(L["shape"], L["seed"], "ep-gloo", range(8))
    whole = oracle.moe_layer(L["shape"], L["get_record"], x, L["router_w"], L["bias"])["y"]
    for r in (0, 1):
        np.testing.assert_allclose(res[r], whole, rtol=1e-12, atol=1e-12 * np.abs(whole).max())
