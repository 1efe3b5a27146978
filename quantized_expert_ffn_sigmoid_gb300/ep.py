"""Host plumbing for expert-parallel sharding of the MoE layer.

The colibrì v1.0 README ("Experimental resident CUDA backend") places each
expert whole on one device, and the JustVugg/colibri README ("Local cluster
mode") sends one batch-union request per layer to each worker.  Here shard r
of P owns the routed experts e with e mod P == r (their records stored
consecutively in ascending id order) plus, on shard 0, the shared experts;
every shard runs the router on the same input, computes its partial output
with ``coli_moe_layer`` / ``coli_moe_forward`` under ``Cfg.of(shape, r, P)``,
and one sum over the shards (an all-reduce of y per layer call) gives the
layer's output.  Nothing here computes any part of the layer: it selects
which records a shard holds and sums the shards' outputs with
torch.distributed."""
from __future__ import annotations


def owned_experts(n_experts: int, rank: int, size: int) -> list[int]:
    """Routed expert ids held by shard ``rank`` of ``size`` (ascending; the
    i-th one is the shard's local record i)."""
    if size <= 1:
        if rank != 0:
            raise ValueError("rank must be 0 without sharding")
        return list(range(n_experts))
    if not 0 <= rank < size <= n_experts:
        raise ValueError("need 0 <= rank < size <= n_experts")
    return list(range(rank, n_experts, size))


def shard_weights(experts, expert_scales, shared, shared_scales, rank: int, size: int):
    """The tensors shard ``rank`` holds, cut from a whole layer's records
    ([E, record_bytes] and [E, scales]): its routed records and scales made
    contiguous, and the shared experts on shard 0 only (None elsewhere)."""
    ids = owned_experts(experts.shape[0], rank, size)
    step = max(size, 1)
    rec = experts[rank::step].contiguous()
    sc = expert_scales[rank::step].contiguous()
    assert rec.shape[0] == len(ids)
    if rank == 0:
        return rec, sc, shared, shared_scales
    return rec, sc, None, None


def all_reduce_output(y, group=None):
    """Sum the shards' partial outputs in place (one collective per layer call)."""
    import torch.distributed as dist
    dist.all_reduce(y, op=dist.ReduceOp.SUM, group=group)
    return y
