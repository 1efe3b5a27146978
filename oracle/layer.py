"""Oracle: batch-union dispatch tables and the whole routed-MoE layer.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources: colibrì v1.0 README, "What's implemented" (batch-union MoE: each
unique expert of a batch is read once and applied to every position routed to
it; the always-on shared expert; the sigmoid router with
``routed_scaling_factor``) and "Colibri (colibrì): GLM-5.2 local inference on
25 GB of RAM", "How it works (validated core mechanics)" (the routed output
is the gate-weighted sum over the selected experts).

Layer output for token t:
``y[t] = sum_j w[t,j] * E_{idx[t,j]}(x[t]) + sum_s S_s(x[t])`` with the shared
experts weighted 1.  Batch-union only changes evaluation order: the oracle
groups tokens by expert for speed, and each token's result is computed
independently of the others.
"""
from __future__ import annotations

import numpy as np

from .expert import expert_ffn, U32
from .quant import q8_0_quantize
from .router import route, router_logits


def union_tables(idx: np.ndarray, n_experts: int, n_shared: int):
    """Canonical batch-union tables for routing ``idx`` [T,k].

    Entries are the distinct valid routed experts in ascending id, then the
    ``n_shared`` shared experts.  Each routed entry lists its (t, j) pairs in
    ascending (t, j) order; each shared entry lists every token.  Pair slots
    are numbered consecutively in entry order; ``slot[t,j]`` is the slot of
    pair (t, j), -1 for an id outside [0, n_experts).

    Returns dict(uniq, counts, offsets, pair_token, pair_j, slot)."""
    idx = np.asarray(idx, np.int64)
    T, k = idx.shape
    valid = (idx >= 0) & (idx < n_experts)
    uniq = np.unique(idx[valid])
    counts, pair_token, pair_j = [], [], []
    slot = np.full((T, k), -1, np.int64)
    p = 0
    for e in uniq:
        n = 0
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    pair_token.append(t)
                    pair_j.append(j)
                    slot[t, j] = p
                    p += 1
                    n += 1
        counts.append(n)
    for _ in range(n_shared):
        for t in range(T):
            pair_token.append(t)
            pair_j.append(-1)
        counts.append(T)
    counts = np.asarray(counts, np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return dict(uniq=uniq.astype(np.int64), counts=counts, offsets=offsets,
                pair_token=np.asarray(pair_token, np.int64),
                pair_j=np.asarray(pair_j, np.int64), slot=slot)


def moe_forward(shape, get_record, x: np.ndarray, idx: np.ndarray, w: np.ndarray,
                keep_pairs: bool = False, on_entry=None, map_fn=map, max_tokens: int | None = None):
    """Layer output for given routing (``idx`` [T,k], ``w`` [T,k]).

    ``get_record(kind, e)`` returns ``(record bytes, scales)`` for
    kind 'routed' or 'shared'.  Returns dict(y fp64 [T,H], y_err, qx, dx,
    pairs) where ``pairs[(kind, e)]`` holds the expert dict of ``expert_ffn``
    for the tokens routed to it (if ``keep_pairs``).

    Evaluation order only (each token's result is independent of the
    others, as the batch-union description says): ``max_tokens`` splits an
    expert's tokens into runs of at most that many, ``map_fn`` evaluates the
    (expert, run) jobs (e.g. a thread pool's ``map``; results are combined in
    job order, so the output does not depend on it), and ``on_entry(kind, e,
    out)`` is called with each run's ``expert_ffn`` dict (plus ``tokens`` and
    ``js``, the pairs' (t, j)) before its intermediates are dropped."""
    H = shape.hidden
    x = np.atleast_2d(np.asarray(x, np.float32))
    T = x.shape[0]
    idx = np.asarray(idx, np.int64)
    w = np.asarray(w, np.float64)
    qx, dx = q8_0_quantize(x)
    y = np.zeros((T, H), np.float64)
    yerr = np.zeros((T, H), np.float64)
    pairs = {}
    tabs = union_tables(idx, shape.n_experts, shape.n_shared)
    group = getattr(shape, "group_size", 0)
    run_len = max_tokens or max(T, 1)
    jobs = []
    for e in tabs["uniq"]:
        sel = np.argwhere(idx == e)              # (t, j) ascending
        for c in range(0, len(sel), run_len):
            jobs.append(("routed", int(e), sel[c:c + run_len]))
    for s in range(shape.n_shared):
        sel = np.stack([np.arange(T), np.full(T, -1)], axis=1)
        for c in range(0, T, run_len):
            jobs.append(("shared", s, sel[c:c + run_len]))

    def run(job):
        kind, e, sel = job
        toks = sel[:, 0]
        rec, sc = get_record(kind, e)
        inter = shape.inter if kind == "routed" else shape.shared_inter
        out = expert_ffn(rec, sc, H, inter, shape.weight_bits, qx[toks], dx[toks], group)
        out["tokens"] = toks
        out["js"] = sel[:, 1]
        if on_entry is not None:
            on_entry(kind, e, out)
        return out if keep_pairs else dict(o=out["o"], o_err=out["o_err"])

    for (kind, e, sel), out in zip(jobs, map_fn(run, jobs)):
        for n, (t, j) in enumerate(sel):
            if kind == "routed":
                y[t] += w[t, j] * out["o"][n]
                yerr[t] += abs(w[t, j]) * (out["o_err"][n] + np.abs(out["o"][n]) * 4 * U32)
            else:
                y[t] += out["o"][n]
                yerr[t] += out["o_err"][n]
        if keep_pairs:
            key = (kind, e)
            if key in pairs:   # a later run of the same expert: append its pairs
                prev = pairs[key]
                pairs[key] = {k: (np.concatenate([prev[k], v]) if isinstance(v, np.ndarray) and v.ndim
                                  else v) for k, v in out.items()}
            else:
                pairs[key] = out
    return dict(y=y, y_err=yerr, qx=qx, dx=dx, pairs=pairs, tables=tabs)


def moe_layer(shape, get_record, x, router_w, bias, keep_pairs: bool = False):
    """Router then forward: returns the ``moe_forward`` dict plus idx, w, logits."""
    logits = router_logits(x, router_w)
    idx, w = route(logits, bias, shape)
    out = moe_forward(shape, get_record, x, idx, w, keep_pairs=keep_pairs)
    out.update(idx=idx, w=w, logits=logits)
    return out


def dense_reference(shape, get_record, x, gate_dense: np.ndarray):
    """Every routed expert on every token, weighted by a dense gate matrix
    ``gate_dense`` [T,E] (zeros off the selection), plus the shared experts.

    Independent of the union tables and of the per-pair bookkeeping; the
    combine invariant says it equals ``moe_forward`` for the same gates."""
    H = shape.hidden
    x = np.atleast_2d(np.asarray(x, np.float32))
    qx, dx = q8_0_quantize(x)
    y = np.zeros((x.shape[0], H))
    for e in range(shape.n_experts):
        rec, sc = get_record("routed", e)
        o = expert_ffn(rec, sc, H, shape.inter, shape.weight_bits, qx, dx,
                         getattr(shape, "group_size", 0))["o"]
        y += gate_dense[:, e:e + 1] * o
    for s in range(shape.n_shared):
        rec, sc = get_record("shared", s)
        y += expert_ffn(rec, sc, H, shape.shared_inter, shape.weight_bits, qx, dx,
                         getattr(shape, "group_size", 0))["o"]
    return y
