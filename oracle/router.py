"""Oracle: the sigmoid ``noaux_tc`` group-limited top-k router.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "Colibri (colibrì): GLM-5.2 local inference on 25 GB of RAM",
sections "What it is" and "How it works (validated core mechanics)":

* affinity ``s = sigmoid(logit)``;
* a per-expert correction bias is added to ``s`` for ranking only;
* the selected experts are ordered by biased score, a tie going to the lower
  expert id;
* gate weights are the unbiased ``s`` of the selected experts renormalised
  to sum to 1, then multiplied by ``routed_scaling_factor`` (the page applies
  that constant downstream; colibrì v1.0 README "What's implemented" lists
  the factor as part of the router);
* non-finite logits or bias are rejected with an error, never ranked.

Group limiting (the DeepSeek-V3 ``noaux_tc`` pattern the page cites, not
spelled out on the pages).  Readings taken here:

* experts are split into ``n_groups`` consecutive groups of equal size;
* a group's score is the sum of its two largest biased scores (its largest
  one if a group has a single expert);
* the ``topk_group`` best groups are kept (ties to the lower group id);
  experts of dropped groups are never selectable (masked to -inf, not 0);
* the top-k experts by biased score among the kept groups are selected,
  ties to the lower expert id, reported in descending biased-score order.
* if every selected affinity underflows to 0 the weights are 0.
"""
from __future__ import annotations

import numpy as np


def sigmoid(v: np.ndarray) -> np.ndarray:
    """fp64 logistic function ``1 / (1 + exp(-v))``."""
    v = np.asarray(v, np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-v))


def router_logits(x: np.ndarray, router_w: np.ndarray) -> np.ndarray:
    """Router logits ``x @ router_w.T`` in fp64 (x [T,H], router_w [E,H])."""
    return np.asarray(x, np.float64) @ np.asarray(router_w, np.float64).T


def _check_cfg(cfg, n_experts):
    g = cfg.n_groups
    if n_experts % g:
        raise ValueError("n_experts must be divisible by n_groups")
    if not (1 <= cfg.topk_group <= g):
        raise ValueError("topk_group out of range")
    if not (1 <= cfg.top_k <= cfg.topk_group * (n_experts // g)):
        raise ValueError("top_k larger than the experts of the kept groups")


def _group_scores(c_row: np.ndarray, n_groups: int) -> np.ndarray:
    per = c_row.reshape(n_groups, -1)
    m = min(2, per.shape[1])
    top = -np.sort(-per, axis=1)[:, :m]
    return top.sum(axis=1)


def _select_one(c_row: np.ndarray, cfg):
    E = c_row.shape[0]
    G = cfg.n_groups
    gs = _group_scores(c_row, G)
    group_order = sorted(range(G), key=lambda g: (-gs[g], g))
    kept = sorted(group_order[:cfg.topk_group])
    size = E // G
    cand = [e for g in kept for e in range(g * size, (g + 1) * size)]
    order = sorted(cand, key=lambda e: (-c_row[e], e))
    return order, gs, group_order


def route(logits: np.ndarray, bias: np.ndarray, cfg):
    """Select experts and gate weights.

    ``logits`` [T,E] (any float), ``bias`` [E] fp32, ``cfg`` with n_groups,
    topk_group, top_k, routed_scaling_factor.  Returns ``(idx int64 [T,k],
    w float64 [T,k])``.  Raises ValueError on non-finite logits or bias."""
    logits = np.asarray(logits, np.float64)
    bias = np.asarray(bias, np.float64)
    if not np.all(np.isfinite(logits)) or not np.all(np.isfinite(bias)):
        raise ValueError("non-finite router logits or correction bias")
    T, E = logits.shape
    _check_cfg(cfg, E)
    k = cfg.top_k
    s = sigmoid(logits)
    c = s + bias[None, :]
    idx = np.zeros((T, k), np.int64)
    w = np.zeros((T, k), np.float64)
    for t in range(T):
        order, _, _ = _select_one(c[t], cfg)
        sel = order[:k]
        idx[t] = sel
        tot = s[t, sel].sum()
        if tot > 0:
            w[t] = s[t, sel] / tot * cfg.routed_scaling_factor
    return idx, w


def route_margins(logits: np.ndarray, bias: np.ndarray, cfg) -> np.ndarray:
    """Smallest score gap that decides each token's routing (fp64).

    The minimum over: consecutive biased scores among the first k+1
    candidates of the kept groups (order and membership of the selection),
    and the gap between the ``topk_group``-th and the next group score (which
    groups are kept).  A second implementation whose scores differ from these
    by less than half the margin selects the same experts in the same order."""
    logits = np.asarray(logits, np.float64)
    bias = np.asarray(bias, np.float64)
    T, E = logits.shape
    _check_cfg(cfg, E)
    k = cfg.top_k
    s = sigmoid(logits)
    c = s + bias[None, :]
    out = np.full(T, np.inf)
    for t in range(T):
        order, gs, gorder = _select_one(c[t], cfg)
        vals = c[t, order[:k + 1]]
        if len(vals) > 1:
            out[t] = np.min(vals[:-1] - vals[1:])
        if cfg.topk_group < cfg.n_groups:
            gsorted = gs[gorder]
            out[t] = min(out[t], gsorted[cfg.topk_group - 1] - gsorted[cfg.topk_group])
    return out
