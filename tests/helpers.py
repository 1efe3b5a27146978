"""Test-side helpers: inputs whose routing has a margin, weights on either
device, comparisons.  May use the oracle (tests only)."""
from __future__ import annotations

import numpy as np

import oracle
import synth

DELTA = 1e-4  # minimum routing margin of a generated position (fp64 score units)


def margin_batch(shape, seed, stream, n, router_w, bias, start=0, delta=DELTA, max_attempts=64):
    """n positions (from `start`), each the first attempt whose routing margin
    is at least `delta`.  Returns (x [n,H] f32, attempts, rejected count)."""
    xs = synth.token_batch(shape, seed, stream, range(start, start + n))
    attempts = np.zeros(n, np.int64)
    rejected = 0
    todo = np.arange(n)
    while todo.size:
        m = oracle.route_margins(oracle.router_logits(xs[todo], router_w), bias, shape)
        bad = todo[m < delta]
        rejected += bad.size
        if bad.size and attempts[bad].max() >= max_attempts:
            raise RuntimeError("could not find positions with a routing margin")
        for i in bad:
            attempts[i] += 1
            xs[i] = synth.token_x(shape, seed, stream, start + int(i), int(attempts[i]))
        todo = bad
    return xs, attempts, rejected


def normwise_err(y_gpu, y_ref):
    """max over positions of max|dy| / max|y_ref| (the layer output tolerance)."""
    y_gpu = np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    den = np.abs(y_ref).max(axis=1)
    den = np.where(den > 0, den, 1.0)
    return float((np.abs(y_gpu - y_ref).max(axis=1) / den).max()) if y_ref.size else 0.0


def unpermute_int4(q):
    """Undo the library's in-block order 0,2,4,6,1,3,5,7 (int4 layouts)."""
    q = np.asarray(q)
    g = q.reshape(*q.shape[:-1], q.shape[-1] // 8, 8)
    out = np.empty_like(g)
    out[..., 0::2] = g[..., 0:4]
    out[..., 1::2] = g[..., 4:8]
    return out.reshape(q.shape)


def unpermute_int2(q):
    """Undo the library's in-block order for packed-int2 layouts: within each
    16 codes, natural element 4j+m is stored at position 4m+j."""
    q = np.asarray(q)
    g = q.reshape(*q.shape[:-1], q.shape[-1] // 16, 16)
    src = [4 * (i % 4) + i // 4 for i in range(16)]
    return g[..., src].reshape(q.shape)


def elementwise_err(y_gpu, y_ref, floor=1e-3):
    """max_i |dy_i| / max(|y_ref_i|, floor * rms(y_ref)) over each position's
    elements (reported beside the normwise figure, not asserted: near-zero
    elements make it a measure of fp32 summation error rather than of the
    layer)."""
    y_gpu = np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    if not y_ref.size:
        return 0.0
    rms = np.sqrt((y_ref ** 2).mean(axis=1, keepdims=True))
    den = np.maximum(np.abs(y_ref), floor * rms)
    den = np.where(den > 0, den, 1.0)
    return float((np.abs(y_gpu - y_ref) / den).max())


# ------------------------------------------------------------- exact ties
# The GLM-5.2 write-up's router check ("How it works (validated core
# mechanics)") sends an exact tie to the lower expert id; the same rule is
# taken for group ties.  With zero router rows every logit is 0 and every
# affinity sigmoid(0) = 1/2 exactly, and a bias on a 2^-10 grid keeps every
# biased score and every two-score group sum exact in fp32 and in fp64, so
# both sides see bit-identical ties.
TIE_UNIT = 2.0 ** -10


def tie_design(shape):
    """(bias [E] fp32, expected ids [k]) for the tiny or the GLM-5.2 router
    shape, with the selection derived by hand from the tie rules:

    tiny (16 experts, 4 groups of 4, keep 2, top 4): groups 1, 2, 3 tie at
    1 + 5u, so groups 1 and 2 are kept and group 3 -- which holds the best
    single expert, 12 at +8u -- is dropped; experts 4 and 9 tie at +5u (4
    first), then 5 and 6 win the tie at 1/2 against 7, 8, 10.

    GLM-5.2 (256 experts, 8 groups of 32, keep 4, top 8): groups 1 and 5 tie
    at 1 + 20u, groups 2, 3 and 7 at 1 + 15u, so 1, 5, 2, 3 are kept and 7 --
    whose expert 224 at +15u would rank second -- is dropped; then 67 (+20u),
    97 (+15u), the four-way tie 37, 41, 167, 168 at +10u in id order, and
    the lowest ids of the tie at 1/2: 32, 33."""
    E = shape.n_experts
    b = np.zeros(E)
    if E == 16:
        b[4] = 5
        b[9], b[11] = 5, -5
        b[12], b[13], b[14], b[15] = 8, -3, -20, -20
        expect = [4, 9, 5, 6]
    elif E == 256:
        b[37] = b[41] = 10                         # group 1
        b[64:96] = -5
        b[67] = 20                                 # group 2
        b[97] = 15                                 # group 3
        b[167] = b[168] = 10                       # group 5
        b[192:224] = -10                           # group 6
        b[224:256] = -30
        b[224], b[225] = 15, 0                     # group 7
        expect = [67, 97, 37, 41, 167, 168, 32, 33]
    else:
        raise ValueError("tie designs exist for the tiny and GLM-5.2 router shapes")
    return (b * TIE_UNIT).astype(np.float32), expect


def duplicate_group(router_w, bias, shape, src, dst):
    """Router rows and bias of group ``dst`` replaced by those of group
    ``src``: every expert of dst ties exactly with its twin in src, and the
    two group scores are equal."""
    n = shape.n_experts // shape.n_groups
    wr = np.array(router_w, copy=True)
    b = np.array(bias, copy=True)
    wr[dst * n:(dst + 1) * n] = wr[src * n:(src + 1) * n]
    b[dst * n:(dst + 1) * n] = b[src * n:(src + 1) * n]
    return wr, b


def route_margins_except_exact(logits, bias, shape):
    """Like ``oracle.route_margins`` but skipping gaps that are exactly 0 in
    fp64 (the designed ties between duplicated router rows): the smallest
    nonzero gap among consecutive biased scores of the first k + 1
    candidates and between consecutive group scores around the cut."""
    s = oracle.sigmoid(np.asarray(logits, np.float64))
    c = s + np.asarray(bias, np.float64)[None, :]
    T, E = c.shape
    G, n, k, tg = shape.n_groups, E // shape.n_groups, shape.top_k, shape.topk_group
    out = np.full(T, np.inf)
    for t in range(T):
        per = c[t].reshape(G, n)
        gs = -np.sort(-per, axis=1)[:, :min(2, n)].sum(axis=1)
        order = sorted(range(G), key=lambda g: (-gs[g], g))
        gv = gs[order]
        gaps = [gv[i] - gv[i + 1] for i in range(G - 1) if i in (tg - 1, tg - 2, tg)]
        kept = sorted(order[:tg])
        cand = sorted((e for g in kept for e in range(g * n, (g + 1) * n)), key=lambda e: (-c[t, e], e))
        cv = c[t, cand[:k + 1]]
        gaps += list(cv[:-1] - cv[1:])
        nz = [v for v in gaps if v != 0.0]
        out[t] = min(nz) if nz else np.inf
    return out
