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
