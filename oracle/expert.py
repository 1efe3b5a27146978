"""Oracle: one routed (or shared) SwiGLU expert on Q8_0 activations.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: colibrì v1.0 README, "What's implemented" (integer-dot kernels on
Q8_0-style int8 activations; int8 / packed int4 / packed int2 weights with
per-row scales)
and "Experimental Metal backend" (the routed-expert SwiGLU).  Group-scaled
int4 ("gs64": one scale per 64 weights of a row instead of one per row) is the
container the colibri GLM-5.2 quick start recommends ("2. Get the model").

Per expert with intermediate size I, weights gate [I,H], up [I,H], down [H,I]
(codes ``q``, per-row fp32 scales ``s``); per token with Q8_0 codes ``qx`` and
block scales ``dx``:

* block dot ``acc[r,b] = sum_{i in block b} q[r,i] * qx[i]`` -- exact integer;
* ``g[r] = s_g[r] * sum_b dx[b] * acc_g[r,b]``, same for ``u``;
* ``h = silu(g) * u`` with ``silu(g) = g / (1 + exp(-g))``;
* ``h`` is re-quantised to Q8_0 (every product takes int8 activations);
* ``o[c] = s_d[c] * sum_b dh[b] * acc_d[c,b]``.

With group scales (``group`` = 64, two Q8_0 blocks per group) the row scale
moves inside the block sum: ``g[r] = sum_b s_g[r, b // 2] * dx[b] * acc_g[r,b]``
(reading: the pages give the format, not the order of the scalings; this
is the plain definition, the dot product of the dequantised operands).

fp64 throughout except the Q8_0 step, which takes ``float32(h)`` and decides
the codes in fp32 (see ``quant.py``).
"""
from __future__ import annotations

import numpy as np

from .quant import QBLOCK, q8_0_quantize, q8_0_stable_mask, unpack_weight_rows

U32 = 2.0 ** -24  # unit roundoff of fp32


def block_dots(wq: np.ndarray, qx: np.ndarray) -> np.ndarray:
    """Exact per-32-block integer dot products.

    ``wq`` [R,K] weight codes, ``qx`` [T,K] activation codes ->
    int64 [T,R,K/32].  Checks that every result fits int32.

    Each block is one library matrix product in fp64.  The codes are 8-bit
    integers, so every product and every partial sum of 32 of them is an
    integer below 2**21 in magnitude and is represented exactly: the fp64
    product IS the integer dot product, in any summation order."""
    wq = np.asarray(wq)
    qx = np.atleast_2d(np.asarray(qx))
    R, K = wq.shape
    if K % QBLOCK or qx.shape[1] != K:
        raise ValueError("shape mismatch")
    if wq.dtype.itemsize > 1 or qx.dtype.itemsize > 1:
        if (np.abs(wq).max(initial=0) > 255) or (np.abs(qx).max(initial=0) > 255):
            raise ValueError("block dots take 8-bit codes")
    nb = K // QBLOCK
    W = wq.reshape(R, nb, QBLOCK).astype(np.float64).transpose(1, 2, 0)            # [nb, 32, R]
    X = np.ascontiguousarray(qx.reshape(qx.shape[0], nb, QBLOCK).astype(np.float64).transpose(1, 0, 2))
    acc = np.matmul(X, W).transpose(1, 2, 0).astype(np.int64)                          # [T, R, nb]
    if acc.size and (acc.max() > 2**31 - 1 or acc.min() < -2**31):
        raise OverflowError("block dot exceeds int32")
    return acc


def _scaled_rows(acc, d, s):
    """fp64 ``s[r] * sum_b d[t,b] * acc[t,r,b]`` and its fp32-evaluation bound.

    ``s`` [R] row scales, or [R, nb/bpg] group scales (one per ``bpg``
    consecutive blocks), then ``sum_b s[r, b // bpg] * d[t,b] * acc[t,r,b]``.
    The bound is the standard worst case for evaluating the same sum in fp32
    in any order: (terms + 4) * u * sum |s * d * acc| (Higham, gamma_n)."""
    d64 = np.asarray(d, np.float64)[:, None, :]
    terms = d64 * acc.astype(np.float64)
    s64 = np.asarray(s, np.float64)
    nterm = acc.shape[2]
    if s64.ndim == 2:
        bpg = nterm // s64.shape[1]
        terms = terms * np.repeat(s64, bpg, axis=1)[None, :, :]
        return terms.sum(axis=2), (nterm + 4) * U32 * np.abs(terms).sum(axis=2)
    val = s64[None, :] * terms.sum(axis=2)
    bound = (nterm + 4) * U32 * np.abs(s64)[None, :] * np.abs(terms).sum(axis=2)
    return val, bound


def _split_scales(scales, H: int, I: int, group: int):
    """(s_g, s_u, s_d): per-row [I], [I], [H], or per group [I, H/g], [I, H/g], [H, I/g]."""
    if not group:
        return scales[:I], scales[I:2 * I], scales[2 * I:2 * I + H]
    n = I * H // group
    return (scales[:n].reshape(I, H // group), scales[n:2 * n].reshape(I, H // group),
            scales[2 * n:3 * n].reshape(H, I // group))


def _split_record(record: np.ndarray, H: int, I: int, bits: int):
    rb = {2: lambda k: k // 4, 4: lambda k: k // 2, 8: lambda k: k}[bits]
    n_gu = I * rb(H)
    n_d = H * rb(I)
    rec = np.asarray(record, np.uint8).reshape(-1)
    if rec.size != 2 * n_gu + n_d:
        raise ValueError("record size does not match the shape")
    wg = unpack_weight_rows(rec[:n_gu], I, H, bits)
    wu = unpack_weight_rows(rec[n_gu:2 * n_gu], I, H, bits)
    wd = unpack_weight_rows(rec[2 * n_gu:], H, I, bits)
    return wg, wu, wd


def expert_ffn(record, scales, H: int, I: int, bits: int, qx, dx, group: int = 0):
    """Run one expert on tokens with Q8_0 activations ``qx`` [T,H], ``dx``.
    ``group``: 0 for per-row scales, else the weights per group scale (64).

    Returns a dict with the integer accumulators (``acc_g``, ``acc_u``,
    ``acc_d``), ``g``, ``u``, ``h`` (fp64), the requantised ``qh``/``dh``,
    the uniqueness mask ``qh_stable`` of each ``qh`` code against an fp32
    evaluation of g/u/h (see ``quant.q8_0_stable_mask``) and the output ``o``
    [T,H] (fp64)."""
    qx = np.atleast_2d(qx)
    dx = np.atleast_2d(dx)
    scales = np.asarray(scales, np.float32)
    s_g, s_u, s_d = _split_scales(scales, H, I, group)
    wg, wu, wd = _split_record(record, H, I, bits)
    acc_g = block_dots(wg, qx)
    acc_u = block_dots(wu, qx)
    g, eg = _scaled_rows(acc_g, dx, s_g)
    u, eu = _scaled_rows(acc_u, dx, s_u)
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-g))
    silu = g * sig
    h = silu * u
    # error of an fp32 evaluation of h from fp32 g, u (plus expf/div/mul ulps)
    dsilu = sig * (1.0 + g * (1.0 - sig))
    eh = np.abs(dsilu * u) * eg + np.abs(silu) * eu + np.abs(h) * 16 * U32
    h32 = h.astype(np.float32)
    qh, dh = q8_0_quantize(h32)
    stable = q8_0_stable_mask(h, 4.0 * eh)
    acc_d = block_dots(wd, qh)
    o, eo = _scaled_rows(acc_d, dh, s_d)
    return dict(acc_g=acc_g, acc_u=acc_u, acc_d=acc_d, g=g, u=u, h=h,
                h_err=eh, qh=qh, dh=dh, qh_stable=stable, o=o, o_err=eo)


def expert_ffn_dequant_fp64(record, scales, H: int, I: int, bits: int, x, group: int = 0):
    """The same expert evaluated by plain fp64 matrix products on dequantised
    operands: W = s * q for the weights, x and h as Q8_0 round trips.

    Mathematically equal to ``expert_ffn`` (the block decomposition only
    regroups the sum), so the two agree to fp64 rounding; used as a pin."""
    from .quant import q8_0_dequantize
    scales = np.asarray(scales, np.float64)
    s_g, s_u, s_d = _split_scales(scales, H, I, group)
    wg, wu, wd = _split_record(record, H, I, bits)

    def deq(w, s):  # W = s * q, the scale of a row or of each group of a row
        return w.astype(np.float64) * (np.repeat(s, group, axis=1) if group else s[:, None])
    Wg, Wu, Wd = deq(wg, s_g), deq(wu, s_u), deq(wd, s_d)
    qx, dx = q8_0_quantize(np.atleast_2d(x).astype(np.float32))
    xs = q8_0_dequantize(qx, dx)
    g = xs @ Wg.T
    u = xs @ Wu.T
    h = g / (1.0 + np.exp(-g)) * u
    qh, dh = q8_0_quantize(h.astype(np.float32))
    hs = q8_0_dequantize(qh, dh)
    return hs @ Wd.T
