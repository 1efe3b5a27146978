"""Oracle: Q8_0-style activation codes and packed int4 weight codes.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: colibrì v1.0 README, section "What's implemented" -- integer-dot
kernels with "Q8_0-style" int8 activations, and quantization kernels for int8,
packed int4 and packed int2 weights with per-row scales, dequantised on use,
whose packing is checked to be bit-identical to the int8 container.

The pages name the format but print no definition.  Readings taken here:

* Q8_0 block: 32 consecutive values, one fp32 scale ``d = amax / 127`` (IEEE
  fp32 division), ``inv = 1/d`` (fp32, 0 when d == 0), codes
  ``q = clamp(roundf(x * inv), -127, 127)`` with round-half-away-from-zero.
  All of it in fp32 because the result is an integer code that the kernel must
  reproduce bit for bit.  An all-zero block gives codes 0 and scale 0.
* packed int4: row-major, byte j of a row holds element 2j in the low nibble
  and element 2j+1 in the high nibble, each stored offset-binary (code + 8),
  so the codes span [-8, 7].
* packed int2: row-major, byte j of a row holds elements 4j .. 4j+3, element
  4j+m in bits 2m and 2m+1 (lowest element in the lowest bits, as for int4),
  each stored offset-binary (code + 2), so the codes span [-2, 1].
"""
from __future__ import annotations

import numpy as np

QBLOCK = 32


def _round_half_away(v32: np.ndarray) -> np.ndarray:
    # exact in fp64 for fp32 inputs
    v = v32.astype(np.float64)
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


def q8_0_quantize(x: np.ndarray):
    """Quantise fp32 ``x[..., K]`` (K % 32 == 0) to Q8_0 codes and scales.

    Returns ``(q int8 [..., K], d float32 [..., K/32])``.  Raises on
    non-finite input (the layer rejects corrupted activations rather than
    encoding them)."""
    x = np.asarray(x, dtype=np.float32)
    if x.shape[-1] % QBLOCK:
        raise ValueError("last dimension must be a multiple of 32")
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite activation")
    xb = x.reshape(*x.shape[:-1], x.shape[-1] // QBLOCK, QBLOCK)
    amax = np.abs(xb).max(axis=-1)                      # exact
    d = (amax / np.float32(127.0)).astype(np.float32)   # IEEE fp32 division
    with np.errstate(divide="ignore"):
        inv = np.where(d > 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
    v = (xb * inv[..., None]).astype(np.float32)        # one fp32 product
    q = np.clip(_round_half_away(v), -127, 127).astype(np.int8)
    return q.reshape(x.shape), d


def q8_0_dequantize(q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """fp64 values ``d * q`` of Q8_0 codes (for error bounds)."""
    qb = q.astype(np.float64).reshape(*q.shape[:-1], q.shape[-1] // QBLOCK, QBLOCK)
    return (qb * d.astype(np.float64)[..., None]).reshape(q.shape)


def q8_0_stable_mask(h64: np.ndarray, err: np.ndarray) -> np.ndarray:
    """Which Q8_0 codes of ``float32(h64)`` are unique under input error.

    A second implementation that computes ``h`` with absolute error at most
    ``err`` (per element) and then quantises in fp32 may legitimately produce a
    code one step away where the pre-rounding value ``h * inv`` sits within its
    error of a rounding boundary (a half-integer).  This returns True where the
    code is the same for every ``h`` in the error interval, so that a
    comparison can be exact there and ``|dq| <= 1`` elsewhere."""
    h64 = np.asarray(h64, np.float64)
    err = np.broadcast_to(np.asarray(err, np.float64), h64.shape)
    hb = h64.reshape(*h64.shape[:-1], h64.shape[-1] // QBLOCK, QBLOCK)
    eb = err.reshape(hb.shape)
    h32 = hb.astype(np.float32)
    amax = np.abs(h32).max(axis=-1).astype(np.float64)
    amax_err = eb.max(axis=-1) + amax * 2.0 ** -23
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(amax > 0, 127.0 / amax, 0.0)
        rel_inv = np.where(amax > 0, amax_err / amax, 0.0) + 4 * 2.0 ** -24
    v = h32.astype(np.float64) * inv[..., None]
    dv = (eb + np.abs(h32) * 2.0 ** -24) * inv[..., None] + np.abs(v) * rel_inv[..., None] \
        + np.abs(v) * 2.0 ** -23
    frac = np.abs(v) - np.floor(np.abs(v))
    dist = np.abs(frac - 0.5)
    stable = dist > 2.0 * dv
    # a block whose scale is zero maps everything to 0 on both sides only if
    # the other side also sees amax == 0, i.e. when the error is zero there.
    stable &= ~((amax == 0)[..., None] & (eb > 0))
    return stable.reshape(h64.shape)


def int4_pack(q: np.ndarray) -> np.ndarray:
    """Pack int4 codes ``q[..., K]`` (values in [-8, 7], K even) to bytes."""
    q = np.asarray(q)
    if q.shape[-1] % 2:
        raise ValueError("K must be even")
    if q.min(initial=0) < -8 or q.max(initial=0) > 7:
        raise ValueError("int4 code out of range")
    n = (q.astype(np.int16) + 8).astype(np.uint8)
    return (n[..., 0::2] | (n[..., 1::2] << 4)).astype(np.uint8)


def int4_unpack(b: np.ndarray) -> np.ndarray:
    """Unpack bytes ``b[..., K/2]`` to int4 codes ``[..., K]`` (int8)."""
    b = np.asarray(b, dtype=np.uint8)
    lo = (b & 0x0F).astype(np.int16) - 8
    hi = (b >> 4).astype(np.int16) - 8
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def int2_pack(q: np.ndarray) -> np.ndarray:
    """Pack int2 codes ``q[..., K]`` (values in [-2, 1], K % 4 == 0) to bytes."""
    q = np.asarray(q)
    if q.shape[-1] % 4:
        raise ValueError("K must be a multiple of 4")
    if q.min(initial=0) < -2 or q.max(initial=0) > 1:
        raise ValueError("int2 code out of range")
    n = (q.astype(np.int16) + 2).astype(np.uint8)
    b = np.zeros(q.shape[:-1] + (q.shape[-1] // 4,), np.uint8)
    for m in range(4):
        b |= (n[..., m::4] << (2 * m)).astype(np.uint8)
    return b


def int2_unpack(b: np.ndarray) -> np.ndarray:
    """Unpack bytes ``b[..., K/4]`` to int2 codes ``[..., K]`` (int8)."""
    b = np.asarray(b, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (4 * b.shape[-1],), np.int8)
    for m in range(4):
        out[..., m::4] = ((b >> (2 * m)) & 3).astype(np.int16) - 2
    return out


def unpack_weight_rows(raw: np.ndarray, rows: int, k: int, bits: int) -> np.ndarray:
    """Weight codes [rows, k] from a row-major packed matrix of ``bits`` bits."""
    raw = np.asarray(raw, np.uint8)
    if bits == 4:
        return int4_unpack(raw.reshape(rows, k // 2))
    if bits == 2:
        return int2_unpack(raw.reshape(rows, k // 4))
    if bits == 8:
        return raw.reshape(rows, k).view(np.int8)
    raise ValueError("weight_bits must be 2, 4 or 8")
