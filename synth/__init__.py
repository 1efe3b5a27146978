"""Seeded synthetic inputs for the routed-MoE layer (shared by tests and bench).

This module only draws random numbers and lays them out in the library's
input formats.  It holds none of the layer's arithmetic: no routing, no
activation quantisation, no expert products.  Both the CPU oracle and the
CUDA library consume the bytes made here.

Random source: Philox4x32-10, the counter-based generator of Salmon, Moraes,
Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11).  Each
tensor gets its own 64-bit key derived from (seed, tags) with SplitMix64
(Steele, Lea, Flood, OOPSLA'14); element pair ``c`` of a tensor is the output
of Philox at counter ``(c_lo, c_hi, 0, 0)``.  A CUDA twin of the same
generator (``synth/csrc/synth.cu``) produces the large weight tensors on the
device bit-identically (every step is integer arithmetic, one IEEE double
multiply and one round-to-nearest conversion).

Value recipes (the workload descriptions name normal distributions):

* approximately-normal integers ``z``: Irwin-Hall sum of four uniform 16-bit
  integers, centred: ``z = u0+u1+u2+u3 - 131070``; standard deviation
  ``SIGMA_Z = sqrt(4*(65536**2-1)/12)``.  Two values per Philox call.
* fp32 normal with std ``s``: ``float32(z) * float32(s / SIGMA_Z)`` (one fp32
  multiply, round to nearest).
* quantised weights (per-row absmax): ``q = sign(z)*floor((2*qmax*|z| +
  amax)/(2*amax))`` (round half away from zero of ``qmax*z/amax``, exact in
  integers) and ``scale = float32(float64(amax) * (std/(SIGMA_Z*qmax)))``;
  qmax is 7 for int4, 127 for int8 and 2 for int2, whose codes are then
  clamped to the container's [-2, 1] (so every one of the four codes occurs).
* uniform fp32 in (lo, hi): ``float32(lo + (hi-lo)*(r0+0.5)/2**32)``.
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass

import numpy as np

MASK32 = 0xFFFFFFFF
MASK64 = 0xFFFFFFFFFFFFFFFF
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
IH_CENTER = 131070  # 4 * 32767.5, the mean of four uniform 16-bit integers
SIGMA_Z = math.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0)


# ----------------------------------------------------------------------------
# keys
# ----------------------------------------------------------------------------
def splitmix64(v: int) -> int:
    """One SplitMix64 output step for state ``v`` (returns the mixed value)."""
    z = (v + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def _tag_int(tag) -> int:
    if isinstance(tag, str):
        return zlib.crc32(tag.encode()) | (1 << 40)
    if isinstance(tag, (int, np.integer)):
        return int(tag) & MASK64
    raise TypeError(f"unsupported tag {tag!r}")


def _flat(tags):
    for t in tags:
        if isinstance(t, (tuple, list)):
            yield from _flat(t)
        else:
            yield t


def make_key(seed: int, *tags) -> tuple[int, int]:
    """Derive the Philox key (k0, k1) for a tensor named by ``tags``."""
    h = splitmix64(int(seed) & MASK64)
    for t in _flat(tags):
        h = splitmix64(h ^ _tag_int(t))
    return h & MASK32, (h >> 32) & MASK32


# ----------------------------------------------------------------------------
# Philox4x32-10
# ----------------------------------------------------------------------------
def _mulhilo(a: int, b: np.ndarray):
    p = b.astype(np.uint64) * np.uint64(a)
    return (p >> np.uint64(32)).astype(np.uint32), (p & np.uint64(MASK32)).astype(np.uint32)


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Philox4x32 with 10 rounds on uint32 arrays; returns four uint32 arrays."""
    c0 = np.asarray(c0, np.uint32)
    c1 = np.asarray(c1, np.uint32)
    c2 = np.asarray(c2, np.uint32)
    c3 = np.asarray(c3, np.uint32)
    ka, kb = k0 & MASK32, k1 & MASK32
    for rnd in range(10):
        if rnd:
            ka = (ka + PHILOX_W0) & MASK32
            kb = (kb + PHILOX_W1) & MASK32
        hi0, lo0 = _mulhilo(PHILOX_M0, c0)
        hi1, lo1 = _mulhilo(PHILOX_M1, c2)
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint32(ka), lo1,
                          hi0 ^ c3 ^ np.uint32(kb), lo0)
    return c0, c1, c2, c3


def philox_block(key, first_call: int, n_calls: int):
    """Philox outputs for calls ``first_call .. first_call+n_calls-1``."""
    c = np.arange(first_call, first_call + n_calls, dtype=np.uint64)
    lo = (c & np.uint64(MASK32)).astype(np.uint32)
    hi = (c >> np.uint64(32)).astype(np.uint32)
    z = np.zeros_like(lo)
    return philox4x32_10(lo, hi, z, z, key[0], key[1])


def _ih4(w0: np.ndarray, w1: np.ndarray) -> np.ndarray:
    s = ((w0 & 0xFFFF).astype(np.int64) + (w0 >> 16).astype(np.int64)
         + (w1 & 0xFFFF).astype(np.int64) + (w1 >> 16).astype(np.int64))
    return (s - IH_CENTER).astype(np.int32)


def normal_int(key, n: int, start: int = 0) -> np.ndarray:
    """``n`` approximately-normal integers (std SIGMA_Z) at element ``start``."""
    if n == 0:
        return np.zeros(0, np.int32)
    first = start // 2
    last = (start + n - 1) // 2
    r0, r1, r2, r3 = philox_block(key, first, last - first + 1)
    out = np.empty(2 * (last - first + 1), np.int32)
    out[0::2] = _ih4(r0, r1)
    out[1::2] = _ih4(r2, r3)
    off = start - 2 * first
    return out[off:off + n]


def normal_f32(key, n: int, std: float, start: int = 0) -> np.ndarray:
    z = normal_int(key, n, start)
    return z.astype(np.float32) * np.float32(std / SIGMA_Z)


def uniform_f32(key, n: int, lo: float, hi: float) -> np.ndarray:
    r0, _, _, _ = philox_block(key, 0, n)
    v = lo + (hi - lo) * (r0.astype(np.float64) + 0.5) / 4294967296.0
    return v.astype(np.float32)


def uniform_u32(key, n: int) -> np.ndarray:
    r0, _, _, _ = philox_block(key, 0, n)
    return r0


# ----------------------------------------------------------------------------
# weight quantisation for synthetic experts (per-row absmax)
# ----------------------------------------------------------------------------
def quantize_rows_int(z: np.ndarray, qmax: int):
    """Round-half-away-from-zero of ``qmax*z/amax_row`` in exact integers."""
    z64 = z.astype(np.int64)
    amax = np.abs(z64).max(axis=1, keepdims=True)
    safe = np.maximum(amax, 1)
    q = np.sign(z64) * ((2 * qmax * np.abs(z64) + safe) // (2 * safe))
    q = np.where(amax == 0, 0, q)
    return q.astype(np.int8), amax[:, 0]


def quantize_groups_int(z: np.ndarray, qmax: int, group: int):
    """``quantize_rows_int`` applied to every run of ``group`` consecutive
    elements of a row: codes [rows, K] and the group maxima [rows, K/group]."""
    rows, k = z.shape
    q, amax = quantize_rows_int(z.reshape(rows * (k // group), group), qmax)
    return q.reshape(rows, k), amax.reshape(rows, k // group)


def pack_int2_rows(q: np.ndarray) -> np.ndarray:
    """Pack signed int2 codes [rows, K] into bytes [rows, K/4].

    Byte j of a row holds elements 4j .. 4j+3, element 4j+m in bits 2m and
    2m+1, each stored offset-binary (code + 2)."""
    n = (q.astype(np.int16) + 2).astype(np.uint8)
    b = np.zeros((q.shape[0], q.shape[1] // 4), np.uint8)
    for m in range(4):
        b |= (n[:, m::4] << (2 * m)).astype(np.uint8)
    return b


INT2_LO, INT2_HI = -2, 1


def scale_from_amax(amax: np.ndarray, std: float, qmax: int) -> np.ndarray:
    c = std / (SIGMA_Z * qmax)
    return (amax.astype(np.float64) * c).astype(np.float32)


def pack_int4_rows(q: np.ndarray) -> np.ndarray:
    """Pack signed int4 codes [rows, K] into bytes [rows, K/2].

    Byte j of a row holds element 2j in its low nibble and element 2j+1 in its
    high nibble, each stored offset-binary (code + 8)."""
    n = (q.astype(np.int16) + 8).astype(np.uint8)
    return (n[:, 0::2] | (n[:, 1::2] << 4)).astype(np.uint8)


@dataclass(frozen=True)
class LayerShape:
    hidden: int
    n_experts: int
    n_groups: int
    topk_group: int
    top_k: int
    inter: int
    n_shared: int
    shared_inter: int
    weight_bits: int
    routed_scaling_factor: float
    group_size: int = 0   # 0: one scale per output row; 64: one per 64 weights of a row

    @property
    def qmax(self) -> int:
        return {2: 2, 4: 7, 8: 127}[self.weight_bits]

    def row_bytes(self, k: int) -> int:
        return k * self.weight_bits // 8

    def record_bytes(self, inter: int | None = None) -> int:
        i = self.inter if inter is None else inter
        return 2 * i * self.row_bytes(self.hidden) + self.hidden * self.row_bytes(i)

    def scale_count(self, inter: int | None = None) -> int:
        i = self.inter if inter is None else inter
        if self.group_size:
            return 3 * i * self.hidden // self.group_size
        return 2 * i + self.hidden


WEIGHT_STD = 0.02
ROUTER_STD = 0.02
BIAS_LO, BIAS_HI = -0.1, 0.1
MATRIX_TAGS = ("gate", "up", "down")


def expert_matrix_key(seed, layer, kind, expert, matrix):
    """kind: 'routed' or 'shared'; matrix: 0 gate, 1 up, 2 down."""
    return make_key(seed, "expert", layer, kind, expert, matrix)


def expert_matrix(shape: LayerShape, seed, layer, kind, expert, matrix):
    """Return (codes int8 [rows,K], packed bytes [rows, row_bytes], scales f32:
    [rows], or [rows * K/group] row-major for group-scaled weights)."""
    inter = shape.inter if kind == "routed" else shape.shared_inter
    rows, k = ((inter, shape.hidden) if matrix < 2 else (shape.hidden, inter))
    key = expert_matrix_key(seed, layer, kind, expert, matrix)
    z = normal_int(key, rows * k).reshape(rows, k)
    if shape.group_size:
        q, amax = quantize_groups_int(z, shape.qmax, shape.group_size)
        scales = scale_from_amax(amax, WEIGHT_STD, shape.qmax).reshape(-1)
    else:
        q, amax = quantize_rows_int(z, shape.qmax)
        scales = scale_from_amax(amax, WEIGHT_STD, shape.qmax)
    if shape.weight_bits == 2:
        q = np.clip(q, INT2_LO, INT2_HI).astype(np.int8)
        packed = pack_int2_rows(q)
    elif shape.weight_bits == 4:
        packed = pack_int4_rows(q)
    else:
        packed = q.view(np.uint8)
    return q, packed, scales


def expert_record(shape: LayerShape, seed, layer, kind, expert):
    """One expert's bytes (gate | up | down) and its scales (gate|up|down)."""
    parts, scales = [], []
    for m in range(3):
        _, packed, s = expert_matrix(shape, seed, layer, kind, expert, m)
        parts.append(packed.reshape(-1))
        scales.append(s)
    return np.concatenate(parts), np.concatenate(scales)


def router_weight(shape: LayerShape, seed, layer=0):
    key = make_key(seed, "router_w", layer)
    return normal_f32(key, shape.n_experts * shape.hidden, ROUTER_STD).reshape(
        shape.n_experts, shape.hidden)


def router_bias(shape: LayerShape, seed, layer=0):
    key = make_key(seed, "router_bias", layer)
    return uniform_f32(key, shape.n_experts, BIAS_LO, BIAS_HI)


def zero_router_bias(shape: LayerShape):
    """Correction bias of the uniform-routing (prefill) workload: with every
    expert's bias equal the experts are exchangeable, so positions spread
    uniformly over them (a U(-0.1, 0.1) bias dominates the ranking once the
    selected sigmoid scores saturate near 1 and starves some experts)."""
    return np.zeros(shape.n_experts, np.float32)


def zipf_router_bias(shape: LayerShape, seed, layer, s=1.1, amp=0.3):
    """Correction bias skewed by a Zipf(s) profile over a seeded permutation."""
    base = router_bias(shape, seed, layer).astype(np.float64)
    u = uniform_u32(make_key(seed, "zipf_perm", layer), shape.n_experts)
    perm_rank = np.argsort(u, kind="stable")  # expert perm_rank[r] gets rank r
    rank = np.empty(shape.n_experts, np.int64)
    rank[perm_rank] = np.arange(shape.n_experts)
    prof = amp * (rank + 1.0) ** (-s)
    return (base + prof - prof.mean()).astype(np.float32)


def token_x(shape: LayerShape, seed, stream, position, attempt=0):
    """One activation row x ~ N(0,1) [hidden] for (stream, position, attempt)."""
    key = make_key(seed, "x", stream, position, attempt)
    return normal_f32(key, shape.hidden, 1.0)


def token_batch(shape: LayerShape, seed, stream, positions, attempts=None):
    rows = []
    for i, p in enumerate(positions):
        a = 0 if attempts is None else int(attempts[i])
        rows.append(token_x(shape, seed, stream, p, a))
    return np.stack(rows) if rows else np.zeros((0, shape.hidden), np.float32)


def residual_delta(shape: LayerShape, seed, step, layer, std=0.1):
    """Seeded residual update added between stacked layers."""
    key = make_key(seed, "residual", step, layer)
    return normal_f32(key, 32 * shape.hidden, std)


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------
TINY = LayerShape(hidden=256, n_experts=16, n_groups=4, topk_group=2, top_k=4,
                  inter=128, n_shared=1, shared_inter=128, weight_bits=4,
                  routed_scaling_factor=2.5)
GLM = LayerShape(hidden=6144, n_experts=256, n_groups=8, topk_group=4, top_k=8,
                 inter=2048, n_shared=1, shared_inter=2048, weight_bits=4,
                 routed_scaling_factor=2.5)
GLM_INT8 = LayerShape(hidden=6144, n_experts=256, n_groups=8, topk_group=4,
                      top_k=8, inter=2048, n_shared=1, shared_inter=2048,
                      weight_bits=8, routed_scaling_factor=2.5)
# group-scaled int4 ("gs64": one scale per 64 weights of a row)
TINY_GS64 = LayerShape(hidden=256, n_experts=16, n_groups=4, topk_group=2, top_k=4,
                       inter=128, n_shared=1, shared_inter=128, weight_bits=4,
                       routed_scaling_factor=2.5, group_size=64)
GLM_GS64 = LayerShape(hidden=6144, n_experts=256, n_groups=8, topk_group=4, top_k=8,
                      inter=2048, n_shared=1, shared_inter=2048, weight_bits=4,
                      routed_scaling_factor=2.5, group_size=64)
# packed int2 experts (per-row scales)
TINY_INT2 = LayerShape(hidden=256, n_experts=16, n_groups=4, topk_group=2, top_k=4,
                       inter=128, n_shared=1, shared_inter=128, weight_bits=2,
                       routed_scaling_factor=2.5)
GLM_INT2 = LayerShape(hidden=6144, n_experts=256, n_groups=8, topk_group=4, top_k=8,
                      inter=2048, n_shared=1, shared_inter=2048, weight_bits=2,
                      routed_scaling_factor=2.5)

WORKLOADS = {
    # name: (shape, seed, positions per call, calls)
    "tiny_t8": (TINY, 0, 8, 1),
    "glm_decode_b1": (GLM, 1, 1, 1000),
    "glm_mtp_verify_t4": (GLM, 2, 4, 500),
    "glm_prefill_s2048": (GLM, 3, 2048, 1),
    "glm_stack24_mtp1_b32": (GLM, 4, 32, 200),
}

# Correlation between consecutive positions of the MTP-verify chain, chosen so
# that consecutive top-8 sets share about half of their experts.
MTP_CHAIN_RHO = 0.83


def mtp_chain(shape: LayerShape, seed, call, n_pos=4, attempts=None):
    """x_{p+1} = rho*x_p + sqrt(1-rho^2)*z_p  (fp64, rounded to fp32 per row)."""
    rho = MTP_CHAIN_RHO
    a = [0] * n_pos if attempts is None else list(attempts)
    rows = [token_x(shape, seed, ("mtp", call), 0, a[0]).astype(np.float64)]
    for p in range(1, n_pos):
        z = token_x(shape, seed, ("mtp", call), p, a[p]).astype(np.float64)
        rows.append(rho * rows[-1] + math.sqrt(1.0 - rho * rho) * z)
    return np.stack(rows).astype(np.float32)


def stack_input(shape: LayerShape, seed, step, layer, batch=32):
    """Input of layer ``layer`` at decode step ``step`` of the layer stack:
    x_0 ~ N(0,1) per sequence, then x_{l+1} = x_l + delta_l with a seeded
    residual delta_l ~ N(0, 0.1^2) (fp32 adds, in layer order).  The layer
    outputs are not fed back, so every layer's input is known in advance."""
    x = token_batch(shape, seed, ("stack", step), range(batch))
    for l in range(layer):
        x = (x + residual_delta(shape, seed, step, l)[:batch * shape.hidden].reshape(batch, -1)).astype(np.float32)
    return x
