"""Pins for the oracle's block dot products and the SwiGLU expert."""
import numpy as np
import pytest

import oracle
import synth


def test_block_dot_closed_forms():
    w = np.full((2, 64), 7, np.int8)
    x = np.full((1, 64), 127, np.int8)
    assert oracle.block_dots(w, x).tolist() == [[[28448, 28448], [28448, 28448]]]
    alt = np.tile(np.array([1, -1], np.int8), 32)[None, :]
    assert oracle.block_dots(np.full((1, 64), 5, np.int8), alt).tolist() == [[[0, 0]]]
    # largest int8 x int8 block fits int32
    assert oracle.block_dots(np.full((1, 32), -127, np.int8),
                             np.full((1, 32), -127, np.int8))[0, 0, 0] == 32 * 127 * 127


def test_block_dot_brute_force():
    rng = np.random.default_rng(3)
    w = rng.integers(-8, 8, (5, 96)).astype(np.int8)
    x = rng.integers(-127, 128, (3, 96)).astype(np.int8)
    acc = oracle.block_dots(w, x)
    for t in range(3):
        for r in range(5):
            for b in range(3):
                ref = sum(int(w[r, 32 * b + i]) * int(x[t, 32 * b + i]) for i in range(32))
                assert acc[t, r, b] == ref


def test_block_dot_full_int8_range_brute_force():
    # int8 weights and codes at the extremes of their range, a GLM-5.2-sized
    # reduction: sampled blocks against Python integer arithmetic
    rng = np.random.default_rng(11)
    w = rng.choice(np.array([-128, -127, -1, 0, 1, 126, 127], np.int8), (7, 6144))
    x = rng.integers(-127, 128, (4, 6144)).astype(np.int8)
    x[0] = -127
    w[0] = -128
    acc = oracle.block_dots(w, x)
    assert acc.dtype == np.int64 and acc.shape == (4, 7, 192)
    assert acc[0, 0, 0] == 32 * 128 * 127
    for t, r, b in [(0, 0, 191), (1, 3, 0), (2, 6, 77), (3, 1, 150), (3, 6, 191)]:
        ref = sum(int(w[r, 32 * b + i]) * int(x[t, 32 * b + i]) for i in range(32))
        assert acc[t, r, b] == ref


def _record(gate, up, down, bits=4):
    pk = {4: oracle.int4_pack, 2: oracle.int2_pack,
          8: lambda q: q.astype(np.int8).view(np.uint8)}[bits]
    return np.concatenate([pk(gate).reshape(-1), pk(up).reshape(-1), pk(down).reshape(-1)])


def test_expert_uniform_closed_form():
    # H = I = 32, all weight codes 1, scales 1, x all 1:
    # qx = 127, dx = 1/127 -> g = u = 32, h = silu(32)*32, o = 32*h
    H = I = 32
    one = np.ones((32, 32), np.int8)
    rec = _record(one, one, one)
    scales = np.ones(2 * I + H, np.float32)
    qx, dx = oracle.q8_0_quantize(np.ones((1, H), np.float32))
    out = oracle.expert_ffn(rec, scales, H, I, 4, qx, dx)
    assert np.all(out["acc_g"] == 32 * 127)
    g = 32 * 127 * float(np.float32(1.0) / np.float32(127.0))
    h = g / (1 + np.exp(-g)) * g
    assert np.allclose(out["h"], h, rtol=1e-15)
    assert np.all(out["qh"] == 127)
    assert np.allclose(out["o"], 32 * 127 * float(np.float32(np.float32(h) / np.float32(127))),
                       rtol=1e-12)


def test_expert_single_code_locates_row_and_column():
    # one non-zero gate code at (row 5, col 40) and one up code at (5, 40):
    # only h[5] is non-zero; one down code at (row 9, col 5) -> only o[9]
    H, I = 64, 32
    gate = np.zeros((I, H), np.int8)
    up = np.zeros((I, H), np.int8)
    down = np.zeros((H, I), np.int8)
    gate[5, 40] = 3
    up[5, 40] = -2
    down[9, 5] = 7
    rec = _record(gate, up, down)
    scales = np.concatenate([np.full(I, 0.5), np.full(I, 0.25), np.full(H, 2.0)]).astype(np.float32)
    x = np.zeros((1, H), np.float32)
    x[0, 40] = 1.0
    x[0, 33] = -0.5
    qx, dx = oracle.q8_0_quantize(x)
    out = oracle.expert_ffn(rec, scales, H, I, 4, qx, dx)
    g = 0.5 * float(dx[0, 1]) * 3 * int(qx[0, 40])
    u = 0.25 * float(dx[0, 1]) * -2 * int(qx[0, 40])
    assert np.flatnonzero(out["g"][0]).tolist() == [5]
    assert np.isclose(out["g"][0, 5], g) and np.isclose(out["u"][0, 5], u)
    assert np.flatnonzero(out["o"][0]).tolist() == [9]
    hq = out["qh"][0, 5]
    assert np.isclose(out["o"][0, 9], 2.0 * float(out["dh"][0, 0]) * 7 * int(hq))


def test_zero_expert_gives_zero():
    H, I = 64, 32
    rec = _record(np.zeros((I, H), np.int8), np.zeros((I, H), np.int8), np.zeros((H, I), np.int8))
    qx, dx = oracle.q8_0_quantize(np.random.default_rng(0).standard_normal((2, H)).astype(np.float32))
    out = oracle.expert_ffn(rec, np.ones(2 * I + H, np.float32), H, I, 4, qx, dx)
    assert np.all(out["o"] == 0) and np.all(out["qh"] == 0) and np.all(out["dh"] == 0)


def test_int2_expert_closed_form():
    # H = I = 32, gate codes -2, up codes 1, down codes alternating -2 / 1,
    # scales 1, x all 1 (qx = 127, dx = 1/127): g = -2 * 32 = -64, u = 32,
    # h = silu(-64) * 32 (tiny, negative, all equal -> qh = -127),
    # o[c] = dh * (-127) * sum(down row c) = dh * (-127) * 16 * (-1)
    H = I = 32
    gate = np.full((I, H), -2, np.int8)
    up = np.ones((I, H), np.int8)
    down = np.tile(np.array([-2, 1], np.int8), (H, I // 2))
    rec = _record(gate, up, down, bits=2)
    assert rec.size == 3 * 32 * 32 // 4
    scales = np.ones(2 * I + H, np.float32)
    qx, dx = oracle.q8_0_quantize(np.ones((1, H), np.float32))
    out = oracle.expert_ffn(rec, scales, H, I, 2, qx, dx)
    assert np.all(out["acc_g"] == -2 * 32 * 127) and np.all(out["acc_u"] == 32 * 127)
    d = float(np.float32(1.0) / np.float32(127.0))
    g, u = -2 * 32 * 127 * d, 32 * 127 * d
    h = g / (1 + np.exp(-g)) * u
    assert np.allclose(out["h"], h, rtol=1e-15)
    assert np.all(out["qh"] == -127)
    assert np.all(out["acc_d"] == -127 * 16 * (-2 + 1))
    dh = float(np.float32(np.float32(abs(h)) / np.float32(127)))
    assert np.allclose(out["o"], dh * 127 * 16, rtol=1e-12)


def test_int2_expert_equals_int8_container():
    # the same codes through the int2 and the int8 containers give identical results
    rng = np.random.default_rng(5)
    H, I = 64, 32
    gate, up = rng.integers(-2, 2, (I, H)), rng.integers(-2, 2, (I, H))
    down = rng.integers(-2, 2, (H, I))
    scales = rng.uniform(0.01, 0.1, 2 * I + H).astype(np.float32)
    qx, dx = oracle.q8_0_quantize(rng.standard_normal((3, H)).astype(np.float32))
    a = oracle.expert_ffn(_record(gate, up, down, 2), scales, H, I, 2, qx, dx)
    b = oracle.expert_ffn(_record(gate, up, down, 8), scales, H, I, 8, qx, dx)
    for key in ("acc_g", "acc_u", "acc_d", "qh", "dh", "o"):
        assert np.array_equal(a[key], b[key]), key


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_expert_matches_fp64_dequantised_products(bits):
    shape = {4: synth.TINY, 2: synth.TINY_INT2,
             8: synth.LayerShape(256, 16, 4, 2, 4, 128, 1, 128, 8, 2.5)}[bits]
    rec, sc = synth.expert_record(shape, 11, 0, "routed", 3)
    x = synth.token_batch(shape, 11, 0, range(6))
    qx, dx = oracle.q8_0_quantize(x)
    out = oracle.expert_ffn(rec, sc, shape.hidden, shape.inter, bits, qx, dx)
    ref = oracle.expert_ffn_dequant_fp64(rec, sc, shape.hidden, shape.inter, bits, x)
    assert np.allclose(out["o"], ref, rtol=1e-10, atol=1e-12 * np.abs(ref).max())


def test_h_error_bound_covers_fp32_evaluation():
    # evaluate g, u, h in fp32 (sequential order) and check the oracle's bound
    shape = synth.TINY
    rec, sc = synth.expert_record(shape, 12, 0, "routed", 1)
    x = synth.token_batch(shape, 12, 0, range(4))
    qx, dx = oracle.q8_0_quantize(x)
    out = oracle.expert_ffn(rec, sc, shape.hidden, shape.inter, 4, qx, dx)
    I = shape.inter
    g32 = np.zeros(out["g"].shape, np.float32)
    u32 = np.zeros(out["u"].shape, np.float32)
    for b in range(out["acc_g"].shape[2]):
        g32 += dx[:, None, b] * out["acc_g"][:, :, b].astype(np.float32)
        u32 += dx[:, None, b] * out["acc_u"][:, :, b].astype(np.float32)
    g32 *= sc[:I]
    u32 *= sc[I:2 * I]
    h32 = g32 / (np.float32(1) + np.exp(-g32)) * u32
    assert np.all(np.abs(h32 - out["h"]) <= out["h_err"])
