"""Pins for group-scaled int4 weights ("gs64": one fp32 scale per 64 weights
of a row) in the oracle and in the input generator."""
import numpy as np

import oracle
import synth


def _record(gate, up, down):
    return np.concatenate([oracle.int4_pack(gate).reshape(-1), oracle.int4_pack(up).reshape(-1),
                           oracle.int4_pack(down).reshape(-1)])


def test_gs64_gate_closed_form_locates_the_group():
    # H = 128 (two groups, four Q8_0 blocks), all gate codes 1, x block b all
    # equal to b + 1: every block quantises to codes 127 with d_b = (b+1)/127,
    # so dot_b = 32*127 and g[r] = 32*127*(s[r,0]*(d_0+d_1) + s[r,1]*(d_2+d_3)).
    # A group index of b % 2 instead of b // 2, or the groups of a row stored
    # column-major, gives a different value.
    H, I = 128, 64
    gate = np.ones((I, H), np.int8)
    up = np.ones((I, H), np.int8)
    down = np.ones((H, I), np.int8)
    r = np.arange(I, dtype=np.float64)
    sg = np.stack([0.01 * (r + 1), 0.03 * (r + 2)], axis=1).astype(np.float32)     # [I, 2]
    su = np.full((I, 2), 0.5, np.float32)
    sd = np.full((H, 1), 0.25, np.float32)
    scales = np.concatenate([sg.reshape(-1), su.reshape(-1), sd.reshape(-1)])
    x = np.repeat(np.arange(1, 5, dtype=np.float32), 32)[None, :]
    qx, dx = oracle.q8_0_quantize(x)
    assert np.all(qx == 127)
    out = oracle.expert_ffn(_record(gate, up, down), scales, H, I, 4, qx, dx, group=64)
    d = dx[0].astype(np.float64)
    want = 32 * 127 * (sg[:, 0].astype(np.float64) * (d[0] + d[1]) + sg[:, 1].astype(np.float64) * (d[2] + d[3]))
    assert np.allclose(out["g"][0], want, rtol=1e-14)
    want_u = 32 * 127 * 0.5 * d.sum()
    assert np.allclose(out["u"][0], want_u, rtol=1e-14)


def test_gs64_equal_group_scales_reduce_to_per_row():
    # a row whose groups all carry the row's scale is the per-row format
    shape = synth.TINY
    rec, s_row = synth.expert_record(shape, 21, 0, "routed", 2)
    H, I = shape.hidden, shape.inter
    s_g, s_u, s_d = s_row[:I], s_row[I:2 * I], s_row[2 * I:]
    grp = np.concatenate([np.repeat(s_g, H // 64), np.repeat(s_u, H // 64), np.repeat(s_d, I // 64)])
    x = synth.token_batch(shape, 21, "gs64", range(3))
    qx, dx = oracle.q8_0_quantize(x)
    a = oracle.expert_ffn(rec, s_row, H, I, 4, qx, dx)
    b = oracle.expert_ffn(rec, grp, H, I, 4, qx, dx, group=64)
    for k in ("acc_g", "acc_u", "acc_d", "qh"):
        assert np.array_equal(a[k], b[k]), k
    assert np.allclose(a["o"], b["o"], rtol=1e-12, atol=0)


def test_gs64_layout_against_dense_dequantised_matrices():
    # the scale array is [gate rows x H/64 | up rows x H/64 | down rows x I/64],
    # each row-major: rebuild W = s * q densely from that description and
    # compare the oracle's g, u and o with plain fp64 matrix products
    shape = synth.TINY_GS64
    H, I = shape.hidden, shape.inter
    rec, sc = synth.expert_record(shape, 22, 0, "routed", 5)
    wg = oracle.unpack_weight_rows(rec[:I * H // 2], I, H, 4).astype(np.float64)
    wu = oracle.unpack_weight_rows(rec[I * H // 2:I * H], I, H, 4).astype(np.float64)
    wd = oracle.unpack_weight_rows(rec[I * H:], H, I, 4).astype(np.float64)
    n = I * H // 64
    Wg = np.empty_like(wg)
    Wu = np.empty_like(wu)
    Wd = np.empty_like(wd)
    for row in range(I):
        for k in range(H):
            Wg[row, k] = wg[row, k] * float(sc[row * (H // 64) + k // 64])
            Wu[row, k] = wu[row, k] * float(sc[n + row * (H // 64) + k // 64])
    for row in range(H):
        for k in range(I):
            Wd[row, k] = wd[row, k] * float(sc[2 * n + row * (I // 64) + k // 64])
    x = synth.token_batch(shape, 22, "gs64", range(2))
    qx, dx = oracle.q8_0_quantize(x)
    out = oracle.expert_ffn(rec, sc, H, I, 4, qx, dx, group=64)
    xs = oracle.q8_0_dequantize(qx, dx)
    assert np.allclose(out["g"], xs @ Wg.T, rtol=1e-12, atol=1e-15)
    assert np.allclose(out["u"], xs @ Wu.T, rtol=1e-12, atol=1e-15)
    hs = oracle.q8_0_dequantize(out["qh"], out["dh"])
    assert np.allclose(out["o"], hs @ Wd.T, rtol=1e-12, atol=1e-15)


def test_gs64_generator_groups():
    # every 64-element group is quantised on its own maximum: the group's
    # largest |code| is qmax and every code is within half a step
    shape = synth.TINY_GS64
    q, _, s = synth.expert_matrix(shape, 23, 0, "routed", 1, 0)
    key = synth.expert_matrix_key(23, 0, "routed", 1, 0)
    z = synth.normal_int(key, q.size).reshape(q.shape).astype(np.float64)
    g = z.reshape(q.shape[0], -1, 64)
    amax = np.abs(g).max(axis=2)
    qg = q.reshape(g.shape).astype(np.int64)
    assert np.all(np.abs(qg).max(axis=2) == 7)
    assert np.all(np.abs(qg - 7 * g / amax[:, :, None]) <= 0.5)
    assert s.shape == (q.shape[0] * (q.shape[1] // 64),)
    c = synth.WEIGHT_STD / (synth.SIGMA_Z * 7)
    assert np.array_equal(s, (amax.reshape(-1) * c).astype(np.float32))
    assert synth.TINY_GS64.scale_count() == 3 * 128 * 256 // 64
    assert synth.GLM_GS64.scale_count() * 4 * 8 == synth.GLM.record_bytes()   # 12.5 % of the codes' bytes
