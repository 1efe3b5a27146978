"""Pins for the oracle's Q8_0, int4 and int2 code paths (hand-worked blocks,
closed forms and invariants)."""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_q8_0_hand_worked_blocks():
    cases = json.load(open(os.path.join(GOLD, "q8_0_blocks.json")))["blocks"]
    for c in cases:
        q, d = oracle.q8_0_quantize(np.array(c["x"], np.float32))
        assert d.tolist() == [c["d"]], c["why"]
        assert q.tolist() == c["q"], c["why"]


def test_q8_0_invariants_random():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 256)) * rng.uniform(1e-3, 1e3, (64, 1))).astype(np.float32)
    q, d = oracle.q8_0_quantize(x)
    xb = x.reshape(64, 8, 32).astype(np.float64)
    qb = q.reshape(64, 8, 32).astype(np.int64)
    d64 = d.astype(np.float64)[..., None]
    # reconstruction error at most half a step (plus fp32 rounding of d, inv)
    assert np.all(np.abs(xb - d64 * qb) <= d64 * (0.5 + 2e-6))
    # the largest magnitude element maps to +-127, codes stay in range
    amax_pos = np.abs(xb).argmax(axis=-1)
    assert np.all(np.abs(np.take_along_axis(qb, amax_pos[..., None], -1)) == 127)
    assert qb.min() >= -127 and qb.max() <= 127
    # sign is preserved where the code is non-zero
    nz = qb != 0
    assert np.all(np.sign(qb[nz]) == np.sign(xb[nz]))
    # scale equals amax/127 in fp32
    assert np.array_equal(d, (np.abs(x.reshape(64, 8, 32)).max(-1) / np.float32(127)).astype(np.float32))


def test_q8_0_scale_invariance_power_of_two():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 64)).astype(np.float32)
    q1, d1 = oracle.q8_0_quantize(x)
    q2, d2 = oracle.q8_0_quantize(x * np.float32(8.0))
    assert np.array_equal(q1, q2)
    assert np.array_equal(d2, d1 * np.float32(8.0))


def test_q8_0_rejects_nonfinite_and_bad_shape():
    x = np.zeros(32, np.float32)
    x[3] = np.nan
    with pytest.raises(ValueError):
        oracle.q8_0_quantize(x)
    with pytest.raises(ValueError):
        oracle.q8_0_quantize(np.zeros(33, np.float32))


def test_int4_pack_hand_worked():
    cases = json.load(open(os.path.join(GOLD, "int4_pack.json")))["cases"]
    for c in cases:
        b = oracle.int4_pack(np.array(c["codes"]))
        assert b.tolist() == c["bytes"]
        assert oracle.int4_unpack(np.array(c["bytes"], np.uint8)).tolist() == c["codes"]


def test_int4_round_trip_all_codes_and_int8_container():
    codes = np.array([[a, b] for a in range(-8, 8) for b in range(-8, 8)]).reshape(1, -1)
    assert np.array_equal(oracle.int4_unpack(oracle.int4_pack(codes)), codes)
    # unpacked rows equal the same codes stored in the int8 container
    rows = oracle.unpack_weight_rows(oracle.int4_pack(codes).reshape(-1), 1, codes.shape[1], 4)
    rows8 = oracle.unpack_weight_rows(codes.astype(np.int8).view(np.uint8).reshape(-1), 1,
                                      codes.shape[1], 8)
    assert np.array_equal(rows, rows8)
    with pytest.raises(ValueError):
        oracle.int4_pack(np.array([9, 0]))


def test_int2_pack_hand_worked():
    cases = json.load(open(os.path.join(GOLD, "int2_pack.json")))["cases"]
    for c in cases:
        b = oracle.int2_pack(np.array(c["codes"]))
        assert b.tolist() == c["bytes"]
        assert oracle.int2_unpack(np.array(c["bytes"], np.uint8)).tolist() == c["codes"]


def test_int2_round_trip_all_codes_and_int8_container():
    # every byte value once: 256 bytes hold all 4^4 code quadruples
    codes = np.array([[(v >> (2 * m) & 3) - 2 for m in range(4)] for v in range(256)]).reshape(1, -1)
    b = oracle.int2_pack(codes)
    assert b.reshape(-1).tolist() == list(range(256))
    assert np.array_equal(oracle.int2_unpack(b), codes)
    rows = oracle.unpack_weight_rows(b.reshape(-1), 1, codes.shape[1], 2)
    rows8 = oracle.unpack_weight_rows(codes.astype(np.int8).view(np.uint8).reshape(-1), 1,
                                      codes.shape[1], 8)
    assert np.array_equal(rows, rows8)
    # element i of a row sits in byte i // 4 at bit 2 * (i % 4)
    one = np.full((1, 32), -2)
    one[0, 13] = 1
    bb = oracle.int2_pack(one)[0]
    assert bb.tolist() == [0, 0, 0, 3 << 2, 0, 0, 0, 0]
    with pytest.raises(ValueError):
        oracle.int2_pack(np.array([2, 0, 0, 0]))
    with pytest.raises(ValueError):
        oracle.int2_pack(np.array([0, 0]))


def test_stable_mask_flags_boundaries():
    # amax 127 -> inv 1: 2.5 sits on a boundary, 2.2 is far from one
    h = np.zeros(32)
    h[0] = 127.0
    h[1] = 2.5
    h[2] = 2.2
    m = oracle.q8_0_stable_mask(h, np.full(32, 1e-3))
    assert not m[1] and m[2] and m[0]
    assert oracle.q8_0_stable_mask(h, np.zeros(32))[2]
