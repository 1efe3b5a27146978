"""The seeded input generator: Philox known answers, recipes, and the
agreement of its int4 packing with the oracle's independent unpacking."""
import numpy as np

import oracle
import synth


def test_philox4x32_10_known_answers():
    # known-answer vectors distributed with the Random123 reference code
    m = 0xFFFFFFFF
    cases = [((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
             ((m, m, m, m), (m, m), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
             ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
              (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1))]
    for ctr, key, out in cases:
        r = synth.philox4x32_10(*[[c] for c in ctr], *key)
        assert tuple(int(v[0]) for v in r) == out


def test_normal_int_offsets_and_stats():
    key = synth.make_key(0, "t")
    z = synth.normal_int(key, 200001)
    assert np.array_equal(synth.normal_int(key, 1000, start=12345), z[12345:13345])
    assert abs(z.mean()) < 0.01 * synth.SIGMA_Z
    assert abs(z.std() / synth.SIGMA_Z - 1) < 0.01


def test_weight_recipe_packs_like_oracle_unpacks():
    shape = synth.TINY
    for m in range(3):
        q, packed, scales = synth.expert_matrix(shape, 0, 0, "routed", 2, m)
        rows, k = q.shape
        assert np.array_equal(oracle.unpack_weight_rows(packed, rows, k, 4), q)
        assert np.abs(q).max(axis=1).tolist() == [7] * rows
        assert scales.dtype == np.float32 and np.all(scales > 0)


def test_int2_recipe_packs_like_oracle_unpacks():
    shape = synth.TINY_INT2
    for m in range(3):
        q, packed, scales = synth.expert_matrix(shape, 0, 0, "routed", 2, m)
        rows, k = q.shape
        assert packed.shape == (rows, k // 4)
        assert np.array_equal(oracle.unpack_weight_rows(packed, rows, k, 2), q)
        # all four codes of the container occur; the row maximum rounds to 2
        # and is clamped to 1
        assert sorted(np.unique(q).tolist()) == [-2, -1, 0, 1]
        assert scales.dtype == np.float32 and np.all(scales > 0)
    assert synth.GLM_INT2.record_bytes() == 3 * 6144 * 2048 // 4


def test_record_layout_and_sizes():
    for shape in (synth.TINY,):
        rec, sc = synth.expert_record(shape, 0, 0, "routed", 0)
        assert rec.size == shape.record_bytes() and sc.size == shape.scale_count()
    assert synth.GLM.record_bytes() + 4 * synth.GLM.scale_count() == 18915328


def test_keys_differ_per_tensor():
    ks = {synth.make_key(0, "expert", 0, "routed", e, m) for e in range(16) for m in range(3)}
    assert len(ks) == 48
