"""The activation orders the C header states for packed weights, checked on
the CPU: with the oracle's packing, one byte-wise 4-way dot per 32-bit word
(unsigned weight fields against signed activation codes in the stated order)
minus the stated code-sum correction equals the oracle's exact block dot.
Pins the layout contract, not the kernels (those are checked on the GPU)."""
import numpy as np

import oracle

ORDER4 = [0, 2, 4, 6, 1, 3, 5, 7]                                  # per 8 codes
ORDER2 = [0, 4, 8, 12, 1, 5, 9, 13, 2, 6, 10, 14, 3, 7, 11, 15]   # per 16 codes


def _stored(x, order):
    g = len(order)
    return x.reshape(-1, g)[:, order].reshape(-1)


def _dot4(wbytes, abytes):
    """sum over 4 byte lanes of unsigned weight byte x signed activation byte"""
    return int(sum(int(w) * int(a) for w, a in zip(wbytes, abytes)))


def test_int4_order_gives_exact_block_dots():
    rng = np.random.default_rng(7)
    for _ in range(50):
        q = rng.integers(-8, 8, 32)
        x = rng.integers(-127, 128, 32)
        b = oracle.int4_pack(q)                        # 16 bytes
        a = _stored(x, ORDER4).astype(np.int64)        # 32 activation bytes, 8 words
        acc = 0
        for w in range(4):                             # weight word w: bytes 4w..4w+3
            wb = b[4 * w:4 * w + 4]
            acc += _dot4(wb & 0x0F, a[8 * w:8 * w + 4])        # low nibbles: word 2w
            acc += _dot4(wb >> 4, a[8 * w + 4:8 * w + 8])      # high nibbles: word 2w+1
        acc -= 8 * int(x.sum())
        assert acc == int(oracle.block_dots(q[None, :], x[None, :])[0, 0, 0])


def test_int2_order_gives_exact_block_dots():
    rng = np.random.default_rng(8)
    for _ in range(50):
        q = rng.integers(-2, 2, 32)
        x = rng.integers(-127, 128, 32)
        b = oracle.int2_pack(q)                        # 8 bytes
        a = _stored(x, ORDER2).astype(np.int64)
        acc = 0
        for h in range(2):                             # weight word h: bytes 4h..4h+3
            wb = b[4 * h:4 * h + 4].astype(np.int64)
            for m in range(4):                         # field m meets activation word 4h+m
                acc += _dot4((wb >> (2 * m)) & 3, a[16 * h + 4 * m:16 * h + 4 * m + 4])
        acc -= 2 * int(x.sum())
        assert acc == int(oracle.block_dots(q[None, :], x[None, :])[0, 0, 0])


def test_int2_fields_masked_in_place_are_exact_multiples():
    # the field-m products masked without shifting come out times 4^m and fit
    # the 8-bit lanes (max 3 * 64 = 192), so one exact shift per sum undoes it
    rng = np.random.default_rng(9)
    b = rng.integers(0, 256, 4)
    a = rng.integers(-127, 128, 4)
    for m in range(4):
        masked = b & (3 << (2 * m))
        assert masked.max() <= 192
        s = _dot4(masked, a)
        assert s % (4 ** m) == 0 and s // 4 ** m == _dot4((b >> (2 * m)) & 3, a)


def test_expert_parallel_record_index_multiply_high():
    # the kernels find expert e's local record e // ep_size as a multiply-high by
    # 2^32 // ep_size + 1 (2^32 without sharding): exact over the whole range
    # of expert ids and shard counts the library accepts (1024 each)
    for p in range(1, 1025):
        m = (1 << 32) if p == 1 else (1 << 32) // p + 1
        assert all((e * m) >> 32 == e // p for e in range(1024)), p
