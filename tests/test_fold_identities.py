"""Pins for two facts the reduce kernel's folds rely on, checked on the host
over every value they cover (a restatement of the arithmetic in numpy, not a
call into the kernel, whose results the GPU parity tests check against the
oracle).

1. bf16 min and max fold packed pairs of 16-bit order keys: the key of a bf16
   value x (x with its 15 magnitude bits flipped when the sign bit is set, as
   a signed 16-bit integer) orders all 65536 bf16 patterns exactly as the
   32-bit order key of their fp32 widenings does, ties included, with -0
   below +0; and the map is its own inverse.
2. The int32 trees over 16 slots pad positions past W with the op's identity:
   0 for sum, 1 for the wrapping product, INT32_MAX for min, INT32_MIN for
   max; combining with it on either side leaves every int32 value unchanged.
"""
import numpy as np


def key16(x):
    x = x.astype(np.uint16)
    flip = np.where(x & 0x8000, 0x7FFF, 0).astype(np.uint16)
    return (x ^ flip).view(np.int16)


def key32(b):
    b = b.astype(np.uint32)
    flip = np.where(b & 0x80000000, 0x7FFFFFFF, 0).astype(np.uint32)
    return (b ^ flip).view(np.int32)


def test_bf16_16_bit_keys_order_as_the_widened_32_bit_keys():
    x = np.arange(1 << 16, dtype=np.uint32)
    k16 = key16(x).astype(np.int64)
    k32 = key32(x << 16).astype(np.int64)
    # same strict order on every pair: both keys are strictly increasing in
    # the same permutation, so sorting by one sorts the other
    order = np.argsort(k16, kind="stable")
    assert np.all(np.diff(k16[order]) > 0)            # the 16-bit key is a bijection
    assert np.all(np.diff(k32[order]) > 0)
    # -0 (0x8000) sits just below +0 (0x0000)
    assert k16[0x8000] == -1 and k16[0x0000] == 0
    # the map is its own inverse on packed pairs, lane by lane
    pairs = (x[:, None] | (x[::-1, None] << 16)).astype(np.uint32).ravel()
    packed_key = pairs ^ (((pairs >> 15) & 0x00010001) * 0x7FFF)
    lo = packed_key & 0xFFFF
    hi = packed_key >> 16
    assert np.array_equal(lo.astype(np.uint16).view(np.int16), key16(pairs & 0xFFFF))
    assert np.array_equal(hi.astype(np.uint16).view(np.int16), key16(pairs >> 16))
    back = packed_key ^ (((packed_key >> 15) & 0x00010001) * 0x7FFF)
    assert np.array_equal(back, pairs)


def test_int32_identities_are_exact():
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.integers(-2**31, 2**31, 1 << 20, dtype=np.int64),
                        np.array([0, 1, -1, 2**31 - 1, -2**31], dtype=np.int64)]).astype(np.int32)
    u = a.view(np.uint32)
    one = np.uint32(1)
    assert np.array_equal(u + np.uint32(0), u) and np.array_equal(np.uint32(0) + u, u)
    assert np.array_equal(u * one, u) and np.array_equal(one * u, u)
    assert np.array_equal(np.minimum(a, np.int32(2**31 - 1)), a)
    assert np.array_equal(np.maximum(a, np.int32(-2**31)), a)
    assert np.array_equal(np.minimum(np.int32(2**31 - 1), a), a)
    assert np.array_equal(np.maximum(np.int32(-2**31), a), a)
