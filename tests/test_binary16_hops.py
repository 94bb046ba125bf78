"""The packed binary16 hop add of the fused pass rests on one fact: for
binary16 a and b, rounding the binary32 sum to binary16 gives the correctly
rounded binary16 sum (double rounding is innocuous when the wider format has
at least 2p + 2 significand bits: S. A. Figueroa, "When is double rounding
innocuous?", SIGNUM Newsletter 30(3), 1995; binary32 has 24 = 2*11 + 2).

Checked here against the exact sum: two binary16 values are multiples of
2^-24 below 2^17 in magnitude, so their binary64 sum is exact, and numpy
rounds binary64 to binary16 directly (one rounding)."""
import os

import numpy as np


def _check_pairs(a_bits, b_bits):
    a = a_bits.view(np.float16)
    b = b_bits.view(np.float16)
    with np.errstate(over="ignore", invalid="ignore"):
        twice = (a.astype(np.float32) + b.astype(np.float32)).astype(np.float16)
        once = (a.astype(np.float64) + b.astype(np.float64)).astype(np.float16)
    nan = np.isnan(once)
    assert np.array_equal(np.isnan(twice), nan)
    bad = np.nonzero(twice.view(np.uint16)[~nan] != once.view(np.uint16)[~nan])[0]
    assert bad.size == 0, (a[~nan][bad[:4]], b[~nan][bad[:4]])


def _b_set():
    """Every sign and exponent with the mantissas that sit at rounding
    boundaries, plus random patterns."""
    sign_exp = np.arange(64, dtype=np.uint16) << np.uint16(10)
    mant = np.array([0, 1, 2, 3, 0x1FE, 0x1FF, 0x200, 0x201, 0x3FC, 0x3FD, 0x3FE, 0x3FF], dtype=np.uint16)
    edges = (sign_exp[:, None] | mant[None, :]).ravel()
    rnd = np.random.default_rng(16).integers(0, 1 << 16, 256).astype(np.uint16)
    return np.unique(np.concatenate([edges, rnd]))


def test_double_rounded_binary16_sum_is_correctly_rounded():
    a = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    if os.environ.get("DDL_SLOW_TESTS"):
        for hi in range(0, 1 << 16, 256):
            b = np.arange(hi, hi + 256, dtype=np.uint32).astype(np.uint16)
            _check_pairs(np.repeat(a, b.size), np.tile(b, a.size))
        return
    b = _b_set()
    for part in np.array_split(b, 4):
        _check_pairs(np.repeat(a, part.size), np.tile(part, a.size))


def test_widened_sum_is_not_always_exact_in_binary32():
    """The last add of a binary16 fold stays binary32 for this reason: a
    binary16 sum can need more than 24 bits, so fl32(a + b) can differ from
    a + b (here 2048 + 2^-24)."""
    a = np.float16(2048.0)
    b = np.array([1], dtype=np.uint16).view(np.float16)[0]
    assert float(np.float32(a) + np.float32(b)) != float(a) + float(b)
