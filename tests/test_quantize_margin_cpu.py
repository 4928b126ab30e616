"""The quantize kernel's fast path, checked on its arithmetic premise (no GPU needed).

The kernel rounds y = x * rcp(s) to the nearest integer and sends a value down the
exact path only when y lies within 2^-16 of a half-integer.  That is safe when the
exact quotient q = x / s of two fp16 numbers is either a half-integer or more than
2^-13 from every half-integer: y is within 2^-17.6 of q for |q| < 16 (a reciprocal
within 2 ulp, relative error at most 2^-22, and one rounded product), so outside the band y and q
round alike, and a true tie always lands inside the band.  This test checks that
premise by brute force over every positive fp16 x and every normal fp16 scale s with
x / s <= 7.5, in exact integer arithmetic.
"""
from __future__ import annotations

import numpy as np


def _fp16_in_units_of_2_pow_minus_24() -> np.ndarray:
    """Every positive finite fp16 value as an integer multiple of 2^-24 (index = bit pattern)."""
    h = np.arange(1, 0x7C00, dtype=np.int64)
    e, f = h >> 10, h & 0x3FF
    return np.where(e == 0, f, (1024 + f) << np.maximum(e - 1, 0))


def test_fp16_quotients_are_ties_or_clear_of_them():
    X = _fp16_in_units_of_2_pow_minus_24()
    assert X[-1] == 65504 * 2 ** 24 and X[0] == 1  # largest finite and smallest subnormal
    normal_S = X[0x400 - 1:]  # bit patterns 0x0400 .. 0x7BFF
    worst = np.inf
    ties = 0
    for c in range(0, normal_S.size, 512):
        S = normal_S[c:c + 512, None]
        Xs = X[None, :np.searchsorted(X, 15 * int(S[-1, 0]) // 2, side="right")]
        ok = 2 * Xs <= 15 * S  # x / s <= 7.5: the range the fast path accepts
        k = Xs // S
        r = 2 * Xs - (2 * k + 1) * S  # q - (k + 1/2) = r / (2 S)
        ties += int(np.count_nonzero(ok & (r == 0)))
        off = ok & (r != 0)
        # distance |r| / (2 S) must exceed 2^-13, i.e. 4096 |r| > S
        assert np.all(4096 * np.abs(r[off]) > np.broadcast_to(S, r.shape)[off])
        d = np.abs(r[off]) / (2.0 * np.broadcast_to(S, r.shape)[off])
        if d.size:
            worst = min(worst, float(d.min()))
    assert ties > 0  # true ties occur (e.g. x = 2.5 s) and must take the exact path
    assert worst > 2.0 ** -13
    # the reciprocal-and-multiply error for |q| < 16 stays inside the gap to the band
    err = 16 * (2.0 ** -22 + 2.0 ** -24 + 2.0 ** -46)
    assert err < 2.0 ** -17.6 and err < 2.0 ** -16 and 2.0 ** -13 - err > 2.0 ** -16
    # the quantize kernel's fused form: p = x * rcp(s) unrounded (rcp within 2 ulp) is within
    # |q| 2^-23 < 2^-19 of q, and e = fma(x, rcp(s), -r) is p - r within 2^-26, so a fast-path
    # value (|e| <= 1/2 - 2^-16) lies strictly nearer to r than 1/2: r is its code
    assert 16 * 2.0 ** -23 <= 2.0 ** -19 and 0.5 - 2.0 ** -16 + 2.0 ** -26 + 2.0 ** -19 < 0.5


def test_group_quotients_stay_below_16():
    # the scale is fp16(fp32(amax) / 7) (1 when that rounds to zero), so for every finite
    # fp16 amax the largest quotient amax / s of its group stays below 16; it exceeds 7
    # only by the fp16 rounding of the scale, and only subnormal scales go far past 7.49
    h = np.arange(1, 0x7C00, dtype=np.uint16)
    amax = h.view(np.float16).astype(np.float32)
    s = (amax / np.float32(7.0)).astype(np.float16).astype(np.float64)
    s[s == 0] = 1.0
    q = amax.astype(np.float64) / s
    assert q.max() < 16
    normal = s >= 2.0 ** -14
    assert q[normal].max() <= 7 * (1 + 2.0 ** -11) and q.max() > 7.49  # the subnormal case needs the slow path


def test_scale_by_reciprocal_multiply_equals_the_division():
    # The quantize kernel forms the scale as fp16_rne(amax * fp32(1/7)) instead of
    # fp16_rne(fp32_rn(amax / 7)).  amax is a non-negative fp16 value, so checking every
    # one of them (subnormals, the largest finite value and +inf included) proves the two
    # equal; both sides use IEEE round-to-nearest fp32 arithmetic.
    h = np.arange(0, 0x7C01, dtype=np.uint16)
    amax = h.view(np.float16).astype(np.float32)
    inv7 = np.array([0x3E124925], np.uint32).view(np.float32)[0]
    assert inv7 == np.float32(1.0) / np.float32(7.0)
    by_div = (amax / np.float32(7.0)).astype(np.float16).view(np.uint16)
    by_mul = (amax * inv7).astype(np.float16).view(np.uint16)
    assert np.array_equal(by_div, by_mul)
    # the fp32 results themselves do differ for some amax: the equality is a property of
    # the fp16 rounding, not of the fp32 arithmetic
    assert np.any((amax / np.float32(7.0)) != (amax * inv7))


def test_nibble_packing_by_shift_adds():
    # On the quantize kernel's fast path a nibble n in [1, 15] comes as the fp32 bit pattern of
    # 1.5 * 2^23 + n, i.e. 0x4B400000 | n, with bits 4 .. 21 zero; the kernel joins four of them
    # as (m0 + 16 m1) + 256 (m2 + 16 m3) modulo 2^32 and keeps the low 16 bits.  Every
    # combination of four nibbles must land in place.
    import itertools
    import struct
    pat = {n: struct.unpack("<I", struct.pack("<f", 12582912.0 + n))[0] for n in range(1, 16)}
    assert all(pat[n] == (0x4B400000 | n) for n in pat)
    for n0, n1, n2, n3 in itertools.product(range(1, 16), repeat=4):
        b0 = (pat[n0] + 16 * pat[n1]) & 0xFFFFFFFF
        b1 = (pat[n2] + 16 * pat[n3]) & 0xFFFFFFFF
        h = (b0 + 256 * b1) & 0xFFFFFFFF
        assert h & 0xFFFF == n0 | n1 << 4 | n2 << 8 | n3 << 12
