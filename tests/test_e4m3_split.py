"""The arithmetic the e4m3 tensor-core path rests on, checked exhaustively on
the host (no GPU, no library code): every value it feeds the MMAs is exact in
e4m3 and the pieces add back to the integers they came from.

e4m3 (sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is
subnormal, m * 2^-9) represents v exactly when v = M * 2^E with an integer
|M| < 16 and -9 <= E, and |v| <= 448. The kernels use:
  - activation q in [-127, 127]: lo = q & 15 and 16 * (q >> 4), and both / 4;
  - weight code u in {0, 1, 2} at bits 0-1 of a byte: the byte is u * 2^-9;
    at bits 2-3: u * 4 * 2^-9 (u = 2 sets the lowest exponent bit);
  - the epilogue's return from u to w = u - 1: isum = 2^9 * acc - s, with acc
    the accumulator (a multiple of 2^-9) and s the group's activation sum in
    [-16256, 16256], one f32 FMA that must be exact.
"""
import numpy as np
from fractions import Fraction


def e4m3_value(byte):
    sign = -1 if byte & 0x80 else 1
    e, m = (byte >> 3) & 15, byte & 7
    if e == 15 and m == 7:
        return None                                   # NaN
    if e == 0:
        return sign * Fraction(m, 512)
    return sign * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


E4M3 = {e4m3_value(b) for b in range(256)} - {None}


def test_activation_parts_exact():
    for q in range(-127, 128):
        lo, hi16 = q & 15, 16 * (q >> 4)
        assert lo + hi16 == q
        for v in (lo, hi16, Fraction(lo, 4), Fraction(hi16, 4)):
            assert Fraction(v) in E4M3, (q, v)


def test_weight_code_bytes():
    for u in (0, 1, 2):
        assert e4m3_value(u) == Fraction(u, 512)                 # bits 0-1
        assert e4m3_value(u << 2) == Fraction(4 * u, 512)        # bits 2-3
        # after >> 4 the slots 2 and 3 land on bits 0-1 and 2-3 again
        byte = (u << 4) | (u << 6)
        assert e4m3_value((byte >> 4) & 0x03) == Fraction(u, 512)
        assert e4m3_value((byte >> 4) & 0x0C) == Fraction(4 * u, 512)


def test_products_are_multiples_of_two_to_minus_nine():
    for u in (0, 1, 2):
        for q in range(-127, 128):
            lo, hi16 = q & 15, 16 * (q >> 4)
            # slot with factor 1 and slot with factor 4 (B divided by 4)
            assert Fraction(u, 512) * lo + Fraction(u, 512) * hi16 == Fraction(u * q, 512)
            assert (Fraction(4 * u, 512) * Fraction(lo, 4) + Fraction(4 * u, 512) * Fraction(hi16, 4)
                    == Fraction(u * q, 512))


def test_epilogue_correction_exact_in_f32():
    # acc = N * 2^-9 with |N| <= 128 * 2 * 127 (every u = 2, every |q| = 127);
    # 2^9 * acc is a power-of-two scaling, and N - s is an integer below 2^24
    # in magnitude, so f32 gives both exactly: isum = N - s.
    n = np.arange(-128 * 2 * 127, 128 * 2 * 127 + 1, dtype=np.int64)
    acc = (n.astype(np.float64) / 512).astype(np.float32)
    assert np.array_equal(acc.astype(np.float64) * 512, n.astype(np.float64))   # acc exact
    for sq in (-16256, -12345, -1, 0, 1, 9999, 16256):
        isum = acc * np.float32(512) + np.float32(-sq)                           # f32 ops
        assert isum.dtype == np.float32
        assert np.array_equal(isum.astype(np.int64), n - sq)


def test_accumulator_stays_exact_in_f32():
    # Every partial sum of a group (up to 128 products u * q * 2^-9 with
    # |u * q| <= 254) is N * 2^-9 with |N| below 2^15: at most 15 significant
    # bits, so f32 (24) holds every one exactly.
    bound = 128 * 2 * 127
    assert bound < 2 ** 15
