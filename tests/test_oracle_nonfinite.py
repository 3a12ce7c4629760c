"""Pins of the oracle's quantisers on non-finite and subnormal input.

The CANN aclnnMoeDistributeDispatchV2 Formula section states the quantisers
for finite rows; on other input they follow IEEE binary32 arithmetic step by
step (the reading kept for every mode whose result stays well defined):

- per-token int8 (quantMode 2): Max(Abs(x)) skips NaN elements (a running
  greater-than maximum); an infinite element gives dynamicScales = 127/inf = 0,
  so every product is 0 or NaN and every code 0, with the sent scale 1/0 = inf;
  a row whose largest magnitude is subnormal overflows 127/amax to +inf, so its
  nonzero elements give +-inf products, clamped to +-127, its zeros give NaN
  products (0 x inf), converted to 0, and the sent scale is 1/inf = 0; a row of
  NaN only has amax 0 and is the all-zero row;
- static int8 (quantMode 1): +-inf saturate to 127 / -128, NaN converts to 0;
- MX (quantMode 4): a block holding +-inf has the exponent field 255, so
  sharedExp = 128 - emax, and the infinities saturate to the largest finite
  code; finite elements of that block shrink by 2^-(128 - emax) and round to
  (signed) zero unless large; an all-subnormal block takes sharedExp = -127;
  the block maximum skips NaN elements (the same running greater-than
  maximum), so a block's scale byte and its finite elements' codes come from
  its non-NaN elements alone, and a block of NaN only has sharedExp = -127.
  The code of a NaN element itself is left unspecified.

Every expected value below is worked from those rules and the format
definitions by hand, not produced by the oracle.
"""
import numpy as np

import oracle

INF, NINF, QNAN, NAN_LOW, NNAN = 0x7F80, 0xFF80, 0x7FC0, 0x7F81, 0xFFC1
ONE, TWO, NEG_TWO, HALF = 0x3F80, 0x4000, 0xC000, 0x3F00


def row(values, H=32):
    out = np.zeros(H, np.uint16)
    out[: len(values)] = values
    return out


def f32_bits(v):
    return int(np.array([v], np.float32).view(np.uint32)[0])


def test_int8_infinite_element_zeroes_the_row():
    q, inv = oracle.quant_int8_row(row([INF, ONE, NEG_TWO, 0, NINF]))
    assert np.all(q == 0)
    assert np.isposinf(inv)


def test_int8_subnormal_row_overflows_the_scale():
    # 2^-133 (bf16 0x0001) and -3 * 2^-133: amax = 3 * 2^-133, 127 / amax > FLT_MAX
    q, inv = oracle.quant_int8_row(row([0x0001, 0x8003, 0, 0x0002]))
    assert list(q[:4]) == [127, -127, 0, 127]
    assert np.all(q[4:] == 0)
    assert inv == 0.0 and not np.signbit(inv)


def test_int8_nan_elements_are_skipped_and_coded_zero():
    # amax over the non-NaN elements = 2, s = 63.5; 1.0 * 63.5 ties to 64
    q, inv = oracle.quant_int8_row(row([QNAN, TWO, ONE, NAN_LOW, NNAN, HALF]))
    assert list(q[:6]) == [0, 127, 64, 0, 0, 32]   # 0.5 * 63.5 = 31.75 -> 32
    assert f32_bits(inv) == f32_bits(np.float32(1.0) / np.float32(63.5))


def test_int8_all_nan_row_is_the_zero_row():
    q, inv = oracle.quant_int8_row(np.full(16, QNAN, np.uint16))
    assert np.all(q == 0)
    assert inv == 0.0


def test_int8_static_saturates_infinities_and_zeroes_nan():
    # 126.5 ties to 126, -127.5 ties to -128, 300 saturates (all exact in bf16)
    vals = oracle.bf16_from_f32([126.5, -127.5, 300.0])
    q = oracle.quant_int8_static_row(row([INF, NINF, QNAN, *vals], H=8), np.float32(1.0))
    assert list(q[:6]) == [127, -128, 0, 126, -128, 127]


def test_mx_block_with_infinity():
    x = row([INF, NINF, ONE, 0xBF80])   # +inf, -inf, 1.0, -1.0
    # e4m3: emax 8, sharedExp = 128 - 8 = 120, scale byte 247; inf -> 448 = 0x7E;
    # +-1.0 * 2^-120 is below half the smallest subnormal (2^-9): +0 / -0
    codes, sc = oracle.quant_mx_row(4, x)
    assert list(sc) == [247]
    assert list(codes[:4]) == [0x7E, 0xFE, 0x00, 0x80]
    assert np.all(codes[4:] == 0)
    # e5m2: emax 15, sharedExp 113, byte 240; inf -> 57344 = 0x7B
    codes, sc = oracle.quant_mx_row(5, x)
    assert list(sc) == [240]
    assert list(codes[:4]) == [0x7B, 0xFB, 0x00, 0x80]
    # e2m1: emax 2, sharedExp 126, byte 253; inf -> 6 = 0x7, -inf -> 0xF;
    # two codes per byte, element 2i in the low nibble
    codes, sc = oracle.quant_mx_row(6, x)
    assert list(sc) == [253]
    assert list(codes[:2]) == [0xF7, 0x80]


def test_mx_all_subnormal_block():
    # amax subnormal: sharedExp = -127, byte 0, values scaled by 2^127
    # 2^-133 * 2^127 = 2^-6: e4m3 smallest normal (exponent field 1) = 0x08;
    # 3 * 2^-133 -> 1.5 * 2^-5: e4m3 exponent field 2, mantissa 4 = 0x14
    x = row([0x0001, 0x8003])
    codes, sc = oracle.quant_mx_row(4, x)
    assert list(sc) == [0]
    assert list(codes[:2]) == [0x08, 0x94]
    # e2m1: 2^-6 and 1.5 * 2^-5 both round to zero (smallest step 0.5)
    codes, sc = oracle.quant_mx_row(6, x)
    assert list(sc) == [0]
    assert list(codes[:1]) == [0x80]


MINUS_0_296875 = 0xBE98   # -1.1875 * 2^-2, exact in bf16


def test_mx_block_maximum_skips_nan():
    # non-NaN elements: 1.0, -0.296875, 0.5 -> amax 1.0 (unbiased exponent 0);
    # the NaN payloads (magnitude bits above infinity's) take no part
    x = row([QNAN, ONE, MINUS_0_296875, NAN_LOW, NNAN, HALF])
    finite = [1, 2, 5]
    # e4m3: sharedExp = 0 - 8 = -8, byte 119 = 0x77; 1.0 * 2^8 = 256 = 0x78;
    # -76 ties between 72 and 80, even mantissa 80 -> 0xEA; 0.5 * 2^8 = 128 = 0x70
    codes, sc = oracle.quant_mx_row(4, x)
    assert list(sc) == [0x77]
    assert [codes[i] for i in finite] == [0x78, 0xEA, 0x70]
    assert np.all(codes[6:] == 0)
    # e5m2: sharedExp = -15, byte 112 = 0x70; 2^15 -> exponent field 30 = 0x78;
    # -9728 = -1.1875 * 2^13 rounds to -1.25 * 2^13 = 0xF1; 2^14 = 0x74
    codes, sc = oracle.quant_mx_row(5, x)
    assert list(sc) == [0x70]
    assert [codes[i] for i in finite] == [0x78, 0xF1, 0x74]
    # e2m1: sharedExp = -2, byte 125 = 0x7D; 4 = 0x6, -1.1875 -> -1.0 = 0xA,
    # 2 = 0x4 (element 2i in the low nibble of byte i)
    codes, sc = oracle.quant_mx_row(6, x)
    assert list(sc) == [0x7D]
    nib = [(codes[i // 2] >> (4 * (i & 1))) & 0xF for i in finite]
    assert nib == [0x6, 0xA, 0x4]


def test_mx_block_of_nan_only_takes_the_smallest_exponent():
    x = np.full(32, QNAN, np.uint16)
    x[7] = NNAN
    for q in (4, 5, 6):
        _, sc = oracle.quant_mx_row(q, x)
        assert list(sc) == [0]
