"""Exactness of the level arithmetic the dequantising kernels use, checked on
the host for every scale code.

The GEMM's converters and the dequantisation kernel form a uniform level k
(0..7) times a block scale s as one fused multiply-add on a magic-number word:
fma(B + 16 k, s / 16, -B s / 16) = k s, with B = 1024 in FP16, 128 in BF16 and
2^23 in FP32. That equals the plain product k s bit for bit when s / 16 and
B s / 16 are exact in the format and k s is representable in it: the fused
operation then rounds an exact value once. These tests check those three
conditions, and the identity itself in exact arithmetic, for every E4M3 scale
(UFP4, FP16 and FP32) and every E6M2 scale with each halving shift (HiF4,
BF16). The scale sets are the formats' value sets: E4M3 as in the OCP FP8
definition (bias 7, no infinities, 0x7F NaN), E6M2 as HiF4's scale ("Unleashing
Low-Bit Inference on Ascend NPUs: A Comprehensive Evaluation of HiFloat
Formats", Resumen tecnico §2; bias 31, exponent field 0 subnormal)."""
from fractions import Fraction

import numpy as np
import pytest


def e4m3_values():
    vals = []
    for c in range(0x7F):                     # 0x7F is NaN
        e, m = c >> 3, c & 7
        vals.append(Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return vals


def e6m2_values():
    vals = []
    for c in range(256):
        e, m = c >> 2, c & 3
        vals.append(Fraction(m) * Fraction(2) ** -32 if e == 0 else (1 + Fraction(m, 4)) * Fraction(2) ** (e - 31))
    return vals


def representable(x, mant_bits, emin, emax):
    """x exactly representable in a binary format with `mant_bits` fraction
    bits, normal exponents emin..emax and subnormals below 2^emin."""
    if x == 0:
        return True
    a = abs(x)
    if a >= Fraction(2) ** (emax + 1):
        return False
    e = emin
    while a >= Fraction(2) ** (e + 1):
        e += 1
    ulp = Fraction(2) ** (e - mant_bits)
    return (a / ulp).denominator == 1


FP16 = (10, -14, 15)
BF16 = (7, -126, 127)
FP32 = (23, -126, 127)


def check_magic(s, base, fmt):
    m, c = s / 16, -base * s / 16
    assert representable(m, *fmt) and representable(c, *fmt)
    assert representable(Fraction(base + 16 * 7), *fmt) and representable(Fraction(base), *fmt)
    for k in range(8):
        a = Fraction(base + 16 * k)
        assert a * m + c == k * s                  # the identity, exactly
        assert representable(k * s, *fmt)         # so the one rounding is exact


def test_e4m3_value_set():
    v = e4m3_values()
    assert len(v) == 127 and max(v) == 448 and min(x for x in v if x) == Fraction(1, 512)
    assert all(b > a for a, b in zip(v, v[1:]))


def test_e6m2_value_set():
    v = e6m2_values()
    assert v[124] == 1 and v[255] == Fraction(7, 4) * 2 ** 32 and v[1] == Fraction(1, 2 ** 32)


@pytest.mark.parametrize("fmt,base", [(FP16, 1024), (FP32, 2 ** 23)])
def test_ufp4_levels_every_e4m3_scale(fmt, base):
    """UFP4 on the 16-bit contraction (FP16) and in the dequantisation (FP32)."""
    for s in e4m3_values():
        check_magic(s, base, fmt)


def test_hif4_levels_every_e6m2_scale_and_shift():
    """HiF4 on the 16-bit contraction: BF16, the step S 2^-(d_8 + d_4)."""
    for S in e6m2_values():
        for shift in range(3):
            check_magic(S * Fraction(2) ** -shift, 128, BF16)


def test_magic_words_are_the_bit_patterns_used():
    """The high bytes the kernels OR in: 0x6400 is 1024 in FP16, 0x4300 is 128
    in BF16 (the top half of FP32 128), 0x4B000000 is 2^23 in FP32; the
    magnitude goes into bits 4-6, i.e. adds 16 k."""
    assert np.frombuffer(np.uint16(0x6400 | (5 << 4)).tobytes(), np.float16)[0] == 1024 + 16 * 5
    assert np.frombuffer(np.uint32((0x4300 | (5 << 4)) << 16).tobytes(), np.float32)[0] == 128 + 16 * 5
    assert np.frombuffer(np.uint32(0x4B000000 | (5 << 4)).tobytes(), np.float32)[0] == 2 ** 23 + 16 * 5


def test_a_plausible_slip_fails():
    """B = 128 with FP16's step (16 k added to 1024's neighbour) would not give
    k s: the checks above are not vacuous."""
    s = Fraction(3, 2)
    assert Fraction(1024 + 16 * 3) * (s / 16) - 128 * s / 16 != 3 * s
