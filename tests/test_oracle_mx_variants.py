"""Pins of the oracle's E8M0 variants ("Unveiling the Potential of Quantization
with MXFP4 ...", Résumé technique §2 and §2A-§2B): 16-element E8M0 blocks, the
overflow-aware exponent rule (OAS) and the static macro-block scale (MBS),
checked against what the page and the arithmetic fix:

- OAS puts alpha_max / 2^e in (3.5, 7] (the page's interval), the OCP rule in
  [4, 8), at the interval ends, just inside and outside them and on subnormals;
- hand-worked blocks give the codes the interval implies;
- 16-element E8M0 blocks reduce to 32-element MXFP4 when both halves of every
  32-block share their exponent;
- the MBS macro scale is the nearest value with 8 fraction bits to alpha / 6,
  ties to even (exact rational brute force);
- MBS reduces to 16-element E8M0 when every macro scale is a power of two,
  scales with a macro block by powers of two, returns on-grid values exactly
  and zeroes an all-zero macro block.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import fp4q_oracle as o

MB = 128     # macro block length from the page, not from the oracle


def _f32(x):
    return np.float32(x)


def _boundary_amaxes():
    vals = []
    for k in (-140, -130, -127, -126, -20, -1, 0, 1, 7, 60, 124):
        for base in (1.0, 1.75, 3.5, 4.0, 7.0, 8.0, 6.0, 1.5):
            x = np.float32(base * 2.0 ** k) if -149 <= k + 3 else None
            if x is None or x == 0 or not np.isfinite(x):
                continue
            vals += [x, np.nextafter(x, np.float32(0)), np.nextafter(x, np.float32(np.inf))]
    rng = np.random.default_rng(11)
    vals += list((rng.random(4000) * np.exp2(rng.integers(-140, 120, 4000))).astype(np.float32))
    vals += [np.float32(np.finfo(np.float32).max), np.float32(2.0 ** -149)]
    a = np.array([v for v in vals if np.isfinite(v) and v > 0], dtype=np.float32)
    return a


def test_macro_block_length():
    assert o.MACRO_BLOCK == MB


def test_oas_interval():
    a = _boundary_amaxes()
    e = o.e8m0_exponent_oas(a)
    ratio = a.astype(np.float64) / np.exp2(e.astype(np.float64))      # exact: a power-of-two divisor
    inside = (e > -127) & (e < 127)
    assert np.all(ratio[inside] > 3.5) and np.all(ratio[inside] <= 7.0)
    # clamped at -127 only when even 2^-127 leaves the ratio at or below 7
    assert np.all(ratio[e == -127] <= 7.0)
    assert o.e8m0_exponent_oas(np.float32(0.0)) == -127


def test_ocp_interval_on_the_same_values():
    a = _boundary_amaxes()
    e = o.e8m0_exponent(a)
    ratio = a.astype(np.float64) / np.exp2(e.astype(np.float64))
    inside = (e > -127) & (e < 127)
    assert np.all(ratio[inside] >= 4.0) and np.all(ratio[inside] < 8.0)


def test_oas_worked_blocks():
    # alpha = 7 (exactly the top of the interval): e = 0, y = v, 7 saturates to 6
    x = np.zeros((1, 16), np.float32)
    x[0, 0], x[0, 1], x[0, 2] = 7.0, -3.25, 0.24
    r = o.quantize(x, "mxfp4_oas")["row"]
    assert r["scales"][0, 0] == 127
    c = o.unpack_nibbles(r["codes"])[0]
    assert (c[0], c[1], c[2]) == (7, 8 | 5, 0)            # 6, -3 (3.25 -> 3), 0
    # alpha = 7.5: e = 1, y = v / 2: 3.75 -> 4, -1.625 -> -1.5, 0.75 -> 1 (tie to even code 2)
    x[0, 0], x[0, 1], x[0, 2] = 7.5, -3.25, 1.5
    r = o.quantize(x, "mxfp4_oas")["row"]
    assert r["scales"][0, 0] == 128
    c = o.unpack_nibbles(r["codes"])[0]
    assert (c[0], c[1], c[2]) == (6, 8 | 3, 2)
    # the OCP rule keeps e = 0 for 7.5 and saturates it to 6
    r = o.quantize(x, "mxfp4_b16")["row"]
    assert r["scales"][0, 0] == 127
    assert o.unpack_nibbles(r["codes"])[0][0] == 7


def test_oas_never_saturates_more_than_ocp():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((64, 512)) * np.exp(rng.standard_normal((64, 1)))).astype(np.float32)
    y_oas = o.quantize(x, "mxfp4_oas", keep_y=True)["row"]["y"]
    y_ocp = o.quantize(x, "mxfp4_b16", keep_y=True)["row"]["y"]
    assert np.sum(np.abs(y_oas) > 6) < np.sum(np.abs(y_ocp) > 6)
    assert np.all(np.abs(y_oas) <= 7.0)


@pytest.mark.parametrize("rounding", ["rtne", "sr"])
def test_b16_reduces_to_mxfp4_when_halves_share_the_exponent(rounding):
    rng = np.random.default_rng(5)
    x = (rng.uniform(-1, 1, (8, 256)) * 2.0 ** rng.integers(-8, 8, (8, 1))).astype(np.float32)
    # both 16-halves of every 32-block get a maximum with the same binade
    for r in range(8):
        for b in range(8):
            e = int(rng.integers(-5, 5))
            x[r, 32 * b + 3] = np.float32(1.5 * 2.0 ** e)
            x[r, 32 * b + 16 + 7] = np.float32(-1.25 * 2.0 ** e)
            blk = x[r, 32 * b:32 * b + 32]
            np.clip(blk, -1.5 * 2.0 ** e, 1.5 * 2.0 ** e, out=blk)
    a = o.quantize(x, "mxfp4_b16", rounding=rounding, seed=4)["row"]
    b = o.quantize(x, "mxfp4", rounding=rounding, seed=4)["row"]
    assert np.array_equal(a["codes"], b["codes"])
    assert np.array_equal(a["scales"], np.repeat(b["scales"], 2, axis=1))


def _rn8_bruteforce(alpha: np.float32) -> Fraction:
    t = Fraction(float(alpha)) / 6
    if t == 0:
        return Fraction(0)
    e = t.numerator.bit_length() - t.denominator.bit_length()
    if Fraction(2) ** e > t:
        e -= 1
    q = Fraction(2) ** (max(e, -126) - 8)
    lo = (t // q) * q
    hi = lo + q
    if t - lo < hi - t:
        return lo
    if t - lo > hi - t:
        return hi
    return lo if (lo / q) % 2 == 0 else hi


def test_mbs_macro_scale_is_the_nearest_8_bit_value():
    rng = np.random.default_rng(9)
    alphas = list((rng.random(400) * np.exp2(rng.integers(-140, 120, 400))).astype(np.float32))
    # exact ties: alpha / 6 = (1 + (2j + 1) / 512) * 2^k, both neighbours 8-bit
    for j in (0, 1, 2, 100, 255):
        for k in (-130, -3, 0, 9):
            alphas.append(np.float32(6.0 * (1.0 + (2 * j + 1) / 512.0) * 2.0 ** k))
    alphas += [np.float32(0.0), np.float32(6.0), np.float32(np.finfo(np.float32).max), np.float32(2.0 ** -149)]
    for a in alphas:
        s = o.mbs_macro_scale(np.float32(a))
        assert Fraction(float(s)) == _rn8_bruteforce(np.float32(a)), a


def _planted_pow2(rows, cols, seed):
    """Every macro block's maximum is exactly 6 * 2^k, so S = 2^k."""
    rng = np.random.default_rng(seed)
    x = np.zeros((rows, cols), np.float32)
    for r in range(rows):
        for m in range(cols // MB):
            k = int(rng.integers(-10, 10))
            blk = (rng.standard_normal(MB) * 2.0 ** k).astype(np.float32)
            blk = np.clip(blk, -5.9 * 2.0 ** k, 5.9 * 2.0 ** k)
            blk[int(rng.integers(0, MB))] = np.float32(6.0 * 2.0 ** k)
            x[r, m * MB:(m + 1) * MB] = blk
    return x


@pytest.mark.parametrize("rounding", ["rtne", "sr"])
def test_mbs_reduces_to_b16_when_macro_scales_are_powers_of_two(rounding):
    x = _planted_pow2(6, 512, 3)
    mbs = o.quantize(x, "mxfp4_mbs", rounding=rounding, seed=7)["row"]
    b16 = o.quantize(x, "mxfp4_b16", rounding=rounding, seed=7)["row"]
    k = np.log2(mbs["macro_scales"].astype(np.float64))
    assert np.all(k == np.round(k))
    assert np.array_equal(mbs["codes"], b16["codes"])
    shift = np.repeat(k.astype(np.int64), MB // 16, axis=1)
    assert np.array_equal(mbs["scales"].astype(np.int64), b16["scales"].astype(np.int64) - shift)
    y1 = o.dequantize_mbs(mbs["codes"], mbs["scales"], mbs["macro_scales"])
    y2 = o.dequantize(b16["codes"], b16["scales"], 1.0, "mxfp4_b16")
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    assert mbs["stats"]["snr_db"] == pytest.approx(b16["stats"]["snr_db"], rel=1e-12)


@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("k", [-6, 4])
def test_mbs_power_of_two_scaling_of_one_macro_block(rht, k):
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((5, 384)) * np.exp(rng.standard_normal((1, 384)))).astype(np.float32)
    base = o.quantize(x, "mxfp4_mbs", rht=rht)["row"]
    y = x.copy()
    y[1, MB:2 * MB] *= np.float32(2.0 ** k)
    sc = o.quantize(y, "mxfp4_mbs", rht=rht)["row"]
    assert np.array_equal(sc["codes"], base["codes"])
    assert np.array_equal(sc["scales"], base["scales"])
    want = base["macro_scales"].copy()
    want[1, 1] = np.float32(want[1, 1] * np.float32(2.0 ** k))
    assert np.array_equal(sc["macro_scales"].view(np.uint32), want.view(np.uint32))


def test_mbs_on_grid_values_round_trip_exactly():
    rng = np.random.default_rng(12)
    rows, cols = 4, 256
    x = np.zeros((rows, cols), np.float64)
    for r in range(rows):
        for m in range(cols // MB):
            S = (1.0 + int(rng.integers(0, 256)) / 256.0) * 2.0 ** int(rng.integers(-12, 12))
            for b in range(MB // 16):
                e = 0 if b == 0 else int(rng.integers(-6, 1))
                kk = rng.integers(0, 8, 16)
                kk[int(rng.integers(0, 16))] = 7                      # every block reaches 6 * 2^e
                sign = np.where(rng.integers(0, 2, 16), -1.0, 1.0)
                c0 = m * MB + 16 * b
                x[r, c0:c0 + 16] = sign * o.E2M1_LEVELS[kk] * 2.0 ** e * S
    x32 = x.astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), x)
    res = o.quantize(x32, "mxfp4_mbs")["row"]
    back = o.dequantize_mbs(res["codes"], res["scales"], res["macro_scales"])
    assert np.array_equal(back, x32)
    assert np.isinf(res["stats"]["snr_db"])


def test_mbs_zero_macro_block():
    x = np.ones((2, 256), np.float32)
    x[1, MB:] = 0.0
    res = o.quantize(x, "mxfp4_mbs")["row"]
    assert res["macro_scales"][1, 1] == 0.0
    assert np.all(res["scales"][1, MB // 16:] == 0)
    assert np.all(o.unpack_nibbles(res["codes"])[1, MB:] == 0)
    # 1 / 6 = 1.0101...b * 2^-3; 8 fraction bits: 1.01010101b (0.333 of a step
    # rounds down) = 341 / 2048
    assert res["macro_scales"][0, 0] == np.float32(341.0 / 2048.0)


def test_mma_layout_repeats_32_element_scales():
    s = np.arange(12, dtype=np.uint8).reshape(2, 6)
    flat = o.scales_to_mma_layout(s, block=32)
    assert flat.size == o.mma_layout_bytes(2, 12)
    for r in range(2):
        for kb in range(6):
            for h in range(2):
                assert flat[o.mma_scale_offset(r, 2 * kb + h, 12)] == s[r, kb]


def test_mbs_gemm_reduces_to_b16_when_macro_scales_are_powers_of_two():
    """The oracle's GEMM on MBS copies equals its GEMM on the 16-element E8M0
    copies of the same tensors when every macro scale is a power of two."""
    a = _planted_pow2(4, 256, 21)
    b = _planted_pow2(3, 256, 22)
    mbs = o.gemm(o.quantize(a, "mxfp4_mbs")["row"], o.quantize(b, "mxfp4_mbs")["row"])
    b16 = o.gemm(o.quantize(a, "mxfp4_b16")["row"], o.quantize(b, "mxfp4_b16")["row"])
    assert np.array_equal(mbs, b16)


@pytest.mark.parametrize("fmt", ["nvfp4_2l", "mxfp4_mbs"])
def test_fp32_dequantisation_is_one_rounding_of_the_exact_value(fmt):
    """level * block scale is exact in FP32, so the FP32 dequantisation rounds
    the exact value (level * block scale * per-128 scale, exact in FP64) once."""
    rng = np.random.default_rng(31)
    x = (rng.standard_normal((16, 512)) * np.exp(2 * rng.standard_normal((16, 1)))).astype(np.float32)
    r = o.quantize(x, fmt, rht=True, seed=2)["row"]
    exact = o.dequantize_outer_f64(r)
    if fmt == "nvfp4_2l":
        got = o.dequantize_two_level(r["codes"], r["scales"], r["outer_scales"])
    else:
        got = o.dequantize_mbs(r["codes"], r["scales"], r["macro_scales"])
    assert np.array_equal(got.view(np.uint32), exact.astype(np.float32).view(np.uint32))
