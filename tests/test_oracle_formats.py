"""Pins of the oracle's number formats against the format definitions,
brute force and an independent library routine (no GPU)."""
import math
import os
import struct

import numpy as np
import pytest
import torch

from oracle import fp4q_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_grids_match_golden():
    for fmt, code, mag in _read_golden("grids.txt"):
        if fmt == "e2m1":
            assert o.E2M1_LEVELS[int(code)] == float(mag)
        else:  # E1M2 in its own units: integer-unit level / 4
            assert o.UFP4_LEVELS[int(code)] / 4.0 == float(mag)


@pytest.mark.parametrize("fmt", ["nvfp4", "ufp4"])
def test_every_code_round_trips(fmt):
    codes = np.arange(16, dtype=np.uint8)
    vals = o.code_value(codes, fmt)
    # -0.0 for code 8 keeps its sign (reading R4)
    vals = np.where(codes == 8, -0.0, vals).astype(np.float32)
    assert np.array_equal(o.round_rtne(vals, fmt), codes)


def test_rtne_ties_golden():
    for fmt, x, expect in _read_golden("rtne_ties.txt"):
        f = "nvfp4" if fmt == "e2m1" else "ufp4"
        for s in (1.0, -1.0):
            c = o.round_rtne(np.array([s * float(x)], dtype=np.float32), f)
            assert o.code_value(c, f)[0] == s * float(expect), (fmt, x)


def _brute_rtne(a, levels):
    """argmin over all levels in exact rational arithmetic, ties to even index."""
    from fractions import Fraction
    fa = Fraction(min(a, levels[-1]))
    best = None
    for i, lv in enumerate(levels):
        d = abs(Fraction(lv) - fa)
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


@pytest.mark.parametrize("fmt", ["nvfp4", "ufp4"])
def test_exhaustive_bf16_in_one_block(fmt):
    """Every finite BF16 value with |x| <= Qmax, placed in a block whose amax is
    Qmax inside a tensor whose amax is Qmax*448: then g = 1, s_b = 1, y = x and
    the code must be the brute-force nearest level (ties to even)."""
    qmax = o.QMAX[fmt]
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = o.bf16_bits_to_f32(bits)
    x = x[np.isfinite(x) & (np.abs(x) <= qmax)]
    n = x.size
    m = np.zeros((n + 1, 16), dtype=np.float32)
    m[:n, 0] = x
    m[:n, 1] = qmax
    m[n, 0] = qmax * 448.0
    out = o.quantize_copy(m, fmt)
    assert out["tensor_scale"] == np.float32(1.0)
    codes = o.unpack_nibbles(out["codes"])[:n, 0]
    scales = out["scales"][:n, 0]
    assert np.all(o.e4m3_decode(scales) == 1.0)
    levels = [float(v) for v in o.grid_levels(fmt)]
    for xi, ci in zip(x.tolist(), codes.tolist()):
        k = _brute_rtne(abs(xi), levels)
        sign = 1 if math.copysign(1.0, xi) < 0 else 0
        assert ci == (sign << 3 | k), (xi, ci, k)


def test_e4m3_table_definition():
    v = o.E4M3_VALUES
    assert v.size == 127 and v[0] == 0.0 and v[1] == 2.0 ** -9 and v[-1] == 448.0
    assert np.all(np.diff(v) > 0)
    assert v[8] == 2.0 ** -6  # smallest normal
    # every finite code round-trips
    assert np.array_equal(o.e4m3_encode_rne_sat(v.astype(np.float32)), np.arange(127))


def _torch_e4m3(t32):
    return torch.from_numpy(t32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_against_library_cast():
    """torch's float8_e4m3fn cast (an independent RNE implementation) agrees
    on every value, every midpoint, one FP32 ulp either side of every midpoint,
    and 2^20 log-uniform samples in [2^-12, 448]."""
    v = o.E4M3_VALUES
    mids = (v[:-1] + v[1:]) / 2.0
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)  # midpoints are exact in FP32
    rng = np.random.default_rng(5)
    samples = np.exp2(rng.uniform(-12.0, np.log2(448.0), 1 << 20)).astype(np.float32)
    t = np.concatenate([v.astype(np.float32), m32,
                        np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(1e9)),
                        samples]).astype(np.float32)
    t = t[t <= 448.0]
    assert np.array_equal(o.e4m3_encode_rne_sat(t), _torch_e4m3(t))


def test_e4m3_saturates():
    t = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e30, np.inf], dtype=np.float32)
    assert np.all(o.e4m3_encode_rne_sat(t) == 126)


def _floor_log2_bits(a: float) -> int:
    """floor(log2 a) of a positive FP32 number from its IEEE bit fields."""
    b = struct.unpack("<I", struct.pack("<f", a))[0]
    e = (b >> 23) & 0xFF
    m = b & 0x7FFFFF
    if e == 0:
        return m.bit_length() - 1 - 149
    return e - 127


def test_e8m0_exponent():
    for k in range(-126, 128):
        a = np.float32(2.0 ** k)
        assert o.e8m0_exponent(a) == max(-127, min(127, k - 2))
        a2 = np.float32(2.0 ** k * (2.0 - 2.0 ** -23))
        if np.isfinite(a2):
            assert o.e8m0_exponent(a2) == max(-127, k - 2)
    assert o.e8m0_exponent(np.float32(0.0)) == -127
    assert o.e8m0_exponent(np.float32(6.0)) == 0
    assert o.e8m0_exponent(np.float32(2.0 ** -149)) == -127
    rng = np.random.default_rng(7)
    a = np.abs(rng.standard_normal(20000).astype(np.float32)) * np.float32(3.0)
    a = np.concatenate([a, np.float32(1e-40) * np.arange(1, 200, dtype=np.float32)])
    a = a[a > 0]
    e = o.e8m0_exponent(a)
    ref = np.array([max(-127, _floor_log2_bits(float(x)) - 2) for x in a])
    assert np.array_equal(e, ref)
    normal = a >= 2.0 ** -120
    ratio = a[normal].astype(np.float64) / np.exp2(e[normal].astype(np.float64))
    # the block amax lands in [4, 8): values above 6 saturate on the E2M1 grid
    assert np.all((ratio >= 4.0) & (ratio < 8.0))


def test_bf16_widen_and_round():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = o.bf16_bits_to_f32(bits)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    fin = np.isfinite(t)
    assert np.array_equal(x[fin].view(np.uint32), t[fin].view(np.uint32))
    rng = np.random.default_rng(3)
    f = rng.standard_normal(1 << 16).astype(np.float32) * np.float32(1e3)
    rb = o.f32_to_bf16_bits_rne(f)
    tb = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(rb, tb)
