"""Pins of the oracle's two-level NVFP4 (the double-block scale of TetraJet-v2,
Riepilogo Tecnico §2A: a 128-element outer block scaled on its own, 16-element
inner blocks with E4M3 scales), checked against what the method fixes rather
than against the function's own formula:

- when every outer block's amax equals the tensor amax, the outer scale is the
  tensor scale and the result is the (separately pinned) NVFP4 result;
- scaling one outer block by 2^k scales its outer scale by 2^k and changes no
  code and no inner scale, and leaves the other outer blocks alone;
- values built on the grid (q * s_b * g_o with E4M3 s_b and power-of-two g_o)
  come back exactly, with infinite SNR;
- an all-zero outer block has scale 0 and zero scales and codes.
"""
import numpy as np
import pytest

from oracle import fp4q_oracle as o

OB = 128     # outer block length from the page, not from the oracle


def test_outer_block_length():
    assert o.OUTER_BLOCK == OB


def _planted(rows, cols, amax, seed):
    """|x| < amax everywhere, and +-amax at one position in the first half of
    every 128-element outer block (so any other outer-block size breaks it)."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, cols)) * 0.2 * amax).astype(np.float32)
    x = np.clip(x, -0.9 * amax, 0.9 * amax).astype(np.float32)
    for r in range(rows):
        for ob in range(cols // OB):
            j = ob * OB + int(rng.integers(0, OB // 2))
            x[r, j] = np.float32(amax if rng.integers(0, 2) else -amax)
    return x


@pytest.mark.parametrize("rounding", ["rtne", "sr"])
def test_reduces_to_nvfp4_when_outer_amax_is_the_tensor_amax(rounding):
    x = _planted(12, 512, 3.75, 1)
    two = o.quantize(x, "nvfp4_2l", rounding=rounding, seed=9)["row"]
    one = o.quantize(x, "nvfp4", rounding=rounding, seed=9)["row"]
    assert np.all(two["outer_scales"] == one["tensor_scale"])
    assert np.array_equal(two["codes"], one["codes"])
    assert np.array_equal(two["scales"], one["scales"])
    assert two["stats"]["snr_db"] == pytest.approx(one["stats"]["snr_db"], rel=1e-12)
    assert two["stats"]["shrink_bias"] == pytest.approx(one["stats"]["shrink_bias"], rel=1e-12)
    y2 = o.dequantize_two_level(two["codes"], two["scales"], two["outer_scales"])
    y1 = o.dequantize(one["codes"], one["scales"], one["tensor_scale"], "nvfp4")
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("rounding", ["rtne", "sr"])
@pytest.mark.parametrize("k", [-7, 5])
def test_power_of_two_scaling_of_one_outer_block(rht, rounding, k):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((6, 384)) * np.exp(rng.standard_normal((1, 384)))).astype(np.float32)
    base = o.quantize(x, "nvfp4_2l", rht=rht, rounding=rounding, seed=3)["row"]
    y = x.copy()
    y[2, OB:2 * OB] *= np.float32(2.0 ** k)          # row 2, second outer block
    sc = o.quantize(y, "nvfp4_2l", rht=rht, rounding=rounding, seed=3)["row"]
    assert np.array_equal(sc["codes"], base["codes"])
    assert np.array_equal(sc["scales"], base["scales"])
    want = base["outer_scales"].copy()
    want[2, 1] = np.float32(want[2, 1] * np.float32(2.0 ** k))
    assert np.array_equal(sc["outer_scales"].view(np.uint32), want.view(np.uint32))


def test_on_grid_values_round_trip_exactly():
    rng = np.random.default_rng(7)
    rows, cols = 5, 256
    q_mag = o.E2M1_LEVELS
    v = np.zeros((rows, cols), dtype=np.float64)
    g_o = np.zeros((rows, cols // OB))
    codes = np.zeros((rows, cols), dtype=np.uint8)
    s_codes = np.zeros((rows, cols // 16), dtype=np.uint8)
    for r in range(rows):
        for ob in range(cols // OB):
            g = 2.0 ** int(rng.integers(-20, 10))
            g_o[r, ob] = g
            for ib in range(OB // 16):
                b = ob * (OB // 16) + ib
                # the outer block's largest inner block carries s = 448 and q = 6
                sc = 126 if ib == 0 else int(rng.integers(40, 126))
                s_codes[r, b] = sc
                k = rng.integers(0, 8, 16)
                k[int(rng.integers(0, 16))] = 7                    # block max is 6 * s
                sign = rng.integers(0, 2, 16)
                codes[r, b * 16:(b + 1) * 16] = (sign << 3) | k
                v[r, b * 16:(b + 1) * 16] = np.where(sign, -1, 1) * q_mag[k] * o.e4m3_decode(sc) * g
    x = v.astype(np.float32)
    assert np.array_equal(x.astype(np.float64), v)           # exactly representable
    res = o.quantize(x, "nvfp4_2l")["row"]
    assert np.array_equal(res["outer_scales"], g_o.astype(np.float32))
    assert np.array_equal(res["scales"], s_codes)
    assert np.array_equal(o.unpack_nibbles(res["codes"]), codes)
    back = o.dequantize_two_level(res["codes"], res["scales"], res["outer_scales"])
    assert np.array_equal(back, x)
    assert np.isinf(res["stats"]["snr_db"])


def test_zero_outer_block():
    x = np.ones((3, 256), dtype=np.float32)
    x[1, :OB] = 0.0
    res = o.quantize(x, "nvfp4_2l")["row"]
    assert res["outer_scales"][1, 0] == 0.0
    assert np.all(res["scales"][1, :OB // 16] == 0)
    assert np.all(o.unpack_nibbles(res["codes"])[1, :OB] == 0)
    assert res["outer_scales"][1, 1] == np.float32(1.0) / np.float32(2688.0)


def test_gemm_reduces_to_nvfp4_when_outer_amax_is_the_tensor_amax():
    """The oracle's GEMM on two-level copies equals its (separately pinned)
    NVFP4 GEMM when every outer scale is the tensor scale."""
    a = _planted(6, 512, 3.75, 11)
    b = _planted(5, 512, 3.75, 12)
    two = o.gemm(o.quantize(a, "nvfp4_2l")["row"], o.quantize(b, "nvfp4_2l")["row"])
    one = o.gemm(o.quantize(a, "nvfp4")["row"], o.quantize(b, "nvfp4")["row"])
    assert np.array_equal(two, one)


def test_gemm_of_power_of_two_outer_scales_matches_the_fp32_dequantisation():
    """With power-of-two outer scales every dequantised value is exact in FP32,
    so the FP64 GEMM equals the product of the FP32 dequantised operands."""
    rng = np.random.default_rng(13)
    ca = {"fmt": "nvfp4_2l", "codes": o.pack_nibbles(rng.integers(0, 16, (4, 256)).astype(np.uint8)),
          "scales": ((rng.integers(-3, 3, (4, 16)) + 7) << 3).astype(np.uint8),
          "outer_scales": np.exp2(rng.integers(-4, 4, (4, 2))).astype(np.float32)}
    cb = {"fmt": "nvfp4_2l", "codes": o.pack_nibbles(rng.integers(0, 16, (3, 256)).astype(np.uint8)),
          "scales": ((rng.integers(-3, 3, (3, 16)) + 7) << 3).astype(np.uint8),
          "outer_scales": np.exp2(rng.integers(-4, 4, (3, 2))).astype(np.float32)}
    da = o.dequantize_two_level(ca["codes"], ca["scales"], ca["outer_scales"]).astype(np.float64)
    db = o.dequantize_two_level(cb["codes"], cb["scales"], cb["outer_scales"]).astype(np.float64)
    assert np.array_equal(o.gemm(ca, cb), da @ db.T)
