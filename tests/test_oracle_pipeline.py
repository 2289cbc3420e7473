"""Pins of the oracle's full quantise / statistics / dequantise / GEMM chain
(no GPU): closed forms, exact special cases and an integer brute force."""
import os

import numpy as np
import pytest

from oracle import fp4q_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _closed_form_rows():
    levels, ranges = [], []
    with open(os.path.join(GOLDEN, "shrinkage_closed_form.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            p = line.split()
            if p[0] == "range":
                ranges.append((p[1], float(p[2]), float(p[3]), float(p[4])))
            else:
                levels.append((p[0], float(p[1]), float(p[2]), float(p[3]), float(p[4])))
    return levels, ranges


def _anchored(samples: np.ndarray, qmax: float) -> np.ndarray:
    """Blocks [Qmax, y1..y15] plus one block holding the tensor amax Qmax*448:
    g = 1 and every anchored block has s_b = 1, so y = v exactly."""
    per = 15
    nb = -(-samples.size // per)
    pad = np.zeros(nb * per, dtype=np.float32)
    pad[:samples.size] = samples
    m = np.zeros((nb + 1, 16), dtype=np.float32)
    m[:nb, 0] = qmax
    m[:nb, 1:] = pad.reshape(nb, per)
    m[nb, 0] = qmax * 448.0
    return m


def _midpoints(lo, hi, n):
    h = (hi - lo) / n
    return (lo + h * (np.arange(n) + 0.5))


def test_shrinkage_per_level_closed_form():
    levels, _ = _closed_form_rows()
    for grid, q, l, r, expect in levels:
        fmt = "nvfp4" if grid == "e2m1" else "ufp4"
        y = _midpoints(q - l, q + r, 3 * 4096).astype(np.float32)
        c = o.round_rtne(y, fmt)
        assert np.all(o.code_value(c, fmt) == q)
        err = np.mean(o.code_value(c, fmt) - y.astype(np.float64))
        assert abs(err - expect) < 1e-9, (grid, q)


def test_shrinkage_bias_statistic_closed_form():
    _, ranges = _closed_form_rows()
    for grid, lo, hi, expect in ranges:
        fmt = "nvfp4" if grid == "e2m1" else "ufp4"
        qmax = o.QMAX[fmt]
        n = int(round((hi - lo) / 0.25)) * 4000   # every bin edge is a cell edge
        y64 = _midpoints(lo, hi, n)
        y = y64.astype(np.float32)
        m = _anchored(y, qmax)
        st = o.quantize_copy(m, fmt)["stats"]
        nel = m.size
        # the samples sum to n * expect; rounding the sample points to FP32
        # shifts the sum by -sum(y32 - y64); the tensor-amax element adds at
        # most one FP32 ulp of Qmax
        want = (n * expect - float(np.sum(y.astype(np.float64) - y64))) / (qmax * nel)
        assert abs(st["shrink_bias"] - want) < 1e-6 / (qmax * nel)


def test_snr_closed_form():
    nb = 100
    m = np.zeros((nb + 1, 16), dtype=np.float32)
    m[:nb, 0] = 6.0
    m[:nb, 1:] = 0.25          # ties to 0: error 0.25 each
    m[nb, 0] = 6.0 * 448.0
    st = o.quantize_copy(m, "nvfp4")["stats"]
    sig = nb * (36.0 + 15 * 0.0625) + 2688.0 ** 2
    err = nb * 15 * 0.0625
    assert st["sum_sig2"] == sig
    assert st["sum_err2"] == err
    assert abs(st["snr_db"] - 10 * np.log10(sig / err)) < 1e-12


def test_on_grid_tensor_is_exact():
    rng = np.random.default_rng(11)
    for fmt in ("nvfp4", "ufp4"):
        qmax = o.QMAX[fmt]
        lv = o.grid_levels(fmt)
        y = (lv[rng.integers(0, 8, 15 * 500)] * np.where(rng.random(15 * 500) < 0.5, -1, 1)).astype(np.float32)
        m = _anchored(y, qmax)
        q = o.quantize_copy(m, fmt)
        assert q["stats"]["snr_db"] == float("inf")
        back = o.dequantize(q["codes"], q["scales"], q["tensor_scale"], fmt)
        assert np.array_equal(back[:-1], m[:-1])
    # MXFP4: x = level * 2^e with block amax 6 * 2^e has e_b = e and is exact
    e = rng.integers(-20, 20, 64)
    lvl = o.E2M1_LEVELS[rng.integers(0, 8, (64, 32))]
    lvl[:, 0] = 6.0
    x = (lvl * np.exp2(e)[:, None]).astype(np.float32)
    q = o.quantize_copy(x, "mxfp4")
    assert np.array_equal(q["scales"][:, 0].astype(np.int64), e + 127)
    assert np.array_equal(o.dequantize(q["codes"], q["scales"], 1.0, "mxfp4"), x)
    assert q["stats"]["snr_db"] == float("inf")


def test_zero_and_negative_zero():
    m = np.zeros((2, 32), dtype=np.float32)
    m[1] = -0.0
    for fmt in o.FORMATS:
        q = o.quantize_copy(m, fmt)
        c = o.unpack_nibbles(q["codes"])
        assert np.all(c[0] == 0) and np.all(c[1] == 8)
        assert q["stats"]["snr_db"] == float("inf")
        if fmt in o.E8M0_FORMATS:      # amax 0: the smallest exponent, code 0
            assert q["tensor_scale"] == 1.0 and np.all(q["scales"] == 0)
        else:
            assert q["tensor_scale"] == 0.0 and np.all(q["scales"] == 0)


def test_nvfp4_scale_chain_example():
    """A worked case by hand: tensor amax 2688 -> g = 1; a block with amax 3
    has t = 3/6 = 0.5 -> s_b = 0.5 (E4M3 code 0x30), r_b = 2, so 1.1 -> y = 2.2
    -> 2.0 and -2.9 -> -5.8 -> -6."""
    m = np.zeros((2, 16), dtype=np.float32)
    m[0, 0] = 2688.0
    m[1, :3] = [3.0, 1.1, -2.9]
    q = o.quantize_copy(m, "nvfp4")
    assert q["tensor_scale"] == 1.0
    assert q["scales"][1, 0] == 0x30 and o.e4m3_decode(0x30) == 0.5
    vals = o.code_value(o.unpack_nibbles(q["codes"])[1, :3], "nvfp4")
    assert list(vals) == [6.0, 2.0, -6.0]


def test_gemm_exact_integer_case():
    """Power-of-two block scales and g = 1: the FP64 product is exact and must
    equal an int64 matrix product of the integer-scaled codes."""
    rng = np.random.default_rng(4)
    M, N, K = 128, 64, 256

    def make(rows):
        codes = rng.integers(0, 16, (rows, K)).astype(np.uint8)
        kexp = rng.integers(-6, 4, (rows, K // 16))
        scales = ((kexp + 7) << 3).astype(np.uint8)   # E4M3 code of 2^k
        assert np.array_equal(o.e4m3_decode(scales), np.exp2(kexp))
        cp = {"fmt": "nvfp4", "codes": o.pack_nibbles(codes), "scales": scales,
              "tensor_scale": np.float32(1.0)}
        half = {0: 0, 1: 1, 2: 2, 3: 3, 4: 4, 5: 6, 6: 8, 7: 12}   # 2 * E2M1 level
        iv = np.vectorize(lambda c: (-1 if c & 8 else 1) * half[int(c) & 7])(codes).astype(np.int64)
        iv = iv * (np.repeat(np.left_shift(1, kexp + 6), 16, axis=1))
        return cp, iv

    a, ai = make(M)
    b, bi = make(N)
    y = o.gemm(a, b)
    yi = np.einsum("mk,nk->mn", ai, bi)            # int64, no BLAS
    assert np.array_equal(y, yi.astype(np.float64) / 2.0 ** 14)
    rows = np.array([3, 77])
    cols = np.array([0, 5, 63])
    assert np.array_equal(o.gemm(a, b, rows, cols), y[np.ix_(rows, cols)])


def test_mma_scale_layout():
    n, nkb = 256, 8
    r, kb = np.meshgrid(np.arange(n), np.arange(nkb), indexing="ij")
    off = o.mma_scale_offset(r, kb, nkb)
    assert np.array_equal(np.sort(off.ravel()), np.arange(n * nkb))   # a bijection
    assert o.mma_scale_offset(0, 0, nkb) == 0
    assert o.mma_scale_offset(1, 0, nkb) == 16
    assert o.mma_scale_offset(32, 0, nkb) == 4
    assert o.mma_scale_offset(33, 2, nkb) == 16 + 4 + 2
    assert o.mma_scale_offset(0, 4, nkb) == 512           # next block group
    assert o.mma_scale_offset(128, 0, nkb) == 2 * 512     # next row tile
    s = np.arange(100 * 6, dtype=np.uint8).reshape(100, 6)
    flat = o.scales_to_mma_layout(s)
    assert flat.size == o.mma_layout_bytes(100, 6) == 128 * 8
    assert flat[o.mma_scale_offset(99, 5, 8)] == s[99, 5]
    assert flat[o.mma_scale_offset(100, 0, 8)] == 0


def test_col_copy_is_transposed_row_copy():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((48, 32)).astype(np.float32)
    both = o.quantize(x, "nvfp4", rht=True, seed=5, axis="both")
    colq = o.quantize_copy(np.ascontiguousarray(x.T), "nvfp4", True, "rtne", 5, 1)
    assert np.array_equal(both["col"]["codes"], colq["codes"])
    assert both["col"]["codes"].shape == (32, 24)
    assert both["row"]["codes"].shape == (48, 16)


def test_rht_definition_mode_close_to_butterfly():
    rng = np.random.default_rng(9)
    x = o.bf16_bits_to_f32(o.f32_to_bf16_bits_rne(rng.standard_normal((64, 64)).astype(np.float32)))
    a = o.quantize(x, "nvfp4", rht=True, seed=3, rht_mode="butterfly")["row"]
    b = o.quantize(x, "nvfp4", rht=True, seed=3, rht_mode="definition")["row"]
    assert np.mean(a["codes"] == b["codes"]) > 0.99


def test_sr_pipeline_uses_copy_index():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((32, 64)).astype(np.float32)
    a = o.quantize(x, "nvfp4", rounding="sr", seed=1234, axis="both")
    b = o.quantize(x, "nvfp4", rounding="sr", seed=1234, axis="both")
    c = o.quantize(x, "nvfp4", rounding="sr", seed=1235, axis="both")
    assert np.array_equal(a["row"]["codes"], b["row"]["codes"])
    assert not np.array_equal(a["row"]["codes"], c["row"]["codes"])
    # SR lies on one of the two neighbouring levels of the RTNE result
    r = o.quantize(x, "nvfp4", axis="row")["row"]
    assert np.array_equal(a["row"]["scales"], r["scales"])


def test_nonfinite_flag():
    x = np.zeros((16, 16), dtype=np.float32)
    assert not o.quantize(x, "nvfp4")["nonfinite"]
    x[3, 4] = np.nan
    assert o.quantize(x, "nvfp4")["nonfinite"]
