"""GPU parity of the quantise / dequantise path against the CPU oracle.

Codes and scales must be bit-exact with the oracle's FP32 butterfly reading
(RHT off, RHT on, RTNE and SR); the RHT-on codes are also checked against the
dense FP64 definition of the transform with mismatches allowed only next to a
rounding boundary. Statistics: shrink bias within 1e-5 of the mean absolute
rounding error (FP32 partial sums of at most 16 terms, Kahan-compensated across
blocks, FP64 across CTAs), SNR within 1e-3 dB.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import fp4q_oracle as o

pytestmark = pytest.mark.gpu

SHAPES = {"nvfp4": (208, 272), "ufp4": (208, 272), "mxfp4": (224, 288)}


def _bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return synth.bf16_bits(t.cpu())
    return t.cpu().numpy()


def _input(fmt, dtype, seed=5, shape=None):
    rows, cols = shape or SHAPES[fmt]
    if dtype == torch.bfloat16:
        return synth.normal_with_outliers(rows, cols, 1.0, 0.01, 20.0, seed)
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(1, cols, generator=g))
    return x.float()


def check_copy(gq, oq, layout):
    codes = gq.codes.cpu().numpy()
    assert codes.shape == oq["codes"].shape
    mism = np.flatnonzero(codes.ravel() != oq["codes"].ravel())
    assert mism.size == 0, f"{mism.size} code bytes differ, first at {mism[:5]}"
    sc = gq.scales.cpu().numpy()
    if layout == "linear":
        assert np.array_equal(sc, oq["scales"])
    else:
        assert np.array_equal(sc.ravel(), o.scales_to_mma_layout(oq["scales"], oq["block"]))
    ts = gq.tensor_scale.cpu().numpy().view(np.uint32)[0]
    assert ts == np.float32(oq["tensor_scale"]).view(np.uint32)


def snr_error_bound(snr_db: float) -> float:
    """The kernel forms each error v - v_hat from FP32 values carrying at most
    three roundings (y = v * r_b, r_b = 1 / p, the product back), so each error
    is off by at most 3 * 2^-24 |v|. With S = sum v^2 / sum e^2 the error energy
    is then off by a relative 6 * 2^-24 sqrt(S) + 9 * 2^-48 S."""
    s = 10.0 ** (snr_db / 10.0)
    return 6 * 2.0 ** -24 * np.sqrt(s) + 9 * 2.0 ** -48 * s


def snr_tolerance_db(snr_db: float) -> float:
    """The bound above in dB, plus 1e-3 dB for the summation order."""
    return 1e-3 + 10.0 * np.log10(1.0 + snr_error_bound(snr_db))


def check_stats(gs, os_):
    assert gs["n"] == os_["n"]
    tol = 1e-5 * os_["mean_abs_bias"] + 1e-12
    assert abs(gs["shrink_bias"] - os_["shrink_bias"]) <= tol, (gs, os_)
    if np.isinf(os_["snr_db"]):
        assert np.isinf(gs["snr_db"]) or gs["snr_db"] > 120
    elif snr_error_bound(os_["snr_db"]) < 1.0:
        tol_db = snr_tolerance_db(os_["snr_db"])
        assert abs(gs["snr_db"] - os_["snr_db"]) <= tol_db, (gs["snr_db"], os_["snr_db"], tol_db)
    else:
        # the error energy is below what FP32 arithmetic resolves: only the
        # order of magnitude is meaningful
        assert gs["snr_db"] > os_["snr_db"] - snr_tolerance_db(os_["snr_db"]) or np.isinf(gs["snr_db"])


@pytest.mark.parametrize("layout", ["linear", "mma"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("axis", ["row", "col", "both"])
@pytest.mark.parametrize("rounding", ["rtne", "sr"])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "ufp4"])
def test_quantize_parity(lib, fmt, rht, rounding, axis, dtype, layout):
    x = _input(fmt, dtype)
    seed = 1234
    r, c = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=rht, rounding=rounding, seed=seed,
                             axis=axis, layout=layout)
    rs, cs = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(_bits(x), fmt, rht=rht, rounding=rounding, seed=seed, axis=axis)
    if axis in ("row", "both"):
        check_copy(r, ref["row"], layout)
        check_stats(rs, ref["row"]["stats"])
    if axis in ("col", "both"):
        check_copy(c, ref["col"], layout)
        check_stats(cs, ref["col"]["stats"])


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("layout", ["linear", "mma"])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "ufp4"])
def test_dequantize_parity(lib, fmt, layout, rht, out_dtype):
    x = _input(fmt, torch.bfloat16, seed=9)
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=rht, seed=77, axis="row", layout=layout)
    y = lib.fp4q_dequantize(r, inverse_rht=rht, seed=77, out_dtype=out_dtype)
    ref = o.quantize(_bits(x), fmt, rht=rht, seed=77, axis="row")["row"]
    want = o.dequantize(ref["codes"], ref["scales"], ref["tensor_scale"], fmt,
                        inverse_rht=rht, seed=77)
    if out_dtype == torch.float32:
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))
    else:
        got = synth.bf16_bits(y.cpu())
        assert np.array_equal(got, o.f32_to_bf16_bits_rne(want))


@pytest.mark.parametrize("fmt", ["nvfp4", "ufp4", "mxfp4"])
def test_rht_codes_against_dense_definition(lib, fmt):
    """Codes vs the FP64 dense transform: a code may differ only where the
    oracle's pre-rounding value lies within 2 FP32 ulp of a bin boundary, or
    in a block whose scale sits on an E4M3 rounding boundary (adjacent code)."""
    x = synth.activation(512, 1024)
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=True, seed=31, axis="row")
    ref = o.quantize(_bits(x), fmt, rht=True, seed=31, rht_mode="definition", keep_y=True)["row"]
    b = o.BLOCK[fmt]
    gs = r.scales.cpu().numpy().astype(np.int64)
    os_ = ref["scales"].astype(np.int64)
    dscale = gs != os_
    assert np.all(np.abs(gs - os_)[dscale] == 1)
    assert dscale.mean() < 1e-3
    gc = o.unpack_nibbles(r.codes.cpu().numpy())
    oc = o.unpack_nibbles(ref["codes"])
    bad = gc != oc
    bad &= ~np.repeat(dscale, b, axis=1)
    if bad.any():
        y = np.abs(ref["y"][bad].astype(np.float64))
        lv = o.grid_levels(fmt)
        mids = (lv[:-1] + lv[1:]) / 2
        dist = np.min(np.abs(y[:, None] - mids[None, :]), axis=1)
        ulp = np.spacing(np.float32(y).astype(np.float32)).astype(np.float64)
        assert np.all(dist <= 2 * ulp)
    assert bad.mean() < 1e-4


def test_act_small_nvfp4_exact(lib):
    """1024 x 1024 N(0,1) with 0.5% x20 outliers, NVFP4, RTNE, no RHT, row-wise:
    codes, scales, tensor scale bit-exact; bias and SNR reported."""
    x = synth.act_small()
    r, _ = lib.fp4q_quantize(x.cuda(), fmt="nvfp4", axis="row")
    rs, _ = lib.fp4q_stats()
    ref = o.quantize(_bits(x), "nvfp4")["row"]
    check_copy(r, ref, "linear")
    check_stats(rs, ref["stats"])
    y = lib.fp4q_dequantize(r)
    want = o.dequantize(ref["codes"], ref["scales"], ref["tensor_scale"], "nvfp4")
    assert np.array_equal(y.cpu().numpy(), want)


# ---- edge cases ------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "ufp4"])
def test_zeros_and_signed_zeros(lib, fmt):
    rows, cols = 64, 128
    x = torch.zeros(rows, cols, dtype=torch.bfloat16)
    x[1::2] = -0.0
    x[5, 7] = -1e-30   # a negative value that rounds to zero keeps its sign
    r, c = lib.fp4q_quantize(x.cuda(), fmt=fmt, axis="both")
    ref = o.quantize(_bits(x), fmt, axis="both")
    check_copy(r, ref["row"], "linear")
    check_copy(c, ref["col"], "linear")
    rs, cs = lib.fp4q_stats()
    check_stats(rs, ref["row"]["stats"])
    check_stats(cs, ref["col"]["stats"])


@pytest.mark.parametrize("fmt", ["nvfp4", "ufp4", "mxfp4"])
@pytest.mark.parametrize("mag", [1e-30, 1e-3, 1e30])
def test_extreme_magnitudes(lib, fmt, mag):
    x = (_input(fmt, torch.float32, seed=3) * mag).float()
    r, c = lib.fp4q_quantize(x.cuda(), fmt=fmt, axis="both")
    rs, cs = lib.fp4q_stats()
    ref = o.quantize(x.numpy(), fmt, axis="both")
    check_copy(r, ref["row"], "linear")
    check_copy(c, ref["col"], "linear")
    check_stats(rs, ref["row"]["stats"])


@pytest.mark.parametrize("fmt", ["nvfp4", "ufp4"])
def test_blocks_whose_scale_rounds_to_zero(lib, fmt):
    """One huge element: blocks far below it get scale 0 and all-zero codes."""
    x = (torch.randn(128, 256, generator=torch.Generator().manual_seed(2)) * 1e-4).float()
    x[3, 5] = 1e4
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=fmt, axis="row")
    rs, _ = lib.fp4q_stats()
    ref = o.quantize(x.numpy(), fmt, axis="row")["row"]
    assert np.mean(ref["scales"] == 0) > 0.9
    check_copy(r, ref, "linear")
    check_stats(rs, ref["stats"])


def test_empty_input(lib):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    r, _ = lib.fp4q_quantize(x, fmt="nvfp4", axis="row")
    rs, _ = lib.fp4q_stats()
    assert r.tensor_scale.item() == 0.0
    assert rs["n"] == 0


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_nonfinite_sets_status(lib, fmt):
    x = torch.randn(64, 128).to(torch.bfloat16)
    x[10, 20] = float("nan")
    lib.fp4q_quantize(x.cuda(), fmt=fmt, axis="row")
    assert lib.fp4q_status() == 4
    assert lib.fp4q_status() == 0     # cleared by the read
    x[10, 20] = float("inf")
    lib.fp4q_quantize(x.cuda(), fmt=fmt, axis="col")
    assert lib.fp4q_status() == 4


def test_invalid_arguments_rejected(lib):
    x = torch.randn(64, 120, device="cuda").to(torch.bfloat16)    # 120 % 16 != 0
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_quantize(x, fmt="nvfp4", axis="row")
    assert e.value.code == 1
    y = torch.randn(48, 64, device="cuda").to(torch.bfloat16)     # 48 % 32 != 0
    with pytest.raises(lib.FP4QError):
        lib.fp4q_quantize(y, fmt="mxfp4", axis="col")
    z = torch.randn(208, 100, device="cuda").to(torch.bfloat16)   # column-wise, 100 % 16 != 0
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_quantize(z, fmt="nvfp4", axis="col")
    assert e.value.code == 1
    # UFP4 runs on the dequantising GEMM, whose K must be a multiple of 64
    r, _ = lib.fp4q_quantize(torch.randn(128, 96, device="cuda"), fmt="ufp4", layout="mma")
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_gemm(r, r)
    assert e.value.code == 1


def test_repeated_calls_reuse_workspace(lib):
    """Counters wrap back to zero: many calls in a row stay correct."""
    x = _input("nvfp4", torch.bfloat16, seed=21)
    ref = o.quantize(_bits(x), "nvfp4", rht=True, seed=4, axis="both")
    xd = x.cuda()
    for _ in range(5):
        r, c = lib.fp4q_quantize(xd, fmt="nvfp4", rht=True, seed=4, axis="both")
        rs, cs = lib.fp4q_stats()
        check_copy(r, ref["row"], "linear")
        check_copy(c, ref["col"], "linear")
        check_stats(cs, ref["col"]["stats"])


@pytest.mark.parametrize("fmt,rht,axis", [("nvfp4", False, "row"), ("nvfp4", True, "both"),
                                          ("ufp4", True, "col"), ("mxfp4", True, "both")])
def test_split_amax_then_quantize(lib, fmt, rht, axis):
    """fp4q_amax followed by fp4q_quantize(amax_ready) equals one fp4q_quantize
    call and the oracle, byte for byte."""
    x = _input(fmt, torch.bfloat16, seed=13)
    xd = x.cuda()
    lib.fp4q_amax(xd, fmt=fmt, rht=rht, seed=99, axis=axis)
    r, c = lib.fp4q_quantize(xd, fmt=fmt, rht=rht, seed=99, axis=axis, amax_ready=True)
    rs, cs = lib.fp4q_stats()
    ref = o.quantize(_bits(x), fmt, rht=rht, seed=99, axis=axis)
    if axis in ("row", "both"):
        check_copy(r, ref["row"], "linear")
        check_stats(rs, ref["row"]["stats"])
    if axis in ("col", "both"):
        check_copy(c, ref["col"], "linear")
        check_stats(cs, ref["col"]["stats"])


# ---- the row-wise stream kernels: ragged tails, tiled scales, subnormals ----------

RAGGED = [(1, 16), (3, 48), (207, 272), (129, 8208), (33, 4096 + 32)]


@pytest.mark.parametrize("shape", RAGGED)
@pytest.mark.parametrize("fmt,rht,rounding,layout", [
    ("nvfp4", False, "rtne", "linear"), ("nvfp4", True, "rtne", "mma"), ("nvfp4", True, "sr", "linear"),
    ("ufp4", True, "rtne", "mma"), ("ufp4", False, "sr", "linear"),
    ("mxfp4", False, "rtne", "mma"), ("mxfp4", True, "sr", "linear"),
    ("mxfp4_b16", True, "sr", "mma"), ("mxfp4_oas", False, "rtne", "linear"), ("mxfp4_oas", True, "sr", "mma")])
def test_rowwise_stream_ragged(lib, shape, fmt, rht, rounding, layout):
    """Row-wise copies whose element count leaves a partial chunk and, where
    rows x cols is an odd multiple of 16, a half-filled last thread segment;
    odd block counts per row exercise the tiled scale layout's row split."""
    rows, cols = shape
    if fmt == "mxfp4" and cols % 32:
        pytest.skip("MXFP4 needs cols % 32 == 0")
    x = synth.normal_with_outliers(rows, cols, 1.0, 0.01, 20.0, 17)
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=rht, rounding=rounding, seed=5, axis="row",
                             layout=layout)
    rs, _ = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(_bits(x), fmt, rht=rht, rounding=rounding, seed=5, axis="row")["row"]
    check_copy(r, ref, layout)
    check_stats(rs, ref["stats"])


@pytest.mark.parametrize("fmt", ["nvfp4", "ufp4", "mxfp4"])
@pytest.mark.parametrize("rht", [False, True])
def test_fp32_subnormal_inputs(lib, fmt, rht):
    """FP32 inputs in the subnormal range next to normal ones: every packed
    FP32x2 step must keep subnormals (no flush to zero), as the oracle does."""
    g = torch.Generator().manual_seed(23)
    x = torch.randn(64, 256, generator=g) * 1e-39          # mostly subnormal
    x[:, ::7] *= 1e6                                        # some normal neighbours
    x[5] = torch.randn(256, generator=g) * 1e-44            # a row of the smallest subnormals
    x = x.float()
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=rht, seed=3, axis="row")
    rs, _ = lib.fp4q_stats()
    ref = o.quantize(x.numpy(), fmt, rht=rht, seed=3, axis="row")["row"]
    check_copy(r, ref, "linear")
    y = lib.fp4q_dequantize(r, inverse_rht=rht, seed=3)
    want = o.dequantize(ref["codes"], ref["scales"], ref["tensor_scale"], fmt, inverse_rht=rht, seed=3)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_rowwise_nonfinite_sets_status(lib, fmt):
    for bad in (float("nan"), float("inf"), float("-inf")):
        x = torch.randn(40, 256).to(torch.bfloat16)
        x[17, 3] = bad
        lib.fp4q_quantize(x.cuda(), fmt=fmt, axis="row", rht=True, seed=1)
        assert lib.fp4q_status() == 4, bad


# Byte offset of the one-launch quantiser's grid-barrier arrival count in the
# workspace header: after status, amax_nparts, stat_nparts, copies (4 x u32),
# tensor_scale[2] and qmax (3 x f32).
_GBAR_COUNT_OFFSET = 28


@pytest.mark.parametrize("leftover", [3, 100000])
def test_fused_barrier_ignores_a_stale_arrival_count(lib, leftover):
    """A grid barrier whose wait ran out leaves its arrival count part-way.
    Planted here on the host (no kernel is made to time out): the next
    one-launch quantisation on that workspace must still see every CTA's
    amax, so its tensor scale, scales and codes match the oracle."""
    ws = torch.zeros(lib.fp4q_workspace_size(), dtype=torch.uint8, device="cuda")
    big = synth.normal_with_outliers(512, 1024, 1000.0, 0.01, 20.0, 31)
    small = synth.normal_with_outliers(512, 1024, 1.0, 0.01, 20.0, 32)
    lib.fp4q_quantize(big.cuda(), fmt="nvfp4", rht=True, seed=8, axis="row", ws=ws)
    torch.cuda.synchronize()
    ws[_GBAR_COUNT_OFFSET:_GBAR_COUNT_OFFSET + 4] = torch.tensor(
        [leftover], dtype=torch.int32).view(torch.uint8).cuda()
    r, _ = lib.fp4q_quantize(small.cuda(), fmt="nvfp4", rht=True, seed=8, axis="row", ws=ws)
    rs, _ = lib.fp4q_stats(ws)
    assert lib.fp4q_status(ws) == 0
    ref = o.quantize(_bits(small), "nvfp4", rht=True, seed=8, axis="row")["row"]
    check_copy(r, ref, "linear")
    check_stats(rs, ref["stats"])
