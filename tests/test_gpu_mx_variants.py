"""GPU parity of the E8M0 variants of "Unveiling the Potential of Quantization
with MXFP4 ...", Résumé technique §2 and §2A-§2B, against the CPU oracle:
MXFP4 on 16-element blocks, the overflow-aware exponent rule (OAS) and the
static macro-block scale (MBS). Codes, E8M0 scales and macro scales
bit-exact, dequantised values bit-exact, statistics within the tolerance of
the other formats; the native GEMM with E8M0 scales (32- and 16-element
blocks) against the oracle's FP64 dequantise-then-matmul."""
import numpy as np
import pytest
import torch

import synth
from oracle import fp4q_oracle as o

from test_gpu_quantize import _bits, _input, check_copy, check_stats

pytestmark = pytest.mark.gpu

MX16 = ["mxfp4_b16", "mxfp4_oas"]


@pytest.mark.parametrize("layout", ["linear", "mma"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("axis", ["row", "col", "both"])
@pytest.mark.parametrize("rounding", ["rtne", "sr"])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("fmt", MX16)
def test_mx16_parity(lib, fmt, rht, rounding, axis, dtype, layout):
    x = _input("nvfp4", dtype, seed=21, shape=(208, 400))     # ragged tiles: 400 = 3 x 128 + 16
    r, c = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=rht, rounding=rounding, seed=99, axis=axis, layout=layout)
    rs, cs = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(_bits(x), fmt, rht=rht, rounding=rounding, seed=99, axis=axis)
    if axis in ("row", "both"):
        check_copy(r, ref["row"], layout)
        check_stats(rs, ref["row"]["stats"])
    if axis in ("col", "both"):
        check_copy(c, ref["col"], layout)
        check_stats(cs, ref["col"]["stats"])


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("fmt,layout", [("mxfp4_b16", "linear"), ("mxfp4_oas", "mma"), ("mxfp4", "mma")])
def test_mx_dequantize(lib, fmt, layout, rht, out_dtype):
    x = _input("nvfp4", torch.bfloat16, seed=23, shape=(96, 512))
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=rht, seed=6, layout=layout)
    y = lib.fp4q_dequantize(r, inverse_rht=rht, seed=6, out_dtype=out_dtype)
    ref = o.quantize(_bits(x), fmt, rht=rht, seed=6)["row"]
    want = o.dequantize(ref["codes"], ref["scales"], 1.0, fmt, rht, 6)
    if out_dtype == torch.float32:
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))
    else:
        assert np.array_equal(synth.bf16_bits(y.cpu()), o.f32_to_bf16_bits_rne(want))


def check_mbs(gq, oq, layout):
    codes = gq.codes.cpu().numpy()
    mism = np.flatnonzero(codes.ravel() != oq["codes"].ravel())
    assert mism.size == 0, f"{mism.size} code bytes differ, first at {mism[:5]}"
    sc = gq.scales.cpu().numpy()
    if layout == "linear":
        assert np.array_equal(sc, oq["scales"])
    else:
        assert np.array_equal(sc.ravel(), o.scales_to_mma_layout(oq["scales"]))
    S = gq.tensor_scale.cpu().numpy()
    if layout == "mma":                 # the tiled layout keeps the macro scales column-major
        S = np.ascontiguousarray(S.T)
    assert S.shape == oq["macro_scales"].shape
    assert np.array_equal(S.view(np.uint32), oq["macro_scales"].view(np.uint32))


@pytest.mark.parametrize("layout", ["linear", "mma"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding", ["rtne", "sr"])
@pytest.mark.parametrize("rht", [False, True])
def test_mbs_parity(lib, rht, rounding, dtype, layout):
    x = _input("nvfp4", dtype, seed=31, shape=(208, 384))     # 9.75 chunks: a ragged last chunk
    r, _ = lib.fp4q_quantize(x.cuda(), fmt="mxfp4_mbs", rht=rht, rounding=rounding, seed=55, layout=layout)
    rs, _ = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(_bits(x), "mxfp4_mbs", rht=rht, rounding=rounding, seed=55)["row"]
    check_mbs(r, ref, layout)
    check_stats(rs, ref["stats"])


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rht", [False, True])
def test_mbs_dequantize(lib, rht, out_dtype):
    x = _input("nvfp4", torch.bfloat16, seed=32, shape=(96, 512))
    r, _ = lib.fp4q_quantize(x.cuda(), fmt="mxfp4_mbs", rht=rht, seed=8)
    y = lib.fp4q_dequantize(r, inverse_rht=rht, seed=8, out_dtype=out_dtype)
    ref = o.quantize(_bits(x), "mxfp4_mbs", rht=rht, seed=8)["row"]
    want = o.dequantize_mbs(ref["codes"], ref["scales"], ref["macro_scales"], rht, 8)
    if out_dtype == torch.float32:
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))
    else:
        assert np.array_equal(synth.bf16_bits(y.cpu()), o.f32_to_bf16_bits_rne(want))


@pytest.mark.parametrize("mag", [1e-39, 1e-30, 1e30])
@pytest.mark.parametrize("fmt", ["mxfp4_mbs", "mxfp4_oas"])
def test_mx_extreme_magnitudes(lib, fmt, mag):
    """Subnormal inputs (1e-39) put the macro scale below 2^-128, where 1/S
    overflows and is held at FLT_MAX, and the E8M0 exponents at their floor."""
    x = (_input("nvfp4", torch.float32, seed=4, shape=(64, 256)) * mag).float()
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=fmt)
    rs, _ = lib.fp4q_stats()
    ref = o.quantize(x.numpy(), fmt)["row"]
    if fmt == "mxfp4_mbs":
        check_mbs(r, ref, "linear")
    else:
        check_copy(r, ref, "linear")
    if mag > 1e-38:
        check_stats(rs, ref["stats"])


def test_mbs_zero_macro_blocks(lib):
    x = torch.randn(32, 384).to(torch.bfloat16)
    x[5, 128:256] = 0.0
    x[9, :128] = -0.0
    r, _ = lib.fp4q_quantize(x.cuda(), fmt="mxfp4_mbs")
    ref = o.quantize(_bits(x), "mxfp4_mbs")["row"]
    check_mbs(r, ref, "linear")
    assert r.tensor_scale[5, 1].item() == 0.0


def test_mbs_full_size_activation(lib):
    """The activation-like 8192 x 4096 tensor, with the RHT, as one pass."""
    x = synth.activation(8192, 4096)
    r, _ = lib.fp4q_quantize(x.cuda(), fmt="mxfp4_mbs", rht=True, seed=1234)
    rs, _ = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(synth.bf16_bits(x), "mxfp4_mbs", rht=True, seed=1234)["row"]
    check_mbs(r, ref, "linear")
    check_stats(rs, ref["stats"])


def test_mx_rejections(lib):
    x = torch.randn(64, 384, device="cuda").to(torch.bfloat16)
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_quantize(x, fmt="mxfp4_mbs", axis="col")
    assert e.value.code == 1                        # rows % 128 (outer blocks down the columns)
    y = torch.randn(64, 272, device="cuda").to(torch.bfloat16)
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_quantize(y, fmt="mxfp4_mbs")
    assert e.value.code == 1                        # cols % 128
    a, _ = lib.fp4q_quantize(torch.randn(128, 256, device="cuda"), fmt="mxfp4_mbs", layout="mma")
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_gemm_dequant(a, a)
    assert e.value.code == 2


# ---- the native GEMM with E8M0 scales ----------------------------------------------

def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _e8m0_copy(lib, rng, fmt, rows, k, elo, ehi):
    blk = o.BLOCK[fmt]
    codes = rng.integers(0, 16, (rows, k)).astype(np.uint8)
    scales = (rng.integers(elo, ehi + 1, (rows, k // blk)) + 127).astype(np.uint8)
    cp = {"fmt": fmt, "codes": o.pack_nibbles(codes), "scales": scales, "tensor_scale": np.float32(1.0)}
    dev = "cuda"
    q = lib.QCopy(torch.from_numpy(cp["codes"]).to(dev),
                  torch.from_numpy(o.scales_to_mma_layout(scales, blk)).to(dev),
                  torch.ones(1, dtype=torch.float32, device=dev), fmt, rows, k, "mma")
    return cp, q


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp4_b16"])
@pytest.mark.parametrize("shape", [(128, 256, 256), (256, 128, 512), (128, 512, 768)])
def test_gemm_e8m0_exact(lib, fmt, shape):
    """Power-of-two block scales in a narrow range: every product and partial
    sum is exact in FP32, so the result must match the FP64 product bit for bit."""
    M, N, K = shape
    rng = np.random.default_rng(M * 7 + N + K)
    a, qa = _e8m0_copy(lib, rng, fmt, M, K, -2, 1)
    b, qb = _e8m0_copy(lib, rng, fmt, N, K, -2, 1)
    y = lib.fp4q_gemm(qa, qb, out_dtype=torch.float32).cpu().numpy()
    assert lib.fp4q_status() == 0
    ref = o.gemm(a, b)
    bad = np.argwhere(y != ref)
    assert bad.size == 0, f"{len(bad)} of {y.size} differ; first {bad[:6].tolist()}; rel {_rel(y, ref):.3e}"


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp4_b16", "mxfp4_oas"])
@pytest.mark.parametrize("shape", [(256, 512, 1024), (384, 128, 512), (512, 256, 2048)])
def test_quantize_then_gemm_e8m0(lib, fmt, shape, out_dtype):
    M, N, K = shape
    a = synth.gemm_operand("a", M, K)
    b = synth.gemm_operand("b", N, K)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt=fmt, rht=True, seed=1234, layout="mma")
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt=fmt, rht=True, seed=1234, layout="mma")
    y = lib.fp4q_gemm(qa, qb, out_dtype=out_dtype)
    assert lib.fp4q_status() == 0
    ra = o.quantize(_bits(a), fmt, rht=True, seed=1234)["row"]
    rb = o.quantize(_bits(b), fmt, rht=True, seed=1234)["row"]
    ref = o.gemm(ra, rb)
    if out_dtype == torch.float32:
        assert _rel(y.cpu().numpy(), ref) <= 1e-5
    else:
        want = o.bf16_bits_to_f32(o.f32_to_bf16_bits_rne(ref.astype(np.float32)))
        assert _rel(o.bf16_bits_to_f32(synth.bf16_bits(y.cpu())), want) <= 1e-3
