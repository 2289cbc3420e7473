"""GPU parity of the GEMM on operands with an FP32 scale per 128 elements
along K (two-level NVFP4, "TetraJet-v2 ...", Riepilogo Tecnico §2A; MBS-static,
"Unveiling the Potential of Quantization with MXFP4 ...", Resume technique
§2B) against the oracle's FP64 dequantise-then-matmul.

Bars as for the one-scale GEMM: FP32 output within Frobenius relative error
1e-5 of the FP64 product, BF16 output within 1e-3 of the FP64 product rounded
to BF16; with power-of-two inner and outer scales in a narrow range every
product and partial sum is exact in FP32, and the result must match bit for
bit."""
import numpy as np
import pytest
import torch

import synth
from oracle import fp4q_oracle as o

pytestmark = pytest.mark.gpu


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _host_copy(lib, rng, fmt, rows, k):
    """Random codes, power-of-two inner scales in [1/2, 1] and outer scales in
    [1/2, 2], laid out as the tiled (GEMM) layouts."""
    codes = rng.integers(0, 16, (rows, k)).astype(np.uint8)
    e = rng.integers(-1, 1, (rows, k // 16))
    scales = (((e + 7) << 3) if fmt == "nvfp4_2l" else (e + 127)).astype(np.uint8)
    outer = np.exp2(rng.integers(-1, 2, (rows, k // 128))).astype(np.float32)
    key = "outer_scales" if fmt == "nvfp4_2l" else "macro_scales"
    cp = {"fmt": fmt, "codes": o.pack_nibbles(codes), "scales": scales, key: outer}
    dev = "cuda"
    q = lib.QCopy(torch.from_numpy(cp["codes"]).to(dev), torch.from_numpy(o.scales_to_mma_layout(scales)).to(dev),
                  torch.from_numpy(np.ascontiguousarray(outer.T)).to(dev), fmt, rows, k, "mma")
    return cp, q


@pytest.mark.parametrize("fmt", ["nvfp4_2l", "mxfp4_mbs"])
@pytest.mark.parametrize("shape", [(128, 128, 256), (256, 384, 512), (384, 256, 768)])
def test_gemm_outer_exact(lib, fmt, shape):
    M, N, K = shape
    rng = np.random.default_rng(M + 3 * N + K)
    a, qa = _host_copy(lib, rng, fmt, M, K)
    b, qb = _host_copy(lib, rng, fmt, N, K)
    y = lib.fp4q_gemm(qa, qb, out_dtype=torch.float32).cpu().numpy()
    assert lib.fp4q_status() == 0
    ref = o.gemm(a, b)
    bad = np.argwhere(y != ref)
    assert bad.size == 0, f"{len(bad)} of {y.size} differ; first {bad[:6].tolist()}; rel {_rel(y, ref):.3e}"


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", ["nvfp4_2l", "mxfp4_mbs"])
@pytest.mark.parametrize("shape", [(256, 512, 1024), (384, 128, 512), (128, 384, 2048), (512, 256, 768)])
def test_quantize_then_gemm_outer(lib, fmt, shape, out_dtype):
    M, N, K = shape
    a = synth.gemm_operand("a", M, K)
    b = synth.gemm_operand("b", N, K)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt=fmt, rht=True, seed=1234, layout="mma")
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt=fmt, rht=True, seed=1234, layout="mma")
    y = lib.fp4q_gemm(qa, qb, out_dtype=out_dtype)
    assert lib.fp4q_status() == 0
    ra = o.quantize(synth.bf16_bits(a), fmt, rht=True, seed=1234)["row"]
    rb = o.quantize(synth.bf16_bits(b), fmt, rht=True, seed=1234)["row"]
    ref = o.gemm(ra, rb)
    if out_dtype == torch.float32:
        assert _rel(y.cpu().numpy(), ref) <= 1e-5
    else:
        want = o.bf16_bits_to_f32(o.f32_to_bf16_bits_rne(ref.astype(np.float32)))
        assert _rel(o.bf16_bits_to_f32(synth.bf16_bits(y.cpu())), want) <= 1e-3


def test_gemm_outer_full_size_sampled(lib):
    """8192^3 two-level NVFP4 with the RHT: sampled rows and columns of Y
    against the oracle."""
    n = 8192
    a = synth.gemm_operand("a", n, n)
    b = synth.gemm_operand("b", n, n)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt="nvfp4_2l", rht=True, seed=1234, layout="mma")
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt="nvfp4_2l", rht=True, seed=1234, layout="mma")
    y = lib.fp4q_gemm(qa, qb, out_dtype=torch.float32)
    assert lib.fp4q_status() == 0
    rows = np.arange(5, n, 997)
    cols = np.arange(11, n, 1013)
    ra = o.quantize(synth.bf16_bits(a), "nvfp4_2l", rht=True, seed=1234, rows_subset=rows)["row"]
    rb = o.quantize(synth.bf16_bits(b), "nvfp4_2l", rht=True, seed=1234, rows_subset=cols)["row"]
    ref = o.gemm(ra, rb)
    got = y.cpu().numpy()[np.ix_(rows, cols)]
    assert _rel(got, ref) <= 1e-5
