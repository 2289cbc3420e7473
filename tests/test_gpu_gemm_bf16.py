"""The dequantise-then-BF16 GEMM path (UFP4 on the contraction: "Replanteamiento
del Sesgo de Contraccion ...", Metodologia §2 and Resultados; MXFP4; NVFP4 for
comparison with the native block-scaled GEMM) against the oracle's FP64
dequantise-then-matmul. The BF16 operands are exact, so the only error is the
FP32 accumulation: a relative Frobenius error of 1e-5 leaves room for it at
K <= 1024 (the bound is about sqrt(K) 2^-24 per output)."""
import numpy as np
import pytest
import torch

import synth
from oracle import fp4q_oracle as o

pytestmark = pytest.mark.gpu


def _rel_fro(y, ref):
    return float(np.linalg.norm(y - ref) / np.linalg.norm(ref))


@pytest.mark.parametrize("fmt,rht", [("ufp4", True), ("ufp4", False), ("mxfp4", False), ("nvfp4", True),
                                     ("mxfp4_b16", False), ("mxfp4_oas", True)])
@pytest.mark.parametrize("layout", ["linear", "mma"])
@pytest.mark.parametrize("shape", [(256, 384, 512), (128, 128, 1024), (96, 200, 256)])
def test_gemm_via_bf16_against_oracle(lib, fmt, rht, layout, shape):
    M, N, K = shape
    a = synth.gemm_operand("a", M, K)
    b = synth.gemm_operand("b", N, K)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt=fmt, rht=rht, seed=77, layout=layout)
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt=fmt, rht=rht, seed=77, layout=layout)
    y = lib.fp4q_gemm_via_bf16(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    ra = o.quantize(synth.bf16_bits(a), fmt, rht=rht, seed=77)["row"]
    rb = o.quantize(synth.bf16_bits(b), fmt, rht=rht, seed=77)["row"]
    ref = o.gemm(ra, rb)
    assert _rel_fro(y, ref) < 1e-5
    yb = lib.fp4q_gemm_via_bf16(qa, qb, out_dtype=torch.bfloat16).float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(yb - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(ref).max())


def test_gemm_via_bf16_matches_native_nvfp4(lib):
    a = synth.gemm_operand("a", 256, 1024)
    b = synth.gemm_operand("b", 512, 1024)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt="nvfp4", rht=True, seed=5, layout="mma")
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt="nvfp4", rht=True, seed=5, layout="mma")
    y1 = lib.fp4q_gemm(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    y2 = lib.fp4q_gemm_via_bf16(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    assert _rel_fro(y2, y1) < 1e-5


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp4_oas"])
def test_gemm_via_bf16_matches_native_e8m0(lib, fmt):
    """The two routes for E8M0 operands agree: exact BF16 block values with a
    library GEMM, and the tensor cores with UE8M0 scales (MXFP4's 32-element
    scales stored for both halves of the tiled layout)."""
    a = synth.gemm_operand("a", 384, 768)
    b = synth.gemm_operand("b", 256, 768)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt=fmt, rht=True, seed=9, layout="mma")
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt=fmt, rht=True, seed=9, layout="mma")
    y1 = lib.fp4q_gemm(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    y2 = lib.fp4q_gemm_via_bf16(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    assert _rel_fro(y2, y1) < 1e-5


def test_gemm_via_bf16_rejections(lib):
    x = torch.randn(128, 256, device="cuda")
    q2, _ = lib.fp4q_quantize(x, fmt="nvfp4_2l")
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_gemm_via_bf16(q2, q2)
    assert e.value.code == 2
    q, _ = lib.fp4q_quantize(x, fmt="ufp4")
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_gemm_via_bf16(q, q, scratch=small)
    assert e.value.code == 1
