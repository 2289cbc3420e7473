"""The GEMM on dequantised operands (UFP4 on the contraction: "Replanteamiento
del Sesgo de Contraccion ...", Metodologia §2 and Resultados; NVFP4 and the
E8M0 formats for comparison with the block-scaled GEMM) against the oracle's
FP64 dequantise-then-matmul.

The kernel forms each block value level * s_b exactly in FP16 (UFP4, NVFP4)
or BF16 (E8M0 formats) in shared memory, and the tensor cores multiply them
with FP32 accumulation. The products are exact, so the only error is the
FP32 accumulation over K: a relative Frobenius error of 1e-5 leaves room for
it at K <= 1024 (about sqrt(K) 2^-24 per output). A case whose every partial
sum is representable must match bit for bit."""
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
@pytest.mark.parametrize("shape", [(256, 384, 512), (128, 128, 1024), (96, 200, 256), (130, 264, 64)])
def test_gemm_dequant_against_oracle(lib, fmt, rht, layout, shape):
    """Tile multiples and ragged M and N (rows past the operand are zeros and
    never stored)."""
    M, N, K = shape
    a = synth.gemm_operand("a", M, K)
    b = synth.gemm_operand("b", N, K)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt=fmt, rht=rht, seed=77, layout=layout)
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt=fmt, rht=rht, seed=77, layout=layout)
    y = lib.fp4q_gemm_dequant(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    assert lib.fp4q_status() == 0
    ra = o.quantize(synth.bf16_bits(a), fmt, rht=rht, seed=77)["row"]
    rb = o.quantize(synth.bf16_bits(b), fmt, rht=rht, seed=77)["row"]
    ref = o.gemm(ra, rb)
    assert _rel_fro(y, ref) < 1e-5
    yb = lib.fp4q_gemm_dequant(qa, qb, out_dtype=torch.bfloat16).float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(yb - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(ref).max())


def test_gemm_dequant_ufp4_exact(lib):
    """UFP4 with power-of-two block scales and g = 1: every product and every
    partial sum over K = 512 is a small dyadic number that FP32 holds, so the
    output matches the FP64 oracle bit for bit. Several tiles per CTA
    (4096 x 2560 outputs in 128 x 256 tiles: 320 tiles)."""
    rng = np.random.default_rng(11)
    M, N, K = 4096, 2560, 512

    def copy(rows):
        codes = rng.integers(0, 16, (rows, K)).astype(np.uint8)
        kexp = rng.integers(-2, 2, (rows, K // 16))
        scales = ((kexp + 7) << 3).astype(np.uint8)          # E4M3 code of 2^kexp
        return {"fmt": "ufp4", "codes": o.pack_nibbles(codes), "scales": scales, "tensor_scale": np.float32(1.0)}

    ca, cb = copy(M), copy(N)

    def dev(c, rows):
        return lib.QCopy(torch.from_numpy(c["codes"]).cuda(), torch.from_numpy(c["scales"]).cuda(),
                         torch.ones(1, dtype=torch.float32, device="cuda"), "ufp4", rows, K, "linear")

    y = lib.fp4q_gemm_dequant(dev(ca, M), dev(cb, N), out_dtype=torch.float32).cpu().numpy()
    ref = o.gemm(ca, cb)
    assert lib.fp4q_status() == 0
    bad = np.argwhere(y != ref)
    assert bad.size == 0, f"{len(bad)} of {y.size} differ; first {bad[:6].tolist()}"


def test_fp4q_gemm_routes_ufp4_to_the_dequant_kernel(lib):
    """fp4q_gemm takes UFP4 (no tensor-core format) through the same kernel."""
    a = synth.gemm_operand("a", 256, 1024)
    b = synth.gemm_operand("b", 512, 1024)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt="ufp4", rht=True, seed=5, layout="mma")
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt="ufp4", rht=True, seed=5, layout="mma")
    y1 = lib.fp4q_gemm(qa, qb, out_dtype=torch.float32)
    y2 = lib.fp4q_gemm_dequant(qa, qb, out_dtype=torch.float32)
    assert torch.equal(y1, y2)


def test_gemm_dequant_matches_native_nvfp4(lib):
    a = synth.gemm_operand("a", 256, 1024)
    b = synth.gemm_operand("b", 512, 1024)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt="nvfp4", rht=True, seed=5, layout="mma")
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt="nvfp4", rht=True, seed=5, layout="mma")
    y1 = lib.fp4q_gemm(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    y2 = lib.fp4q_gemm_dequant(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    assert _rel_fro(y2, y1) < 1e-5


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp4_oas"])
def test_gemm_dequant_matches_native_e8m0(lib, fmt):
    """The two routes for E8M0 operands agree: exact BF16 block values on the
    16-bit MMA, and the block-scaled MMA with UE8M0 scales."""
    a = synth.gemm_operand("a", 384, 768)
    b = synth.gemm_operand("b", 256, 768)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt=fmt, rht=True, seed=9, layout="mma")
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt=fmt, rht=True, seed=9, layout="mma")
    y1 = lib.fp4q_gemm(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    y2 = lib.fp4q_gemm_dequant(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    assert _rel_fro(y2, y1) < 1e-5


def test_gemm_dequant_rejections(lib):
    x = torch.randn(128, 256, device="cuda")
    q2, _ = lib.fp4q_quantize(x, fmt="nvfp4_2l")
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_gemm_dequant(q2, q2)
    assert e.value.code == 2
    q, _ = lib.fp4q_quantize(torch.randn(128, 96, device="cuda"), fmt="ufp4")
    with pytest.raises(lib.FP4QError) as e:          # K % 64
        lib.fp4q_gemm_dequant(q, q)
    assert e.value.code == 1
    qa, _ = lib.fp4q_quantize(torch.randn(128, 256, device="cuda"), fmt="ufp4")
    qb, _ = lib.fp4q_quantize(torch.randn(100, 256, device="cuda"), fmt="ufp4")
    with pytest.raises(lib.FP4QError) as e:          # N % 8
        lib.fp4q_gemm_dequant(qa, qb)
    assert e.value.code == 1


@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("shape", [(256, 384, 512), (128, 128, 1024), (96, 200, 256), (130, 264, 64)])
def test_gemm_dequant_hif4_against_oracle(lib, rht, shape):
    """HiF4 ("Unleashing Low-Bit Inference on Ascend NPUs ...", Resumen técnico
    §2) on the 16-bit MMA: block values level * S * 2^-(d_8 + d_4) exact in
    BF16, one scale word per row and 64-element K stage."""
    M, N, K = shape
    a = synth.gemm_operand("a", M, K)
    b = synth.gemm_operand("b", N, K)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt="hif4", rht=rht, seed=77)
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt="hif4", rht=rht, seed=77)
    y = lib.fp4q_gemm_dequant(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    assert lib.fp4q_status() == 0
    ra = o.quantize(synth.bf16_bits(a), "hif4", rht=rht, seed=77)["row"]
    rb = o.quantize(synth.bf16_bits(b), "hif4", rht=rht, seed=77)["row"]
    ref = o.gemm(ra, rb)
    assert _rel_fro(y, ref) < 1e-5
    y2 = lib.fp4q_gemm(qa, qb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    assert np.array_equal(y, y2)                       # fp4q_gemm takes HiF4 through the same kernel


def test_gemm_dequant_hif4_exact(lib):
    """HiF4 with scales 2^-1 or 2^0 and random halving bits: every product is
    k 2^p with k <= 49 and -6 <= p <= 0, every partial sum over K = 512 fits
    FP32 exactly, so the output equals the FP64 oracle bit for bit. Random
    codes and words exercise every bit of the scale word."""
    rng = np.random.default_rng(12)
    M, N, K = 512, 768, 512

    def copy(rows):
        codes = rng.integers(0, 16, (rows, K)).astype(np.uint8)
        e6m2 = np.where(rng.random((rows, K // 64)) < 0.5, 120, 124).astype(np.uint32)     # 2^-1, 2^0
        bits = rng.integers(0, 1 << 24, (rows, K // 64), dtype=np.int64).astype(np.uint32)
        words = (e6m2 | (bits << np.uint32(8))).astype(np.uint32)
        return {"fmt": "hif4", "codes": o.pack_nibbles(codes), "scales": words}

    ca, cb = copy(M), copy(N)

    def dev(c, rows):
        return lib.QCopy(torch.from_numpy(c["codes"]).cuda(), torch.from_numpy(c["scales"].view(np.int32)).cuda(),
                         torch.ones(1, dtype=torch.float32, device="cuda"), "hif4", rows, K, "linear")

    y = lib.fp4q_gemm_dequant(dev(ca, M), dev(cb, N), out_dtype=torch.float32).cpu().numpy()
    ref = o.gemm(ca, cb)
    assert lib.fp4q_status() == 0
    bad = np.argwhere(y != ref)
    assert bad.size == 0, f"{len(bad)} of {y.size} differ; first {bad[:6].tolist()}"


@pytest.mark.parametrize("fmt", ["ufp4", "hif4"])
def test_gemm_dequant_full_size_sampled(lib, fmt):
    """The bench's dequantising-GEMM workloads: A, B 8192 x 8192 N(0, 1/8192),
    UFP4 (tiled scales) or HiF4 (linear scale words) with the RHT along K,
    Y = A B^T through fp4q_gemm. Sampled rows of both operands bit for bit
    against the oracle's quantisation, then the 64 x 64 sampled block of Y
    (FP32 out) within the FP32-accumulation bound at K = 8192 (~sqrt(K) 2^-24)."""
    n = 8192
    a = synth.gemm_operand("a", n, n)
    b = synth.gemm_operand("b", n, n)
    layout = "linear" if fmt == "hif4" else "mma"
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt=fmt, rht=True, seed=1234, layout=layout)
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt=fmt, rht=True, seed=1234, layout=layout)
    y = lib.fp4q_gemm(qa, qb, out_dtype=torch.float32)
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(n, 64, replace=False))
    cols = np.sort(rng.choice(n, 64, replace=False))
    ra = o.quantize(synth.bf16_bits(a), fmt, rht=True, seed=1234, rows_subset=rows)["row"]
    rb = o.quantize(synth.bf16_bits(b), fmt, rht=True, seed=1234, rows_subset=cols)["row"]
    for q, r, sel in ((qa, ra, rows), (qb, rb, cols)):
        idx = torch.from_numpy(sel).cuda()
        assert np.array_equal(q.codes[idx].cpu().numpy(), r["codes"])
        if fmt == "hif4":
            assert np.array_equal(q.scales[idx].cpu().numpy().view(np.uint32), r["scales"])
        else:
            nkb = n // 16
            rr, kb = np.meshgrid(sel, np.arange(nkb), indexing="ij")
            off = torch.from_numpy(o.mma_scale_offset(rr, kb, -(-nkb // 4) * 4).astype(np.int64)).cuda()
            assert np.array_equal(q.scales[off].cpu().numpy(), r["scales"])
            assert np.float32(r["tensor_scale"]).view(np.uint32) == q.tensor_scale.cpu().numpy().view(np.uint32)[0]
    ref = o.gemm(ra, rb)
    got = y[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy().astype(np.float64)
    assert _rel_fro(got, ref) < 2e-5
    assert lib.fp4q_status() == 0
