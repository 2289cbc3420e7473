"""GPU parity of the block-scaled NVFP4 GEMM against the oracle's FP64
dequantise-then-matmul.

Bars: FP32 output within Frobenius relative error 1e-5 of the FP64 product
(FP32 accumulation over K <= 8192); BF16 output within 1e-3 of the FP64
product rounded to BF16 (the output format is part of what is computed); an
exactly representable case (power-of-two scales in a narrow range, g = 1)
must match bit for bit.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import fp4q_oracle as o

pytestmark = pytest.mark.gpu


def _bits(t):
    return synth.bf16_bits(t.cpu())


def _qcopy(lib, codes, scales_linear, g, rows, cols):
    """Wrap host-built codes / scales as a device copy with tiled scales."""
    dev = "cuda"
    c = torch.from_numpy(np.ascontiguousarray(codes)).to(dev)
    s = torch.from_numpy(o.scales_to_mma_layout(scales_linear)).to(dev)
    ts = torch.tensor([g], dtype=torch.float32, device=dev)
    return lib.QCopy(c, s, ts, "nvfp4", rows, cols, "mma")


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _rand_copy(rng, rows, k, kexp_lo, kexp_hi):
    codes = rng.integers(0, 16, (rows, k)).astype(np.uint8)
    kexp = rng.integers(kexp_lo, kexp_hi + 1, (rows, k // 16))
    scales = ((kexp + 7) << 3).astype(np.uint8)           # E4M3 code of 2^kexp
    cp = {"fmt": "nvfp4", "codes": o.pack_nibbles(codes), "scales": scales,
          "tensor_scale": np.float32(1.0)}
    return cp


@pytest.mark.parametrize("variant", ["unit", "a_scales", "b_scales", "both"])
@pytest.mark.parametrize("shape", [(128, 256, 256), (128, 128, 512), (256, 512, 768), (512, 256, 512),
                                   (1024, 512, 256), (384, 768, 512), (256, 256, 256), (4096, 4096, 256),
                                   (2304, 2560, 512)])
def test_gemm_exact_power_of_two(lib, variant, shape):
    """M and N multiples of 256 run on CTA pairs (one 256 x 256 tile per pair,
    several tiles per pair at 4096 x 4096), other shapes on single CTAs."""
    M, N, K = shape
    rng = np.random.default_rng(M + N + K)
    a = _rand_copy(rng, M, K, 0 if variant in ("unit", "b_scales") else -2,
                   0 if variant in ("unit", "b_scales") else 1)
    b = _rand_copy(rng, N, K, 0 if variant in ("unit", "a_scales") else -2,
                   0 if variant in ("unit", "a_scales") else 1)
    ga = _qcopy(lib, a["codes"], a["scales"], 1.0, M, K)
    gb = _qcopy(lib, b["codes"], b["scales"], 1.0, N, K)
    y = lib.fp4q_gemm(ga, gb, out_dtype=torch.float32).cpu().numpy()
    ref = o.gemm(a, b)
    assert lib.fp4q_status() == 0
    bad = np.argwhere(y != ref)
    assert bad.size == 0, (f"{len(bad)} of {y.size} differ; first {bad[:6].tolist()}; "
                           f"rel {_rel(y, ref):.3e}")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(256, 512, 1024), (384, 128, 512), (128, 384, 2048), (512, 512, 1024),
                                   (1024, 256, 512), (512, 384, 768)])
def test_quantize_then_gemm(lib, shape, out_dtype):
    M, N, K = shape
    a = synth.gemm_operand("a", M, K)
    b = synth.gemm_operand("b", N, K)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt="nvfp4", rht=True, seed=1234, layout="mma")
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt="nvfp4", rht=True, seed=1234, layout="mma")
    y = lib.fp4q_gemm(qa, qb, out_dtype=out_dtype)
    ra = o.quantize(_bits(a), "nvfp4", rht=True, seed=1234)["row"]
    rb = o.quantize(_bits(b), "nvfp4", rht=True, seed=1234)["row"]
    ref = o.gemm(ra, rb)
    if out_dtype == torch.float32:
        assert _rel(y.cpu().numpy(), ref) < 1e-5
    else:
        got = y.float().cpu().numpy()
        ref_bf16 = o.bf16_bits_to_f32(o.f32_to_bf16_bits_rne(ref.astype(np.float32)))
        assert _rel(got, ref_bf16) < 1e-3
        assert _rel(got, ref) < 5e-3
    assert lib.fp4q_status() == 0


def test_gemm_full_size_sampled(lib):
    """A, B 8192 x 8192 N(0, 1/8192), NVFP4 with RHT along K, Y = A B^T in BF16:
    2 x 64 sampled rows and columns of Y against the FP64 oracle; SNR of Y
    against the BF16-input product reported."""
    n = 8192
    a = synth.gemm_operand("a", n, n)
    b = synth.gemm_operand("b", n, n)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt="nvfp4", rht=True, seed=1234, layout="mma")
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt="nvfp4", rht=True, seed=1234, layout="mma")
    y = lib.fp4q_gemm(qa, qb, out_dtype=torch.bfloat16)
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(n, 64, replace=False))
    cols = np.sort(rng.choice(n, 64, replace=False))
    ra = o.quantize(_bits(a), "nvfp4", rht=True, seed=1234, rows_subset=rows)["row"]
    rb = o.quantize(_bits(b), "nvfp4", rht=True, seed=1234, rows_subset=cols)["row"]
    # the operands themselves: sampled rows of A and of B (codes, tiled scales,
    # tensor scale from the whole operand) against the oracle, bit for bit
    for q, r, sel in ((qa, ra, rows), (qb, rb, cols)):
        idx = torch.from_numpy(sel).cuda()
        assert np.array_equal(q.codes[idx].cpu().numpy(), r["codes"])
        nkb = n // 16
        nkb_p = -(-nkb // 4) * 4
        rr, kb = np.meshgrid(sel, np.arange(nkb), indexing="ij")
        off = torch.from_numpy(o.mma_scale_offset(rr, kb, nkb_p).astype(np.int64)).cuda()
        assert np.array_equal(q.scales[off].cpu().numpy(), r["scales"])
        assert np.float32(r["tensor_scale"]).view(np.uint32) == q.tensor_scale.cpu().numpy().view(np.uint32)[0]
    yref = o.gemm(ra, rb)                       # the sampled rows x cols block, FP64
    got = y[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].float().cpu().numpy()
    ref_bf16 = o.bf16_bits_to_f32(o.f32_to_bf16_bits_rne(yref.astype(np.float32)))
    assert _rel(got, ref_bf16) < 1e-3
    exact = (a.float()[rows] @ b.float()[cols].T).double().numpy()
    snr = o.snr_db(exact, got)
    assert 15.0 < snr < 40.0, snr
    assert lib.fp4q_status() == 0


@pytest.mark.parametrize("m", [256, 128])
def test_bounded_wait_runs_out_without_fault(lib, m):
    """Failure detection on the device: the first CTA's producer withholds one
    stage, the waits that depend on it run out after 20 ms, the kernel records
    FP4Q_ETIMEOUT and returns; the context stays usable and the next GEMM on
    it is correct. M = 256 runs the two-SM kernel (the pair's waits, relays and
    cross-CTA commits), M = 128 the one-SM kernel."""
    a = synth.gemm_operand("a", m, 512)
    b = synth.gemm_operand("b", 256, 512)
    qa, _ = lib.fp4q_quantize(a.cuda(), fmt="nvfp4", layout="mma")
    qb, _ = lib.fp4q_quantize(b.cuda(), fmt="nvfp4", layout="mma")
    assert lib.fp4q_status() == 0
    lib.fp4q_gemm_selftest_timeout(qa, qb, 20_000_000)
    assert lib.fp4q_status() == 5          # FP4Q_ETIMEOUT, read and cleared
    assert lib.fp4q_status() == 0
    y = lib.fp4q_gemm(qa, qb, out_dtype=torch.float32)
    assert lib.fp4q_status() == 0
    ra = o.quantize(_bits(a), "nvfp4")["row"]
    rb = o.quantize(_bits(b), "nvfp4")["row"]
    assert _rel(y.cpu().numpy(), o.gemm(ra, rb)) < 1e-5
