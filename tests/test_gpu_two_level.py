"""GPU parity of two-level NVFP4 (the double-block scale of TetraJet-v2,
Riepilogo Tecnico §2A: an FP32 scale per 128-element outer block, E4M3 scales
per 16-element inner block, no tensor amax) against the CPU oracle: codes,
inner scales and outer scales bit-exact, dequantised values bit-exact,
statistics within the tolerance of the one-level tests."""
import numpy as np
import pytest
import torch

import synth
from oracle import fp4q_oracle as o

from test_gpu_quantize import _bits, _input, check_stats

pytestmark = pytest.mark.gpu

FMT = "nvfp4_2l"


def check_two_level(gq, oq, layout):
    codes = gq.codes.cpu().numpy()
    mism = np.flatnonzero(codes.ravel() != oq["codes"].ravel())
    assert mism.size == 0, f"{mism.size} code bytes differ, first at {mism[:5]}"
    sc = gq.scales.cpu().numpy()
    if layout == "linear":
        assert np.array_equal(sc, oq["scales"])
    else:
        assert np.array_equal(sc.ravel(), o.scales_to_mma_layout(oq["scales"]))
    g = gq.tensor_scale.cpu().numpy()
    if layout == "mma":                 # the tiled layout keeps the outer scales column-major
        g = np.ascontiguousarray(g.T)
    assert g.shape == oq["outer_scales"].shape
    assert np.array_equal(g.view(np.uint32), oq["outer_scales"].view(np.uint32))


@pytest.mark.parametrize("layout", ["linear", "mma"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding", ["rtne", "sr"])
@pytest.mark.parametrize("rht", [False, True])
def test_two_level_parity(lib, rht, rounding, dtype, layout):
    x = _input("nvfp4", dtype, seed=17, shape=(208, 384))     # 9.75 chunks: a ragged last chunk
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT, rht=rht, rounding=rounding, seed=321, layout=layout)
    rs, _ = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(_bits(x), FMT, rht=rht, rounding=rounding, seed=321)["row"]
    check_two_level(r, ref, layout)
    check_stats(rs, ref["stats"])


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rht", [False, True])
def test_two_level_dequantize(lib, rht, out_dtype):
    x = _input("nvfp4", torch.bfloat16, seed=18, shape=(96, 512))
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT, rht=rht, seed=5)
    y = lib.fp4q_dequantize(r, inverse_rht=rht, seed=5, out_dtype=out_dtype)
    ref = o.quantize(_bits(x), FMT, rht=rht, seed=5)["row"]
    want = o.dequantize_two_level(ref["codes"], ref["scales"], ref["outer_scales"], rht, 5)
    if out_dtype == torch.float32:
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))
    else:
        assert np.array_equal(synth.bf16_bits(y.cpu()), o.f32_to_bf16_bits_rne(want))


@pytest.mark.parametrize("mag", [1e-30, 1e30])
def test_two_level_extreme_magnitudes(lib, mag):
    x = (_input("nvfp4", torch.float32, seed=3, shape=(64, 256)) * mag).float()
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT)
    rs, _ = lib.fp4q_stats()
    ref = o.quantize(x.numpy(), FMT)["row"]
    check_two_level(r, ref, "linear")
    check_stats(rs, ref["stats"])


def test_two_level_zero_outer_blocks(lib):
    x = torch.randn(32, 384).to(torch.bfloat16)
    x[3, 128:256] = 0.0
    x[7, :128] = -0.0
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT)
    ref = o.quantize(_bits(x), FMT)["row"]
    check_two_level(r, ref, "linear")
    assert r.tensor_scale[3, 1].item() == 0.0


def test_two_level_full_size_activation(lib):
    """The activation-like 8192 x 4096 tensor, with the RHT, as one pass."""
    x = synth.activation(8192, 4096)
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT, rht=True, seed=1234)
    rs, _ = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(synth.bf16_bits(x), FMT, rht=True, seed=1234)["row"]
    check_two_level(r, ref, "linear")
    check_stats(rs, ref["stats"])


def test_two_level_rejections(lib):
    x = torch.randn(64, 384, device="cuda").to(torch.bfloat16)
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_quantize(x, fmt=FMT, axis="col")
    assert e.value.code == 1                        # rows % 128 (outer blocks down the columns)
    y = torch.randn(64, 272, device="cuda").to(torch.bfloat16)
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_quantize(y, fmt=FMT)
    assert e.value.code == 1                        # cols % 128
    a, _ = lib.fp4q_quantize(torch.randn(128, 256, device="cuda"), fmt=FMT, layout="linear")
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_gemm(a, a)                         # the GEMM needs the tiled layouts
    assert e.value.code == 1
