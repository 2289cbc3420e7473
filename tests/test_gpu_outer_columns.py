"""GPU parity of the column-wise (transposed) copies of the formats with a
scale per 128 elements: two-level NVFP4 ("TetraJet-v2 ...", Riepilogo Tecnico
§2A: the transposed copy for the weight gradient, the double-block scale) and
MBS-static ("Unveiling the Potential of Quantization with MXFP4 ...", Resume
technique §2B). In the column-wise copy the 16-element blocks and the
128-element outer blocks run down the source's columns. Codes, inner scales
and outer scales are bit-exact with the oracle's copy of X^T; dequantised
values bit-exact; statistics within the tolerance of the other tests."""
import numpy as np
import pytest
import torch

import synth
from oracle import fp4q_oracle as o

from test_gpu_quantize import _bits, _input, check_stats
from test_gpu_two_level import check_two_level
from test_gpu_mx_variants import check_mbs

pytestmark = pytest.mark.gpu

CHECK = {"nvfp4_2l": check_two_level, "mxfp4_mbs": check_mbs}


@pytest.mark.parametrize("fmt", ["nvfp4_2l", "mxfp4_mbs"])
@pytest.mark.parametrize("layout", ["linear", "mma"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding", ["rtne", "sr"])
@pytest.mark.parametrize("rht", [False, True])
def test_column_copy_parity(lib, fmt, rht, rounding, dtype, layout):
    """384 rows (three outer blocks per column) x 208 columns (a ragged last
    tile of 80 columns)."""
    x = _input("nvfp4", dtype, seed=41, shape=(384, 208))
    _, c = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=rht, rounding=rounding, seed=99, axis="col", layout=layout)
    _, cs = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(_bits(x), fmt, rht=rht, rounding=rounding, seed=99, axis="col")["col"]
    CHECK[fmt](c, ref, layout)
    check_stats(cs, ref["stats"])


@pytest.mark.parametrize("fmt", ["nvfp4_2l", "mxfp4_mbs"])
@pytest.mark.parametrize("rht", [False, True])
def test_both_copies_and_statistics(lib, fmt, rht):
    """Both copies from one call (the row kernel, then the column kernel): each
    copy and each copy's statistics against the oracle, twice in a row on one
    workspace, after a call with a larger grid left other partials behind."""
    ws = torch.zeros(lib.fp4q_workspace_size(), dtype=torch.uint8, device="cuda")
    big = _input("nvfp4", torch.bfloat16, seed=3, shape=(2048, 1024))
    lib.fp4q_quantize(big.cuda(), fmt="nvfp4", rht=True, seed=1, axis="both", ws=ws)
    x = _input("nvfp4", torch.bfloat16, seed=42, shape=(256, 384))
    ref = o.quantize(_bits(x), fmt, rht=rht, seed=7, axis="both")
    for _ in range(2):
        r, c = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=rht, seed=7, axis="both", ws=ws)
        rs, cs = lib.fp4q_stats(ws)
        assert lib.fp4q_status(ws) == 0
        CHECK[fmt](r, ref["row"], "linear")
        CHECK[fmt](c, ref["col"], "linear")
        check_stats(rs, ref["row"]["stats"])
        check_stats(cs, ref["col"]["stats"])


@pytest.mark.parametrize("fmt", ["nvfp4_2l", "mxfp4_mbs"])
@pytest.mark.parametrize("rht", [False, True])
def test_column_copy_dequantize(lib, fmt, rht):
    x = _input("nvfp4", torch.bfloat16, seed=43, shape=(256, 96))
    _, c = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=rht, seed=5, axis="col")
    y = lib.fp4q_dequantize(c, inverse_rht=rht, seed=5, out_dtype=torch.float32)
    ref = o.quantize(_bits(x), fmt, rht=rht, seed=5, axis="col")["col"]
    if fmt == "nvfp4_2l":
        want = o.dequantize_two_level(ref["codes"], ref["scales"], ref["outer_scales"], rht, 5)
    else:
        want = o.dequantize_mbs(ref["codes"], ref["scales"], ref["macro_scales"], rht, 5)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_column_copy_zero_outer_blocks(lib):
    x = torch.randn(256, 64).to(torch.bfloat16)
    x[128:256, 5] = 0.0
    x[:128, 9] = -0.0
    for fmt in ("nvfp4_2l", "mxfp4_mbs"):
        _, c = lib.fp4q_quantize(x.cuda(), fmt=fmt, axis="col")
        ref = o.quantize(_bits(x), fmt, axis="col")["col"]
        CHECK[fmt](c, ref, "linear")
        assert c.tensor_scale[5, 1].item() == 0.0 and c.tensor_scale[9, 0].item() == 0.0


def test_column_copy_rejections(lib):
    x = torch.randn(200, 256, device="cuda").to(torch.bfloat16)     # 200 % 128 != 0
    for fmt in ("nvfp4_2l", "mxfp4_mbs"):
        with pytest.raises(lib.FP4QError) as e:
            lib.fp4q_quantize(x, fmt=fmt, axis="col")
        assert e.value.code == 1


@pytest.mark.parametrize("fmt", ["nvfp4_2l", "mxfp4_mbs"])
def test_gradient_both_copies_full_size_sampled(lib, fmt):
    """The gradient workload's shape (4096 x 14336 BF16, N(0, 1e-6) with 0.1%
    x100), RHT and Philox SR, both copies from one call, on sampled rows of
    each copy (both ends, tile and outer-block boundaries, a seeded spread)."""
    x = synth.gradient("a")
    rows, cols = x.shape
    r, c = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=True, rounding="sr", seed=1234, axis="both")
    assert lib.fp4q_status() == 0
    rng = np.random.default_rng(7)
    rsel = np.unique(np.concatenate([[0, 1, 127, 128, rows - 1], rng.integers(0, rows, 24)])).astype(np.int64)
    csel = np.unique(np.concatenate([[0, 1, 127, 128, cols - 1], rng.integers(0, cols, 24)])).astype(np.int64)
    ref = o.quantize(synth.bf16_bits(x), fmt, rht=True, rounding="sr", seed=1234, axis="both",
                     rows_subset=rsel, cols_subset=csel)
    key = "outer_scales" if fmt == "nvfp4_2l" else "macro_scales"
    for got, want, sel in ((r, ref["row"], rsel), (c, ref["col"], csel)):
        idx = torch.from_numpy(sel).cuda()
        assert np.array_equal(got.codes[idx].cpu().numpy(), want["codes"])
        assert np.array_equal(got.scales[idx].cpu().numpy(), want["scales"])
        assert np.array_equal(got.tensor_scale[idx].cpu().numpy().view(np.uint32), want[key].view(np.uint32))
