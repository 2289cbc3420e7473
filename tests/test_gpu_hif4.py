"""GPU parity of HiF4 ("Unleashing Low-Bit Inference on Ascend NPUs: A
Comprehensive Evaluation of HiFloat Formats", Resumen técnico §2 Metodología:
an E6M2 scale per 64 elements, E1M0 factors per 8 and per 4 elements, E1M2
elements) against the CPU oracle: codes and scale words bit-exact, dequantised
values bit-exact, statistics within the tolerance of the other formats."""
import os

import numpy as np
import pytest
import torch

import synth
from oracle import fp4q_oracle as o

from test_gpu_quantize import _bits, check_stats

pytestmark = pytest.mark.gpu

FMT = "hif4"


def _grouped(rows, cols, seed, dtype=torch.bfloat16):
    """N(0,1) values whose 8-element groups carry a log-uniform magnitude over
    e^-3 .. e^3, plus 2% outliers x30: every combination of the per-8 and
    per-4 factors occurs."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g)
    x = x * torch.exp(torch.rand(rows, cols // 8, 1, generator=g) * 6 - 3).expand(-1, -1, 8).reshape(rows, cols)
    x = torch.where(torch.rand(rows, cols, generator=g) < 0.02, x * 30, x)
    return x.to(dtype)


def check_hif4(gq, oq):
    codes = gq.codes.cpu().numpy()
    mism = np.flatnonzero(codes.ravel() != oq["codes"].ravel())
    assert mism.size == 0, f"{mism.size} code bytes differ, first at {mism[:5]}"
    words = gq.scales.cpu().numpy().view(np.uint32)
    assert words.shape == oq["scales"].shape
    bad = np.flatnonzero(words.ravel() != oq["scales"].ravel())
    assert bad.size == 0, f"{bad.size} scale words differ, first {bad[:3]}: " \
                          f"{[hex(int(w)) for w in words.ravel()[bad[:3]]]} vs " \
                          f"{[hex(int(w)) for w in oq['scales'].ravel()[bad[:3]]]}"
    assert gq.tensor_scale.cpu().numpy()[0] == 1.0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding", ["rtne", "sr"])
@pytest.mark.parametrize("rht", [False, True])
def test_hif4_parity(lib, rht, rounding, dtype):
    x = _grouped(208, 384, 17, dtype)                 # 9.75 chunks of 8192: a ragged last chunk
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT, rht=rht, rounding=rounding, seed=321)
    rs, _ = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(_bits(x), FMT, rht=rht, rounding=rounding, seed=321)["row"]
    check_hif4(r, ref)
    check_stats(rs, ref["stats"])


@pytest.mark.parametrize("shape", [(1, 64), (3, 192), (127, 64), (64, 8192 + 64)])
def test_hif4_shapes(lib, shape):
    x = _grouped(*shape, seed=sum(shape))
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT)
    rs, _ = lib.fp4q_stats()
    ref = o.quantize(_bits(x), FMT)["row"]
    check_hif4(r, ref)
    check_stats(rs, ref["stats"])


def test_hif4_outlier_input(lib):
    x = synth.normal_with_outliers(256, 1024, 1.0, 0.01, 20.0, 9)
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT, rht=True, seed=4)
    ref = o.quantize(_bits(x), FMT, rht=True, seed=4)["row"]
    check_hif4(r, ref)


def test_hif4_worked_examples(lib):
    """The hand-derived examples the oracle is pinned to, through the kernel."""
    path = os.path.join(os.path.dirname(__file__), "golden", "hif4_worked.txt")
    rows, words, codes = [], [], []
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "v":
            v = np.zeros(64, np.float32)
            v[:len(rest)] = [float(t) for t in rest]
            rows.append(v)
        elif key == "word":
            words.append(int(rest[0], 16))
        elif key == "codes":
            c = np.zeros(64, np.uint8)
            c[:len(rest)] = [int(t) for t in rest]
            codes.append(c)
    x = torch.from_numpy(np.stack(rows))
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT)
    assert list(r.scales.cpu().numpy().view(np.uint32)[:, 0]) == words
    assert np.array_equal(o.unpack_nibbles(r.codes.cpu().numpy()), np.stack(codes))


@pytest.mark.parametrize("mag", [1e-30, 1e-9, 1e30])
def test_hif4_extreme_magnitudes(lib, mag):
    """Scales that underflow to 0, land among the E6M2 subnormals, or saturate."""
    x = (_grouped(64, 256, 3, torch.float32) * mag).float()
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT)
    rs, _ = lib.fp4q_stats()
    ref = o.quantize(x.numpy(), FMT)["row"]
    check_hif4(r, ref)
    check_stats(rs, ref["stats"])


def test_hif4_zero_blocks_and_signed_zeros(lib):
    x = _grouped(32, 384, 21)
    x[3, 64:128] = 0.0
    x[7, :64] = -0.0
    x[9, 4:8] = 0.0
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT)
    ref = o.quantize(_bits(x), FMT)["row"]
    check_hif4(r, ref)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rht", [False, True])
def test_hif4_dequantize(lib, rht, out_dtype):
    x = _grouped(96, 512, 18)
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT, rht=rht, seed=5)
    y = lib.fp4q_dequantize(r, inverse_rht=rht, seed=5, out_dtype=out_dtype)
    ref = o.quantize(_bits(x), FMT, rht=rht, seed=5)["row"]
    want = o.dequantize_hif4(ref["codes"], ref["scales"], rht, 5)
    if out_dtype == torch.float32:
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))
    else:
        assert np.array_equal(synth.bf16_bits(y.cpu()), o.f32_to_bf16_bits_rne(want))


def test_hif4_empty_and_nonfinite(lib):
    r, _ = lib.fp4q_quantize(torch.empty(0, 128, dtype=torch.bfloat16, device="cuda"), fmt=FMT)
    rs, _ = lib.fp4q_stats()
    assert rs["n"] == 0 and r.tensor_scale.item() == 1.0
    x = _grouped(16, 128, 2)
    x[5, 70] = float("nan")
    lib.fp4q_quantize(x.cuda(), fmt=FMT)
    assert lib.fp4q_status() == 4


def test_hif4_rejections(lib):
    x = torch.zeros(64, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_quantize(x, fmt=FMT)
    assert e.value.code == 1                                   # cols % 64
    y = torch.zeros(96, 128, dtype=torch.bfloat16, device="cuda")
    for axis in ("col", "both"):
        with pytest.raises(lib.FP4QError) as e:
            lib.fp4q_quantize(y, fmt=FMT, axis=axis)
        assert e.value.code == 1                               # rows % 64 for the column-wise copy
    with pytest.raises(lib.FP4QError) as e:
        lib.fp4q_quantize(y, fmt=FMT, layout="mma")
    assert e.value.code == 2                                   # linear scale words only


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding", ["rtne", "sr"])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("shape,axis", [((192, 384), "both"), ((256, 320), "col"), ((64, 4160), "both")])
def test_hif4_column_copy_parity(lib, shape, axis, rht, rounding, dtype):
    """The transposed copy (blocks of 64 down the columns) from the 128-row
    tile kernel, with the row-wise copy from the row kernel when both are
    asked: 192 rows end in half a tile, 4160 columns in a partial one."""
    x = _grouped(*shape, seed=29, dtype=dtype)
    r, c = lib.fp4q_quantize(x.cuda(), fmt=FMT, rht=rht, rounding=rounding, seed=77, axis=axis)
    rs, cs = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(_bits(x), FMT, rht=rht, rounding=rounding, seed=77, axis=axis)
    check_hif4(c, ref["col"])
    check_stats(cs, ref["col"]["stats"])
    if axis == "both":
        check_hif4(r, ref["row"])
        check_stats(rs, ref["row"]["stats"])


@pytest.mark.parametrize("mag", [1e-30, 1e30])
def test_hif4_column_copy_extremes(lib, mag):
    x = (_grouped(128, 256, 31, torch.float32) * mag).float()
    _, c = lib.fp4q_quantize(x.cuda(), fmt=FMT, axis="col")
    _, cs = lib.fp4q_stats()
    ref = o.quantize(x.numpy(), FMT, axis="col")["col"]
    check_hif4(c, ref)
    check_stats(cs, ref["stats"])


def test_hif4_gradient_both_copies_full_size(lib):
    """The 4096 x 14336 gradient tensor, HiF4 + RHT + SR, both copies from one
    call; sampled rows of each copy against the oracle."""
    x = synth.gradient("a")
    rows, cols = x.shape
    r, c = lib.fp4q_quantize(x.cuda(), fmt=FMT, rht=True, rounding="sr", seed=1234, axis="both")
    assert lib.fp4q_status() == 0
    rng = np.random.default_rng(3)
    rsel = np.unique(np.concatenate([[0, 1, 63, 64, rows - 1], rng.integers(0, rows, 30)]))
    csel = np.unique(np.concatenate([[0, 1, 127, 128, cols - 1], rng.integers(0, cols, 30)]))
    ref = o.quantize(synth.bf16_bits(x), FMT, rht=True, rounding="sr", seed=1234, axis="both",
                     rows_subset=rsel, cols_subset=csel)
    for got, want, sel in ((r, ref["row"], rsel), (c, ref["col"], csel)):
        idx = torch.from_numpy(sel).cuda()
        assert np.array_equal(got.codes[idx].cpu().numpy(), want["codes"])
        assert np.array_equal(got.scales[idx].cpu().numpy().view(np.uint32), want["scales"])


def test_hif4_noalloc_matches(lib):
    x = _grouped(128, 256, 23).cuda()
    a, _ = lib.fp4q_quantize(x, fmt=FMT, rounding="sr", seed=9)
    b, _ = lib.fp4q_quantize_noalloc(x, fmt=FMT, rounding="sr", seed=9)
    assert lib.fp4q_status_noalloc() == 0
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)


def test_hif4_activation_full_size(lib):
    """The 8192 x 4096 BF16 activation (N(0,1) with 1% x20 outliers) as the
    benchmark quantises it, whole tensor against the oracle."""
    x = synth.activation(8192, 4096)
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=FMT)
    rs, _ = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(synth.bf16_bits(x), FMT)["row"]
    check_hif4(r, ref)
    check_stats(rs, ref["stats"])
