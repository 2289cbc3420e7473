"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times: the activation-like 8192 x 4096 BF16 tensor quantised three ways (E2M1,
E2M1 + 16-point RHT, UFP4 + RHT; 16-element blocks, RTNE, row-wise) through
the split amax / quantise calls, against the CPU oracle on the whole tensor:
codes, scales and the tensor scale bit-exact, statistics within tolerance."""
import numpy as np
import pytest

import synth
from oracle import fp4q_oracle as o

from test_gpu_quantize import check_copy, check_stats

pytestmark = pytest.mark.gpu

WAYS = [("nvfp4", False), ("nvfp4", True), ("ufp4", True)]
SEED = 1234


@pytest.fixture(scope="module")
def activation():
    x = synth.activation(8192, 4096)
    return x, synth.bf16_bits(x)


@pytest.mark.parametrize("fmt,rht", WAYS)
def test_activation_three_ways_full_size(lib, activation, fmt, rht):
    x, bits = activation
    xd = x.cuda()
    lib.fp4q_amax(xd, fmt=fmt, rht=rht, seed=SEED, axis="row")
    r, _ = lib.fp4q_quantize(xd, fmt=fmt, rht=rht, seed=SEED, axis="row", amax_ready=True)
    rs, _ = lib.fp4q_stats()
    assert lib.fp4q_status() == 0
    ref = o.quantize(bits, fmt, rht=rht, seed=SEED)["row"]
    check_copy(r, ref, "linear")
    check_stats(rs, ref["stats"])
    if fmt == "ufp4":
        y = lib.fp4q_dequantize(r, inverse_rht=True, seed=SEED)
        want = o.dequantize(ref["codes"], ref["scales"], ref["tensor_scale"], fmt, True, SEED)
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))


def _sample(n, tile, k=40):
    """Indices that include both ends, tile boundaries and a seeded spread."""
    rng = np.random.default_rng(n)
    edge = [0, 1, tile - 1, tile, n - tile - 1, n - tile, n - 2, n - 1]
    return np.unique(np.concatenate([edge, rng.integers(0, n, k)])).astype(np.int64)


@pytest.mark.parametrize("which", ["a", "b"])
def test_gradient_both_copies_full_size(lib, which):
    """The gradient workload as bench.py times it (NVFP4, RHT, Philox SR, row-wise
    and column-wise copies from one call), compared on sampled rows of each
    copy: the tensor amax and scale still come from the whole tensor."""
    import torch
    x = synth.gradient(which)
    rows, cols = x.shape
    r, c = lib.fp4q_quantize(x.cuda(), fmt="nvfp4", rht=True, rounding="sr", seed=SEED, axis="both")
    assert lib.fp4q_status() == 0
    rsel, csel = _sample(rows, 64), _sample(cols, 128)
    ref = o.quantize(synth.bf16_bits(x), "nvfp4", rht=True, rounding="sr", seed=SEED, axis="both",
                     rows_subset=rsel, cols_subset=csel)
    for got, want, sel in ((r, ref["row"], rsel), (c, ref["col"], csel)):
        idx = torch.from_numpy(sel).cuda()
        assert np.array_equal(got.codes[idx].cpu().numpy(), want["codes"])
        assert np.array_equal(got.scales[idx].cpu().numpy(), want["scales"])
        ts = got.tensor_scale.cpu().numpy().view(np.uint32)[0]
        assert ts == np.float32(want["tensor_scale"]).view(np.uint32)


@pytest.fixture(scope="module")
def sweep_largest():
    """The size sweep's largest point: 262144 x 4096 BF16 N(0,1) (2^30 elements)."""
    x = synth.sweep(1 << 18, 4096)
    return x, synth.bf16_bits(x)


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_sweep_largest_size_sampled(lib, sweep_largest, fmt):
    """2^30 elements in the launch configuration bench.py times for the size
    sweep: MXFP4 (32-element E8M0 blocks, one pass) and NVFP4 (16-element E4M3
    blocks, one fp4q_quantize call: amax pass then quantisation pass), RTNE, no
    RHT, row-wise, linear scales. Sampled rows (both ends, chunk boundaries, a
    seeded spread) against the oracle; NVFP4's tensor scale comes from the
    whole tensor on both sides."""
    import torch
    x, bits = sweep_largest
    rows, cols = x.shape
    xd = x.cuda()
    r, _ = lib.fp4q_quantize(xd, fmt=fmt, axis="row")
    assert lib.fp4q_status() == 0
    del xd
    sel = np.unique(np.concatenate([_sample(rows, 2, k=60), [rows // 2 - 1, rows // 2]])).astype(np.int64)
    ref = o.quantize(bits, fmt, rows_subset=sel)["row"]
    idx = torch.from_numpy(sel).cuda()
    assert np.array_equal(r.codes[idx].cpu().numpy(), ref["codes"])
    assert np.array_equal(r.scales[idx].cpu().numpy(), ref["scales"])
    ts = r.tensor_scale.cpu().numpy().view(np.uint32)[0]
    assert ts == np.float32(ref["tensor_scale"]).view(np.uint32)
