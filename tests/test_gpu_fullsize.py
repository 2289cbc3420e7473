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
