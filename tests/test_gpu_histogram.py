"""GPU code histogram against the oracle's, on copies the GPU quantised (so the
codes match bit for bit first), and the pages' claim that the RHT raises the
effective bucket ratio of both grids on an outlier-heavy tensor ([UFP4]
Resultados)."""
import numpy as np
import pytest
import torch

import synth
from oracle import fp4q_oracle as o

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(512, 1024), (3, 48), (1, 16)])
@pytest.mark.parametrize("fmt,rht", [("nvfp4", False), ("nvfp4", True), ("ufp4", True), ("mxfp4", False)])
def test_histogram_matches_oracle(lib, fmt, rht, shape):
    rows, cols = shape
    if fmt == "mxfp4" and cols % 32:
        pytest.skip("MXFP4 needs 32-element blocks")
    x = synth.activation(rows, cols)
    r, _ = lib.fp4q_quantize(x.cuda(), fmt=fmt, rht=rht, seed=1234)
    h = lib.fp4q_code_histogram(r).cpu().numpy()
    ref = o.quantize(synth.bf16_bits(x), fmt, rht=rht, seed=1234)["row"]
    assert np.array_equal(r.codes.cpu().numpy(), ref["codes"])
    want = o.code_histogram(ref["codes"])
    assert np.array_equal(h, want)
    assert abs(lib.fp4q_effective_bucket_ratio(h) - o.effective_bucket_ratio(want)) < 1e-12


def test_rht_raises_effective_bucket_ratio(lib):
    x = synth.activation(1024, 4096).cuda()
    for fmt in ("nvfp4", "ufp4"):
        ratios = []
        for rht in (False, True):
            r, _ = lib.fp4q_quantize(x, fmt=fmt, rht=rht, seed=1234)
            ratios.append(lib.fp4q_effective_bucket_ratio(lib.fp4q_code_histogram(r)))
        assert ratios[1] > ratios[0] + 0.1, (fmt, ratios)
