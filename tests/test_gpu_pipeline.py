"""Back-to-back calls on one stream with no synchronisation in between: each
kernel may start while the previous one finishes (programmatic dependent
launch), so these check that no kernel reads or overwrites what the kernel
before it is still producing. Results are compared with the CPU oracle after
one synchronisation at the end."""
import numpy as np
import pytest
import torch

import synth
from oracle import fp4q_oracle as o

from test_gpu_quantize import check_copy

pytestmark = pytest.mark.gpu

CALLS = [  # fmt, rht, rounding, axis, shape, seed
    ("nvfp4", False, "rtne", "row", (512, 1024), 11),
    ("nvfp4", True, "sr", "both", (384, 640), 12),
    ("ufp4", True, "rtne", "row", (256, 2048), 13),
    ("mxfp4", False, "rtne", "both", (320, 512), 14),
    ("nvfp4", True, "rtne", "col", (448, 256), 15),
    ("ufp4", False, "sr", "both", (192, 768), 16),
]


def test_back_to_back_calls_without_sync(lib):
    dev = torch.device("cuda", 0)
    ws = lib.workspace(dev)
    xs, outs, deqs = [], [], []
    torch.cuda.synchronize()
    for fmt, rht, rnd, axis, (rows, cols), seed in CALLS:
        x = synth.normal_with_outliers(rows, cols, 1.0, 0.01, 20.0, seed)
        xs.append(x)
    xd = [x.to(dev) for x in xs]
    torch.cuda.synchronize()
    for (fmt, rht, rnd, axis, shape, seed), x in zip(CALLS, xd):
        r, c = lib.fp4q_quantize(x, fmt=fmt, rht=rht, rounding=rnd, seed=seed, axis=axis, ws=ws)
        outs.append((r, c))
        # dequantise right behind the quantisation that produced the codes
        q = r if r is not None else c
        deqs.append(lib.fp4q_dequantize(q, inverse_rht=rht, seed=seed, out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert lib.fp4q_status(ws) == 0
    for (fmt, rht, rnd, axis, shape, seed), x, (r, c), y in zip(CALLS, xs, outs, deqs):
        ref = o.quantize(synth.bf16_bits(x), fmt, rht=rht, rounding=rnd, seed=seed, axis=axis)
        if axis in ("row", "both"):
            check_copy(r, ref["row"], "linear")
        if axis in ("col", "both"):
            check_copy(c, ref["col"], "linear")
        refq = ref["row"] if axis in ("row", "both") else ref["col"]
        want = o.dequantize(refq["codes"], refq["scales"], refq["tensor_scale"], fmt, rht, seed)
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))
