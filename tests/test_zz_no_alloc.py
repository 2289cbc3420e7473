"""fp4q_quantize_noalloc: the quantise entry point for callers that cannot
allocate device memory (fixed memory pools, latency-critical code that must
avoid cudaMalloc's device-wide synchronisation). Its scratch is an array inside
the library; its output must equal fp4q_quantize's, byte for byte, on every
call, including consecutive calls that reuse that array.

This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

CASES = [
    # (format, rht, rounding, axis, layout, shape, data seed, quantisation seed)
    ("nvfp4", True, "rtne", "both", "linear", (192, 320), 41, 1234),
    ("ufp4", True, "sr", "row", "mma", (160, 272), 42, 77),
    ("mxfp4", False, "rtne", "col", "linear", (224, 96), 43, 5),
]


def _raw_noalloc(fq, x, fmt, rht, rounding, seed, axis, layout):
    """Call the C entry point directly with preallocated outputs."""
    rows, cols = x.shape
    ax = fq.AXES[axis]
    r = fq.alloc_copy(rows, cols, fmt, layout, x.device) if ax & 1 else None
    c = fq.alloc_copy(cols, rows, fmt, layout, x.device) if ax & 2 else None
    rs = r.c_struct() if r else None
    cs = c.c_struct() if c else None
    rc = fq.c_call("fp4q_quantize_noalloc", x.data_ptr(), fq.DTYPES[x.dtype], rows, cols,
                   fq.FORMATS[fmt], fq.BLOCKS[fmt], int(rht), fq.ROUNDING[rounding], seed, ax,
                   ctypes.byref(rs) if rs else None, ctypes.byref(cs) if cs else None,
                   torch.cuda.current_stream().cuda_stream)
    assert rc == 0, fq.fp4q_strerror(rc)
    return r, c


def _same(a, b):
    if a is None or b is None:
        assert a is None and b is None
        return
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes)
    assert torch.equal(a.scales, b.scales)
    assert a.tensor_scale.cpu().numpy().view(np.uint32)[0] == \
        b.tensor_scale.cpu().numpy().view(np.uint32)[0]


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(lib):
    for fmt, rht, rnd, axis, layout, shape, dseed, qseed in CASES:
        x = synth.normal_with_outliers(*shape, 1.0, 0.01, 20.0, dseed).cuda()
        want_r, want_c = lib.fp4q_quantize(x, fmt=fmt, rht=rht, rounding=rnd, seed=qseed,
                                           axis=axis, layout=layout)
        for _ in range(2):      # two calls in a row on the shared scratch
            got_r, got_c = _raw_noalloc(lib, x, fmt, rht, rnd, qseed, axis, layout)
            _same(got_r, want_r)
            _same(got_c, want_c)
    assert lib.fp4q_status() == 0
    assert lib.fp4q_status_noalloc() == 0


def test_noalloc_status_reports_nonfinite_input(lib):
    """The status of a no-allocation call is readable without a workspace:
    a NaN in the input is reported once, then cleared."""
    x = synth.normal(64, 256, 1.0, 45)
    x[9, 17] = float("nan")
    lib.fp4q_quantize_noalloc(x.cuda(), fmt="nvfp4", axis="row")
    assert lib.fp4q_status_noalloc() == 4
    assert lib.fp4q_status_noalloc() == 0


def test_noalloc_binding_and_rejections(lib):
    x = synth.normal(128, 256, 1.0, 44).cuda()
    r, _ = lib.fp4q_quantize_noalloc(x, fmt="nvfp4", axis="row")
    want, _ = lib.fp4q_quantize(x, fmt="nvfp4", axis="row")
    _same(r, want)
    out = lib.alloc_copy(128, 256, "nvfp4")
    s = out.c_struct()
    stream = torch.cuda.current_stream().cuda_stream
    # FP4Q_AMAX_READY has no workspace to come from: rejected on the host
    rc = lib.c_call("fp4q_quantize_noalloc", x.data_ptr(), 0, 128, 256, 0, 16, 0, 0, 0, 1 | 4,
                    ctypes.byref(s), None, stream)
    assert rc == 1
    # the usual argument checks apply (cols not a multiple of the block)
    rc = lib.c_call("fp4q_quantize_noalloc", x.data_ptr(), 0, 128, 250, 0, 16, 0, 0, 0, 1,
                    ctypes.byref(s), None, stream)
    assert rc == 1
