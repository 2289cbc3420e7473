"""The C ABI library: builds, loads without a GPU, exports every function the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp4q.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp4q_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def so():
    import __graft_entry__
    path = __graft_entry__._load_builder().build()
    return ctypes.CDLL(path)


def test_header_declares_the_api():
    names = _declared()
    for n in ("fp4q_quantize", "fp4q_dequantize", "fp4q_stats", "fp4q_gemm",
              "fp4q_status", "fp4q_workspace_size", "fp4q_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(so):
    missing = [n for n in _declared() if not hasattr(so, n)]
    assert not missing, missing


def test_python_binding_uses_the_c_names():
    import fp4_block_scaled_05_b300 as fq
    for n in _declared():
        assert callable(getattr(fq, n)), n


def _header_enum(prefix):
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return {k: int(v) for k, v in re.findall(r"\b(" + prefix + r"[A-Z0-9_]+)\s*=\s*(\d+)", text)}


def test_python_tables_match_the_header():
    """The binding's format, rounding, layout and axis numbers are the header's."""
    import fp4_block_scaled_05_b300 as fq
    fmts = _header_enum("FP4Q_")
    names = {"nvfp4": "FP4Q_NVFP4", "mxfp4": "FP4Q_MXFP4", "ufp4": "FP4Q_UFP4", "nvfp4_2l": "FP4Q_NVFP4_2L",
             "mxfp4_b16": "FP4Q_MXFP4_B16", "mxfp4_oas": "FP4Q_MXFP4_OAS", "mxfp4_mbs": "FP4Q_MXFP4_MBS",
             "hif4": "FP4Q_HIF4"}
    assert set(fq.FORMATS) == set(names)
    for py, c in names.items():
        assert fq.FORMATS[py] == fmts[c], py
    assert fq.ROUNDING == {"rtne": fmts["FP4Q_RTNE"], "sr": fmts["FP4Q_SR"]}
    assert fq.LAYOUTS == {"linear": fmts["FP4Q_SCALES_LINEAR"], "mma": fmts["FP4Q_SCALES_MMA"]}
    assert fq.AXES["row"] == fmts["FP4Q_ROWWISE"] and fq.AXES["col"] == fmts["FP4Q_COLWISE"]
    assert fq.BLOCKS["mxfp4"] == 32 and fq.BLOCKS["hif4"] == 64
    assert all(b == 16 for f, b in fq.BLOCKS.items() if f not in ("mxfp4", "hif4"))


def test_host_validation_without_gpu(so):
    so.fp4q_workspace_size.restype = ctypes.c_size_t
    ws_size = so.fp4q_workspace_size()
    assert 1024 <= ws_size <= (1 << 20)
    so.fp4q_strerror.restype = ctypes.c_char_p
    assert so.fp4q_strerror(1) == b"invalid argument"
    assert so.fp4q_version() >= 100
    so.fp4q_scales_bytes.restype = ctypes.c_size_t
    so.fp4q_scales_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    assert so.fp4q_scales_bytes(100, 96, 16, 0) == 600
    assert so.fp4q_scales_bytes(100, 96, 16, 1) == 128 * 8
    # the tiled layout holds one scale per 16 elements: a 32-element block's twice
    assert so.fp4q_scales_bytes(100, 96, 32, 0) == 300
    assert so.fp4q_scales_bytes(100, 96, 32, 1) == 128 * 8
    # HiF4: one 32-bit word per 64-element block, linear layout only
    assert so.fp4q_scales_bytes(100, 128, 64, 0) == 100 * 2 * 4
    assert so.fp4q_scales_bytes(100, 128, 64, 1) == 0
    q = so.fp4q_quantize
    q.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails validation first
    # bad format / block / dtype / axis / workspace size -> EINVAL or ENOTSUP, no launch
    assert q(fake, 0, 16, 16, 8, 16, 0, 0, 0, 1, None, None, fake, ws_size, None) == 1
    assert q(fake, 0, 16, 16, 0, 32, 0, 0, 0, 1, None, None, fake, ws_size, None) == 2
    assert q(fake, 0, 16, 16, 1, 16, 0, 0, 0, 1, None, None, fake, ws_size, None) == 2
    assert q(fake, 5, 16, 16, 0, 16, 0, 0, 0, 1, None, None, fake, ws_size, None) == 1
    assert q(fake, 0, 16, 16, 0, 16, 0, 0, 0, 4, None, None, fake, ws_size, None) == 1
    assert q(fake, 0, 16, 16, 0, 16, 0, 0, 0, 1, None, None, fake, 16, None) == 1
    assert q(fake, 0, 16, 16, 0, 16, 0, 0, 0, 1, None, None, fake, ws_size, None) == 1  # row_out NULL
    assert q(fake, 0, -1, 16, 0, 16, 0, 0, 0, 1, None, None, fake, ws_size, None) == 1
    # column-wise only still needs source rows of a multiple of 16 elements
    assert q(fake, 0, 32, 100, 0, 16, 0, 0, 0, 2, None, None, fake, ws_size, None) == 1
    # two-level NVFP4 (format 3): whole 128-element outer blocks along the
    # block axis: cols % 128 for the row-wise copy, rows % 128 for the column-wise
    assert q(fake, 0, 32, 256, 3, 16, 0, 0, 0, 2, None, None, fake, ws_size, None) == 1
    assert q(fake, 0, 32, 144, 3, 16, 0, 0, 0, 1, None, None, fake, ws_size, None) == 1
    assert q(fake, 0, 32, 256, 3, 32, 0, 0, 0, 1, None, None, fake, ws_size, None) == 2
    # the MXFP4 variants on 16-element blocks (4, 5) and MBS (6): block 16 only;
    # MBS with whole 128-element macro blocks along the block axis; 8 is no format
    for fmt in (4, 5, 6):
        assert q(fake, 0, 32, 256, fmt, 32, 0, 0, 0, 1, None, None, fake, ws_size, None) == 2
    assert q(fake, 0, 32, 256, 6, 16, 0, 0, 0, 2, None, None, fake, ws_size, None) == 1
    assert q(fake, 0, 32, 144, 6, 16, 0, 0, 0, 1, None, None, fake, ws_size, None) == 1
    assert q(fake, 0, 32, 256, 8, 16, 0, 0, 0, 1, None, None, fake, ws_size, None) == 1
    # HiF4 (7): block 64, whole blocks along the block axis, linear 4-byte-aligned
    # scale words
    from fp4_block_scaled_05_b300 import fp4q_qtensor
    assert q(fake, 0, 32, 256, 7, 16, 0, 0, 0, 1, None, None, fake, ws_size, None) == 2
    assert q(fake, 0, 32, 96, 7, 64, 0, 0, 0, 1, None, None, fake, ws_size, None) == 1
    assert q(fake, 0, 96, 256, 7, 64, 0, 0, 0, 2, None, None, fake, ws_size, None) == 1   # rows % 64
    assert q(fake, 0, 64, 256, 7, 64, 0, 0, 0, 3, None, None, fake, ws_size, None) == 1   # outputs NULL
    assert q(fake, 0, 32, 256, 7, 64, 0, 0, 0, 1, None, None, fake, ws_size, None) == 1   # row_out NULL
    mma = fp4q_qtensor(1 << 20, 1 << 20, 1 << 20, 1)
    assert q(fake, 0, 32, 256, 7, 64, 0, 0, 0, 1, ctypes.addressof(mma), None, fake, ws_size, None) == 2
    odd = fp4q_qtensor(1 << 20, (1 << 20) + 2, 1 << 20, 0)
    assert q(fake, 0, 32, 256, 7, 64, 0, 0, 0, 1, ctypes.addressof(odd), None, fake, ws_size, None) == 1


def test_amax_validation_without_gpu(so):
    so.fp4q_workspace_size.restype = ctypes.c_size_t
    ws_size = so.fp4q_workspace_size()
    a = so.fp4q_amax
    a.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_size_t, ctypes.c_void_p]
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails validation first
    assert a(fake, 0, 16, 16, 8, 16, 0, 0, 1, fake, ws_size, None) == 1      # format
    assert a(fake, 0, 16, 16, 0, 32, 0, 0, 1, fake, ws_size, None) == 2      # block
    assert a(fake, 0, 16, 24, 0, 16, 0, 0, 1, fake, ws_size, None) == 1      # cols % 16
    assert a(fake, 0, 24, 16, 0, 16, 0, 0, 2, fake, ws_size, None) == 1      # rows % 16
    assert a(fake, 0, 32, 24, 0, 16, 1, 0, 2, fake, ws_size, None) == 1      # cols % 16, column-wise only
    assert a(fake, 0, 16, 16, 0, 16, 2, 0, 1, fake, ws_size, None) == 1      # rht flag
    assert a(fake, 0, 16, 16, 0, 16, 0, 0, 4, fake, ws_size, None) == 1      # no copy requested
    assert a(fake, 0, 16, 16, 0, 16, 0, 0, 1, fake, 8, None) == 1            # workspace size
    assert a(None, 0, 16, 16, 0, 16, 0, 0, 1, fake, ws_size, None) == 1      # null source
    # MXFP4 and HiF4 have no tensor amax: valid arguments launch nothing and succeed
    assert a(fake, 0, 32, 32, 1, 32, 0, 0, 3, fake, ws_size, None) == 0
    assert a(fake, 0, 32, 64, 7, 64, 0, 0, 1, fake, ws_size, None) == 0
    assert a(fake, 0, 64, 64, 7, 64, 0, 0, 2, fake, ws_size, None) == 0
    assert a(fake, 0, 96, 64, 7, 64, 0, 0, 2, fake, ws_size, None) == 1      # rows % 64, column-wise
    q = so.fp4q_quantize
    q.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    # unknown flag bits and the ready flag without a copy are rejected
    assert q(fake, 0, 16, 16, 0, 16, 0, 0, 0, 9, None, None, fake, ws_size, None) == 1
    assert q(fake, 0, 16, 16, 0, 16, 0, 0, 0, 4, None, None, fake, ws_size, None) == 1


def test_gemm_selftest_validation_without_gpu(so):
    so.fp4q_workspace_size.restype = ctypes.c_size_t
    f = so.fp4q_gemm_selftest_timeout
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                  ctypes.c_uint64, ctypes.c_void_p]
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the calls below fail validation first
    ws = so.fp4q_workspace_size()
    assert f(fake, fake, 128, 128, 256, 0, fake, 0, fake, ws, 100, None) == 1           # bound too short
    assert f(fake, fake, 128, 128, 256, 0, fake, 0, fake, ws, 10**11, None) == 1        # bound too long
    assert f(fake, fake, 128, 128, 256, 2, fake, 0, fake, ws, 10**7, None) == 2         # UFP4 GEMM
    # the per-128-scaled formats have their own kernel, without the bounded-wait self-test
    assert f(fake, fake, 128, 128, 256, 3, fake, 0, fake, ws, 10**7, None) == 2
    assert f(fake, fake, 128, 128, 256, 6, fake, 0, fake, ws, 10**7, None) == 2
    assert f(fake, fake, 128, 128, 256, 7, fake, 0, fake, ws, 10**7, None) == 2         # HiF4: dequantising GEMM
    assert f(fake, fake, 128, 128, 256, 8, fake, 0, fake, ws, 10**7, None) == 1         # no such format


def test_gemm_format_validation_without_gpu(so):
    """fp4q_gemm refuses unknown formats before touching any pointer and checks
    the descriptors of the others (UFP4 included: it runs on the dequantising
    kernel); fp4q_gemm_dequant refuses the per-128-scaled formats first."""
    so.fp4q_workspace_size.restype = ctypes.c_size_t
    g = so.fp4q_gemm
    g.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails validation first
    ws = so.fp4q_workspace_size()
    assert g(fake, fake, 128, 128, 256, -1, fake, 0, fake, ws, None) == 1
    assert g(fake, fake, 128, 128, 256, 8, fake, 0, fake, ws, None) == 1
    for fmt in (0, 1, 2, 3, 4, 5, 6, 7):                                         # null descriptors
        assert g(None, None, 128, 128, 256, fmt, fake, 0, fake, ws, None) == 1
    d = so.fp4q_gemm_dequant
    d.argtypes = g.argtypes
    assert d(fake, fake, 128, 128, 256, 3, fake, 0, fake, ws, None) == 2      # two-level NVFP4
    assert d(fake, fake, 128, 128, 256, 6, fake, 0, fake, ws, None) == 2      # MBS
    assert d(fake, fake, 128, 128, 256, 8, fake, 0, fake, ws, None) == 1
    for fmt in (0, 1, 2, 4, 5, 7):
        assert d(None, None, 128, 128, 256, fmt, fake, 0, fake, ws, None) == 1
    from fp4_block_scaled_05_b300 import fp4q_qtensor
    lin = fp4q_qtensor(1 << 20, 1 << 20, 1 << 20, 0)
    mma = fp4q_qtensor(1 << 20, 1 << 20, 1 << 20, 1)
    odd = fp4q_qtensor(1 << 20, (1 << 20) + 2, 1 << 20, 0)
    pa = ctypes.addressof
    assert d(pa(lin), pa(mma), 128, 128, 256, 7, fake, 0, fake, ws, None) == 2     # tiled HiF4 scales
    assert d(pa(odd), pa(lin), 128, 128, 256, 7, fake, 0, fake, ws, None) == 1     # words not 4-aligned


def test_effective_bucket_ratio_host(so):
    """The host-side ratio of the C library against the oracle's closed forms."""
    import numpy as np
    from oracle import fp4q_oracle as o
    f = so.fp4q_effective_bucket_ratio
    f.argtypes = [ctypes.POINTER(ctypes.c_ulonglong)]
    f.restype = ctypes.c_double
    for h in ([10] * 8 + [0] * 8, [0, 0, 0, 100] + [0] * 12, [5, 0, 3, 7, 1, 0, 0, 2, 4, 0, 6, 0, 0, 1, 0, 3],
              [0] * 16):
        arr = (ctypes.c_ulonglong * 16)(*h)
        assert abs(f(arr) - o.effective_bucket_ratio(np.array(h))) < 1e-15


def test_code_histogram_validation_without_gpu(so):
    f = so.fp4q_code_histogram
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    fake = ctypes.c_void_p(1 << 20)
    assert f(None, 4, 32, fake, None) == 1                 # no descriptor
    assert f(fake, 4, 32, None, None) == 1                 # no counts
    assert f(fake, 4, 31, fake, None) == 1                 # odd cols
    assert f(fake, -1, 32, fake, None) == 1                # negative rows
    assert f(fake, 4, 32, ctypes.c_void_p((1 << 20) + 4), None) == 1   # counts not 8-byte aligned
