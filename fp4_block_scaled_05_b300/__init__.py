"""Python binding of libfp4q (block-scaled 4-bit quantisation and GEMM on B300).

Argument marshalling only: torch supplies device memory and the current CUDA
stream; every step of the computation runs in the library's sm_103a kernels
through its C ABI (include/fp4q.h). There is no CPU path: if the shared library
is missing, importing this package fails.

Function names follow the C ABI: fp4q_amax, fp4q_quantize, fp4q_dequantize, fp4q_stats,
fp4q_status, fp4q_gemm, fp4q_gemm_dequant, fp4q_gemm_selftest_timeout, fp4q_quantize_noalloc, fp4q_status_noalloc, fp4q_workspace_size, fp4q_workspace_init,
fp4q_scales_bytes, fp4q_strerror, fp4q_version.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp4q.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built: run __graft_entry__.build() "
                      "(or python -m fp4_block_scaled_05_b300._build)")

_lib = ctypes.CDLL(LIB_PATH)

FORMATS = {"nvfp4": 0, "mxfp4": 1, "ufp4": 2, "nvfp4_2l": 3, "mxfp4_b16": 4, "mxfp4_oas": 5, "mxfp4_mbs": 6,
           "hif4": 7}
BLOCKS = {"nvfp4": 16, "mxfp4": 32, "ufp4": 16, "nvfp4_2l": 16, "mxfp4_b16": 16, "mxfp4_oas": 16,
          "mxfp4_mbs": 16, "hif4": 64}
OUTER_BLOCK = 128   # two-level NVFP4 and MBS: one FP32 scale per 128 elements of a row
OUTER_SCALED = ("nvfp4_2l", "mxfp4_mbs")
ROUNDING = {"rtne": 0, "sr": 1}
DTYPES = {torch.bfloat16: 0, torch.float32: 1}
AXES = {"row": 1, "col": 2, "both": 3}
LAYOUTS = {"linear": 0, "mma": 1}
ERRORS = {0: "FP4Q_OK", 1: "FP4Q_EINVAL", 2: "FP4Q_ENOTSUP", 3: "FP4Q_ECUDA",
          4: "FP4Q_ENONFINITE", 5: "FP4Q_ETIMEOUT"}


class fp4q_qtensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p), ("scale_layout", ctypes.c_int)]


class fp4q_stats_t(ctypes.Structure):
    _fields_ = [("shrink_bias", ctypes.c_double), ("snr_db", ctypes.c_double),
                ("sum_sig2", ctypes.c_double), ("sum_err2", ctypes.c_double),
                ("sum_bias", ctypes.c_double), ("n", ctypes.c_int64)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_QP = ctypes.POINTER(fp4q_qtensor)
_SP = ctypes.POINTER(fp4q_stats_t)

_SIGS = {
    "fp4q_workspace_size": ([], _SZ),
    "fp4q_workspace_init": ([_P, _P], _I),
    "fp4q_scales_bytes": ([_I64, _I64, _I, _I], _SZ),
    "fp4q_amax": ([_P, _I, _I64, _I64, _I, _I, _I, ctypes.c_uint64, _I, _P, _SZ, _P], _I),
    "fp4q_quantize": ([_P, _I, _I64, _I64, _I, _I, _I, _I, ctypes.c_uint64, _I, _QP, _QP, _P, _SZ, _P], _I),
    "fp4q_quantize_noalloc": ([_P, _I, _I64, _I64, _I, _I, _I, _I, ctypes.c_uint64, _I, _QP, _QP, _P], _I),
    "fp4q_dequantize": ([_QP, _I64, _I64, _I, _I, _I, ctypes.c_uint64, _P, _I, _P], _I),
    "fp4q_stats": ([_P, _SP, _SP, _P], _I),
    "fp4q_status": ([_P, _P], _I),
    "fp4q_status_noalloc": ([_P], _I),
    "fp4q_gemm": ([_QP, _QP, _I64, _I64, _I64, _I, _P, _I, _P, _SZ, _P], _I),
    "fp4q_gemm_selftest_timeout": ([_QP, _QP, _I64, _I64, _I64, _I, _P, _I, _P, _SZ, ctypes.c_uint64, _P], _I),
    "fp4q_code_histogram": ([_QP, _I64, _I64, _P, _P], _I),
    "fp4q_gemm_dequant": ([_QP, _QP, _I64, _I64, _I64, _I, _P, _I, _P, _SZ, _P], _I),
    "fp4q_effective_bucket_ratio": ([ctypes.POINTER(ctypes.c_ulonglong)], ctypes.c_double),
    "fp4q_strerror": ([_I], ctypes.c_char_p),
    "fp4q_version": ([], _I),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res


class FP4QError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {ERRORS.get(code, code)} ({fp4q_strerror(code)})")
        self.code = code


def _check(fn: str, code: int):
    if code != 0:
        raise FP4QError(fn, code)


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


# ---- thin wrappers with the C names ------------------------------------------

def fp4q_workspace_size() -> int:
    return int(_lib.fp4q_workspace_size())


def fp4q_scales_bytes(rows: int, cols: int, block: int, layout: int) -> int:
    return int(_lib.fp4q_scales_bytes(rows, cols, block, layout))


def fp4q_strerror(code: int) -> str:
    return _lib.fp4q_strerror(code).decode()


def fp4q_version() -> int:
    return int(_lib.fp4q_version())


def fp4q_workspace_init(ws: torch.Tensor) -> None:
    _check("fp4q_workspace_init", _lib.fp4q_workspace_init(ws.data_ptr(), _stream(ws.device)))


_WS: dict = {}


def workspace(device=None) -> torch.Tensor:
    """The default per-device workspace (zero-filled once, reused by every call)."""
    dev = torch.device(device if device is not None else "cuda")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    ws = _WS.get(dev)
    if ws is None:
        ws = torch.zeros(fp4q_workspace_size(), dtype=torch.uint8, device=dev)
        _WS[dev] = ws
    return ws


@dataclass
class QCopy:
    """One quantised copy (device buffers) of a rows x cols matrix."""
    codes: torch.Tensor          # uint8 [rows, cols/2]
    scales: torch.Tensor         # uint8 [rows, cols/block] (linear) or flat (mma);
                                 # HiF4: int32 [rows, cols/64], one scale word per block
    tensor_scale: torch.Tensor   # float32 [1]; two-level NVFP4 and MBS: [rows, cols/128] per-128 scales
                                 # ([cols/128, rows] with the tiled "mma" layout)
    fmt: str
    rows: int
    cols: int
    layout: str = "linear"

    @property
    def block(self) -> int:
        return BLOCKS[self.fmt]

    def c_struct(self) -> fp4q_qtensor:
        return fp4q_qtensor(self.codes.data_ptr(), self.scales.data_ptr(),
                            self.tensor_scale.data_ptr(), LAYOUTS[self.layout])


def alloc_copy(rows: int, cols: int, fmt: str, layout: str = "linear", device=None) -> QCopy:
    dev = device if device is not None else "cuda"
    b = BLOCKS[fmt]
    codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev)
    if fmt == "hif4":
        scales = torch.empty(rows, cols // b, dtype=torch.int32, device=dev)
    elif layout == "linear":
        scales = torch.empty(rows, cols // b, dtype=torch.uint8, device=dev)
    else:
        scales = torch.empty(fp4q_scales_bytes(rows, cols, b, 1), dtype=torch.uint8, device=dev)
    if fmt in OUTER_SCALED:
        # the tiled layout keeps the per-128 scales column-major (one K chunk's rows contiguous)
        shape = (cols // OUTER_BLOCK, rows) if layout == "mma" else (rows, cols // OUTER_BLOCK)
        ts = torch.empty(shape, dtype=torch.float32, device=dev)
    else:
        ts = torch.empty(1, dtype=torch.float32, device=dev)
    return QCopy(codes, scales, ts, fmt, rows, cols, layout)


def _check_src(x: torch.Tensor) -> torch.Tensor:
    if x.dim() != 2 or not x.is_cuda or x.dtype not in DTYPES:
        raise ValueError("x must be a 2-D BF16 or FP32 CUDA tensor")
    return x.contiguous()


def fp4q_amax(x: torch.Tensor, fmt: str = "nvfp4", rht: bool = False, seed: int = 0,
              axis: str = "row", ws: torch.Tensor = None) -> None:
    """Record the tensor amax of the requested copies of ``x`` in ``ws`` (the
    first pass of fp4q_quantize); follow with fp4q_quantize(..., amax_ready=True)."""
    x = _check_src(x)
    if ws is None:
        ws = workspace(x.device)
    rows, cols = x.shape
    rc = _lib.fp4q_amax(x.data_ptr(), DTYPES[x.dtype], rows, cols, FORMATS[fmt], BLOCKS[fmt],
                        int(bool(rht)), seed & 0xFFFFFFFFFFFFFFFF, AXES[axis], ws.data_ptr(),
                        ws.numel(), _stream(x.device))
    _check("fp4q_amax", rc)


def fp4q_quantize(x: torch.Tensor, fmt: str = "nvfp4", rht: bool = False, rounding: str = "rtne",
                  seed: int = 0, axis: str = "row", layout: str = "linear", ws: torch.Tensor = None,
                  row_out: QCopy = None, col_out: QCopy = None, amax_ready: bool = False):
    """Quantise a 2-D BF16/FP32 CUDA tensor. Returns (row_copy, col_copy); the
    copy not requested is None. The column-wise copy is the transposed matrix
    (cols x rows). ``amax_ready``: the amax pass already ran (fp4q_amax)."""
    x = _check_src(x)
    rows, cols = x.shape
    ax = AXES[axis]
    if ws is None:
        ws = workspace(x.device)
    if (ax & 1) and row_out is None:
        row_out = alloc_copy(rows, cols, fmt, layout, x.device)
    if (ax & 2) and col_out is None:
        col_out = alloc_copy(cols, rows, fmt, layout, x.device)
    rs = row_out.c_struct() if ax & 1 else None
    cs = col_out.c_struct() if ax & 2 else None
    rc = _lib.fp4q_quantize(x.data_ptr(), DTYPES[x.dtype], rows, cols, FORMATS[fmt], BLOCKS[fmt],
                            int(bool(rht)), ROUNDING[rounding], seed & 0xFFFFFFFFFFFFFFFF,
                            ax | (4 if amax_ready else 0),
                            ctypes.byref(rs) if rs is not None else None,
                            ctypes.byref(cs) if cs is not None else None,
                            ws.data_ptr(), ws.numel(), _stream(x.device))
    _check("fp4q_quantize", rc)
    return (row_out if ax & 1 else None), (col_out if ax & 2 else None)


def fp4q_quantize_noalloc(x: torch.Tensor, fmt: str = "nvfp4", rht: bool = False,
                          rounding: str = "rtne", seed: int = 0, axis: str = "row",
                          row_out: QCopy = None, col_out: QCopy = None, layout: str = "linear"):
    """fp4q_quantize for callers that cannot allocate device memory: the C call
    uses scratch inside the library instead of a workspace (its statistics are
    not readable). Pass preallocated row_out / col_out to allocate nothing here
    either. Calls that overlap on the GPU race on that shared scratch."""
    x = _check_src(x)
    rows, cols = x.shape
    ax = AXES[axis]
    if (ax & 1) and row_out is None:
        row_out = alloc_copy(rows, cols, fmt, layout, x.device)
    if (ax & 2) and col_out is None:
        col_out = alloc_copy(cols, rows, fmt, layout, x.device)
    rs = row_out.c_struct() if ax & 1 else None
    cs = col_out.c_struct() if ax & 2 else None
    rc = _lib.fp4q_quantize_noalloc(x.data_ptr(), DTYPES[x.dtype], rows, cols, FORMATS[fmt],
                                    BLOCKS[fmt], int(bool(rht)), ROUNDING[rounding],
                                    seed & 0xFFFFFFFFFFFFFFFF, ax,
                                    ctypes.byref(rs) if rs is not None else None,
                                    ctypes.byref(cs) if cs is not None else None,
                                    _stream(x.device))
    _check("fp4q_quantize_noalloc", rc)
    return (row_out if ax & 1 else None), (col_out if ax & 2 else None)


def fp4q_dequantize(q: QCopy, inverse_rht: bool = False, seed: int = 0,
                    out_dtype=torch.float32, out: torch.Tensor = None) -> torch.Tensor:
    if out is None:
        out = torch.empty(q.rows, q.cols, dtype=out_dtype, device=q.codes.device)
    s = q.c_struct()
    rc = _lib.fp4q_dequantize(ctypes.byref(s), q.rows, q.cols, FORMATS[q.fmt], q.block,
                              int(bool(inverse_rht)), seed & 0xFFFFFFFFFFFFFFFF, out.data_ptr(),
                              DTYPES[out.dtype], _stream(out.device))
    _check("fp4q_dequantize", rc)
    return out


def fp4q_code_histogram(q: QCopy, out: torch.Tensor = None) -> torch.Tensor:
    """Counts of the 16 codes of a copy (int64 [16], on the copy's device)."""
    if out is None:
        out = torch.empty(16, dtype=torch.int64, device=q.codes.device)
    s = q.c_struct()
    rc = _lib.fp4q_code_histogram(ctypes.byref(s), q.rows, q.cols, ctypes.c_void_p(out.data_ptr()),
                                  _stream(q.codes.device))
    _check("fp4q_code_histogram", rc)
    return out


def fp4q_effective_bucket_ratio(counts) -> float:
    """exp(H)/8 of a 16-code histogram (see fp4q.h)."""
    h = (ctypes.c_ulonglong * 16)(*[int(v) for v in torch.as_tensor(counts).cpu().tolist()])
    return float(_lib.fp4q_effective_bucket_ratio(h))


def _stats_dict(st: fp4q_stats_t) -> dict:
    return {"shrink_bias": st.shrink_bias, "snr_db": st.snr_db, "sum_sig2": st.sum_sig2,
            "sum_err2": st.sum_err2, "sum_bias": st.sum_bias, "n": st.n}


def fp4q_stats(ws: torch.Tensor = None, device=None):
    """(row_stats, col_stats) of the last quantise call on `ws` (synchronises)."""
    if ws is None:
        ws = workspace(device)
    r, c = fp4q_stats_t(), fp4q_stats_t()
    _check("fp4q_stats", _lib.fp4q_stats(ws.data_ptr(), ctypes.byref(r), ctypes.byref(c),
                                         _stream(ws.device)))
    return _stats_dict(r), _stats_dict(c)


def fp4q_status(ws: torch.Tensor = None, device=None) -> int:
    """Device status since the last call (0, 4 = non-finite, 5 = timeout); clears it."""
    if ws is None:
        ws = workspace(device)
    rc = _lib.fp4q_status(ws.data_ptr(), _stream(ws.device))
    if rc not in (0, 4, 5):
        _check("fp4q_status", rc)
    return rc


def fp4q_status_noalloc(device=None) -> int:
    """Device status of the fp4q_quantize_noalloc calls on the current device
    (0, 4 = non-finite, 5 = timeout); clears it."""
    dev = torch.device(device if device is not None else "cuda")
    rc = _lib.fp4q_status_noalloc(_stream(dev))
    if rc not in (0, 4, 5):
        _check("fp4q_status_noalloc", rc)
    return rc


def fp4q_gemm(a: QCopy, b: QCopy, out_dtype=torch.bfloat16, out: torch.Tensor = None,
              ws: torch.Tensor = None) -> torch.Tensor:
    """Y = dequant(a) @ dequant(b)^T for row-wise copies a (M x K), b (N x K)."""
    if a.cols != b.cols:
        raise ValueError("K mismatch")
    if ws is None:
        ws = workspace(a.codes.device)
    if out is None:
        out = torch.empty(a.rows, b.rows, dtype=out_dtype, device=a.codes.device)
    sa, sb = a.c_struct(), b.c_struct()
    rc = _lib.fp4q_gemm(ctypes.byref(sa), ctypes.byref(sb), a.rows, b.rows, a.cols, FORMATS[a.fmt],
                        out.data_ptr(), DTYPES[out.dtype], ws.data_ptr(), ws.numel(),
                        _stream(out.device))
    _check("fp4q_gemm", rc)
    return out


def fp4q_gemm_dequant(a: QCopy, b: QCopy, out_dtype=torch.bfloat16, out: torch.Tensor = None,
                      ws: torch.Tensor = None) -> torch.Tensor:
    """Y = dequant(a) @ dequant(b)^T on the 16-bit tensor-core MMA (UFP4, NVFP4
    or E8M0 row-wise copies a (M x K), b (N x K)); the block values are formed
    in shared memory, never in HBM."""
    if a.cols != b.cols or a.fmt != b.fmt:
        raise ValueError("K or format mismatch")
    dev = a.codes.device
    if ws is None:
        ws = workspace(dev)
    if out is None:
        out = torch.empty(a.rows, b.rows, dtype=out_dtype, device=dev)
    sa, sb = a.c_struct(), b.c_struct()
    rc = _lib.fp4q_gemm_dequant(ctypes.byref(sa), ctypes.byref(sb), a.rows, b.rows, a.cols, FORMATS[a.fmt],
                                out.data_ptr(), DTYPES[out.dtype], ws.data_ptr(), ws.numel(), _stream(dev))
    _check("fp4q_gemm_dequant", rc)
    return out


def fp4q_gemm_selftest_timeout(a: QCopy, b: QCopy, timeout_ns: int, out: torch.Tensor = None,
                               ws: torch.Tensor = None) -> torch.Tensor:
    """Test hook: the GEMM with one stage withheld and every wait bounded by
    ``timeout_ns``; afterwards fp4q_status(ws) reads 5 (FP4Q_ETIMEOUT)."""
    if ws is None:
        ws = workspace(a.codes.device)
    if out is None:
        out = torch.empty(a.rows, b.rows, dtype=torch.bfloat16, device=a.codes.device)
    sa, sb = a.c_struct(), b.c_struct()
    rc = _lib.fp4q_gemm_selftest_timeout(ctypes.byref(sa), ctypes.byref(sb), a.rows, b.rows, a.cols,
                                         FORMATS[a.fmt], out.data_ptr(), DTYPES[out.dtype], ws.data_ptr(),
                                         ws.numel(), int(timeout_ns), _stream(out.device))
    _check("fp4q_gemm_selftest_timeout", rc)
    return out


def c_call(name: str, *args):
    """Direct access to a C entry point (tests of the raw ABI)."""
    return getattr(_lib, name)(*args)
