// C ABI of libfp4q: argument validation on the host, then dispatch to the
// kernel launchers. Nothing here allocates device memory.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>
#include <cstddef>

#include <cuda_runtime.h>

#include "../../include/fp4q.h"
#include "fp4q_device.cuh"
#include "fp4q_internal.h"

namespace fp4q {

int sm_count() {
  static std::mutex mu;
  static std::unordered_map<int, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  cache[dev] = n;
  return n;
}

int cached_occupancy(const void* kernel, int threads, int smem) {
  static std::mutex mu;
  struct Key {
    const void* k; int dev, t, s;
    bool operator==(const Key& o) const { return k == o.k && dev == o.dev && t == o.t && s == o.s; }
  };
  struct Hash {
    size_t operator()(const Key& x) const {
      return std::hash<const void*>()(x.k) ^ ((size_t)x.dev << 48) ^ ((size_t)x.t << 20) ^ (size_t)x.s;
    }
  };
  static std::unordered_map<Key, int, Hash> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const Key key{kernel, dev, threads, smem};
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    occ = 1;
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = occ;
  return occ;
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    } else {
      cudaGetLastError();
    }
  });
  return fn;
}
}  // namespace

bool encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                     uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fp4q

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int block_for(int fmt) { return fmt == FP4Q_MXFP4 ? 32 : (fmt == FP4Q_HIF4 ? 64 : 16); }

int check_format(int fmt, int block) {
  if (fmt < FP4Q_NVFP4 || fmt > FP4Q_HIF4) return FP4Q_EINVAL;
  if (block != block_for(fmt)) return FP4Q_ENOTSUP;
  return FP4Q_OK;
}

// formats with one FP32 scale per 128 elements of a row in place of the tensor scale
bool outer_scaled(int fmt) { return fmt == FP4Q_NVFP4_2L || fmt == FP4Q_MXFP4_MBS; }
// formats with a per-tensor FP32 scale, set by an amax pass
bool tensor_scaled(int fmt) { return fmt == FP4Q_NVFP4 || fmt == FP4Q_UFP4; }

int check_qtensor(const fp4q_qtensor* q, bool empty = false) {
  if (!q || !q->tensor_scale) return FP4Q_EINVAL;
  if (empty) return aligned(q->tensor_scale, 4) ? FP4Q_OK : FP4Q_EINVAL;
  if (!q->codes || !q->scales) return FP4Q_EINVAL;
  if (q->scale_layout != FP4Q_SCALES_LINEAR && q->scale_layout != FP4Q_SCALES_MMA) return FP4Q_EINVAL;
  if (!aligned(q->codes, 16) || !aligned(q->tensor_scale, 4)) return FP4Q_EINVAL;
  if (q->scale_layout == FP4Q_SCALES_MMA && !aligned(q->scales, 16)) return FP4Q_EINVAL;
  return FP4Q_OK;
}

fp4q::QOut to_qout(const fp4q_qtensor* q) {
  fp4q::QOut o{};
  if (q) {
    o.codes = q->codes;
    o.scales = q->scales;
    o.tensor_scale = q->tensor_scale;
    o.scale_layout = q->scale_layout;
  }
  return o;
}

bool needs_padding(int64_t rows, int64_t nkb) { return (rows % 128) != 0 || (nkb % 4) != 0; }

// Checks shared by fp4q_quantize and fp4q_amax (axis without the flag bits).
int check_source(const void* src, int dtype, int64_t rows, int64_t cols, int fmt, int block,
                 int rht, int axis, const void* workspace, size_t ws_bytes) {
  int rc = check_format(fmt, block);
  if (rc) return rc;
  if (dtype != FP4Q_BF16 && dtype != FP4Q_F32) return FP4Q_EINVAL;
  if (rht != 0 && rht != 1) return FP4Q_EINVAL;
  if (axis < 1 || axis > 3) return FP4Q_EINVAL;
  if (rows < 0 || cols < 0) return FP4Q_EINVAL;
  if (rows > (int64_t(1) << 40) || cols > (int64_t(1) << 40) || (rows && cols > (int64_t(1) << 46) / rows))
    return FP4Q_EINVAL;
  if (!workspace || !aligned(workspace, 16) || ws_bytes < fp4q_workspace_size()) return FP4Q_EINVAL;
  if (rows && cols && (!src || !aligned(src, 16))) return FP4Q_EINVAL;
  if (cols % 16) return FP4Q_EINVAL;     // source rows start on 32-byte boundaries
  if ((axis & FP4Q_ROWWISE) && cols % block) return FP4Q_EINVAL;
  if ((axis & FP4Q_COLWISE) && rows % block) return FP4Q_EINVAL;
  if (outer_scaled(fmt)) {
    if ((axis & FP4Q_ROWWISE) && cols % 128) return FP4Q_EINVAL;   // whole outer blocks per row
    if ((axis & FP4Q_COLWISE) && rows % 128) return FP4Q_EINVAL;   // ... and per column
  }
  return FP4Q_OK;
}

// HiF4 copies: linear scale words (one uint32 per 64-element block), 4-byte aligned.
int check_hif4_qtensor(const fp4q_qtensor* q, bool empty) {
  if (q->scale_layout != FP4Q_SCALES_LINEAR) return FP4Q_ENOTSUP;
  if (!empty && !aligned(q->scales, 4)) return FP4Q_EINVAL;
  return FP4Q_OK;
}

}  // namespace

extern "C" {

size_t fp4q_workspace_size(void) { return (sizeof(fp4q::Workspace) + 255) / 256 * 256; }

int fp4q_workspace_init(void* workspace, void* stream) {
  if (!workspace || !aligned(workspace, 16)) return FP4Q_EINVAL;
  if (cudaMemsetAsync(workspace, 0, fp4q_workspace_size(), (cudaStream_t)stream) != cudaSuccess)
    return FP4Q_ECUDA;
  return FP4Q_OK;
}

size_t fp4q_scales_bytes(int64_t rows, int64_t cols, int block, int scale_layout) {
  if (rows < 0 || cols < 0 || block <= 0) return 0;
  const int64_t nkb = cols / block;
  if (block == 64) {                         // HiF4: a 32-bit word per block, linear only
    return scale_layout == FP4Q_SCALES_LINEAR ? (size_t)rows * (size_t)nkb * 4 : 0;
  }
  if (scale_layout == FP4Q_SCALES_MMA) {     // one scale per 16 elements along the row
    return (size_t)(((rows + 127) / 128) * 128) * (size_t)(((cols / 16 + 3) / 4) * 4);
  }
  return (size_t)rows * (size_t)nkb;
}

int fp4q_amax(const void* src, int dtype, int64_t rows, int64_t cols, int fmt, int block, int rht,
              uint64_t seed, int axis, void* workspace, size_t ws_bytes, void* stream) {
  const int rc = check_source(src, dtype, rows, cols, fmt, block, rht, axis, workspace, ws_bytes);
  if (rc) return rc;
  // power-of-two block scales (the MXFP4 formats) or per-128-element scales
  // (two-level NVFP4, MBS): no tensor amax
  if (!tensor_scaled(fmt)) return FP4Q_OK;
  fp4q::QuantArgs a{};
  a.src = src;
  a.dtype = dtype;
  a.rows = rows;
  a.cols = cols;
  a.fmt = fmt;
  a.rht = rht;
  a.seed = seed;
  a.axis = axis;
  a.ws = workspace;
  return fp4q::run_amax(a, (cudaStream_t)stream) == cudaSuccess ? FP4Q_OK : FP4Q_ECUDA;
}

int fp4q_quantize(const void* src, int dtype, int64_t rows, int64_t cols, int fmt, int block,
                  int rht, int rounding, uint64_t seed, int axis, const fp4q_qtensor* row_out,
                  const fp4q_qtensor* col_out, void* workspace, size_t ws_bytes, void* stream) {
  if (axis & ~(FP4Q_ROWWISE | FP4Q_COLWISE | FP4Q_AMAX_READY)) return FP4Q_EINVAL;
  const int amax_ready = (axis & FP4Q_AMAX_READY) ? 1 : 0;
  axis &= FP4Q_ROWWISE | FP4Q_COLWISE;
  int rc = check_source(src, dtype, rows, cols, fmt, block, rht, axis, workspace, ws_bytes);
  if (rc) return rc;
  if (rounding != FP4Q_RTNE && rounding != FP4Q_SR) return FP4Q_EINVAL;
  const bool empty = rows == 0 || cols == 0;
  if ((axis & FP4Q_ROWWISE) && (rc = check_qtensor(row_out, empty))) return rc;
  if ((axis & FP4Q_COLWISE) && (rc = check_qtensor(col_out, empty))) return rc;
  if (fmt == FP4Q_HIF4 && (axis & FP4Q_ROWWISE) && (rc = check_hif4_qtensor(row_out, empty))) return rc;
  if (fmt == FP4Q_HIF4 && (axis & FP4Q_COLWISE) && (rc = check_hif4_qtensor(col_out, empty))) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  // padding bytes of the tiled scale layout are defined as 0
  if (!empty && (axis & FP4Q_ROWWISE) && row_out->scale_layout == FP4Q_SCALES_MMA && needs_padding(rows, cols / 16)) {
    if (cudaMemsetAsync(row_out->scales, 0, fp4q_scales_bytes(rows, cols, block, FP4Q_SCALES_MMA), s) != cudaSuccess)
      return FP4Q_ECUDA;
  }
  if (!empty && (axis & FP4Q_COLWISE) && col_out->scale_layout == FP4Q_SCALES_MMA && needs_padding(cols, rows / 16)) {
    if (cudaMemsetAsync(col_out->scales, 0, fp4q_scales_bytes(cols, rows, block, FP4Q_SCALES_MMA), s) != cudaSuccess)
      return FP4Q_ECUDA;
  }
  fp4q::QuantArgs a{};
  a.src = src;
  a.dtype = dtype;
  a.rows = rows;
  a.cols = cols;
  a.fmt = fmt;
  a.rht = rht;
  a.rounding = rounding;
  a.seed = seed;
  a.axis = axis;
  a.row = to_qout((axis & FP4Q_ROWWISE) ? row_out : nullptr);
  a.col = to_qout((axis & FP4Q_COLWISE) ? col_out : nullptr);
  a.ws = workspace;
  a.amax_ready = amax_ready;
  return fp4q::run_quantize(a, s) == cudaSuccess ? FP4Q_OK : FP4Q_ECUDA;
}

int fp4q_dequantize(const fp4q_qtensor* q, int64_t rows, int64_t cols, int fmt, int block,
                    int inverse_rht, uint64_t seed, void* dst, int dst_dtype, void* stream) {
  int rc = check_format(fmt, block);
  if (rc) return rc;
  if ((rc = check_qtensor(q))) return rc;
  if (inverse_rht != 0 && inverse_rht != 1) return FP4Q_EINVAL;
  if (dst_dtype != FP4Q_BF16 && dst_dtype != FP4Q_F32) return FP4Q_EINVAL;
  if (rows < 0 || cols < 0 || cols % block) return FP4Q_EINVAL;
  if (outer_scaled(fmt) && cols % 128) return FP4Q_EINVAL;
  if (fmt == FP4Q_HIF4 && (rc = check_hif4_qtensor(q, false))) return rc;
  if (rows == 0 || cols == 0) return FP4Q_OK;
  if (!dst || !aligned(dst, 16)) return FP4Q_EINVAL;
  fp4q::DequantArgs a{};
  a.q = to_qout(q);
  a.rows = rows;
  a.cols = cols;
  a.fmt = fmt;
  a.inverse_rht = inverse_rht;
  a.seed = seed;
  a.dst = dst;
  a.dst_dtype = dst_dtype;
  return fp4q::run_dequantize(a, (cudaStream_t)stream) == cudaSuccess ? FP4Q_OK : FP4Q_ECUDA;
}

int fp4q_gemm_dequant(const fp4q_qtensor* A, const fp4q_qtensor* B, int64_t M, int64_t N, int64_t K,
                      int fmt, void* Y, int out_dtype, void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_format(fmt, block_for(fmt));
  if (rc) return rc;
  // per-128-element scales: not one 16-bit value per element
  if (outer_scaled(fmt)) return FP4Q_ENOTSUP;
  if ((rc = check_qtensor(A)) || (rc = check_qtensor(B))) return rc;
  if (!aligned(A->scales, 2) || !aligned(B->scales, 2)) return FP4Q_EINVAL;
  if (fmt == FP4Q_HIF4 && ((rc = check_hif4_qtensor(A, false)) || (rc = check_hif4_qtensor(B, false)))) return rc;
  if (out_dtype != FP4Q_BF16 && out_dtype != FP4Q_F32) return FP4Q_EINVAL;
  if (M <= 0 || N <= 0 || K <= 0 || K % 64 || N % 8) return FP4Q_EINVAL;
  if (M > (int64_t(1) << 24) || N > (int64_t(1) << 24) || K > (int64_t(1) << 24)) return FP4Q_EINVAL;
  if (!Y || !aligned(Y, 16)) return FP4Q_EINVAL;
  if (!workspace || !aligned(workspace, 16) || ws_bytes < fp4q_workspace_size()) return FP4Q_EINVAL;
  fp4q::GemmArgs a{};
  a.a = to_qout(A);
  a.b = to_qout(B);
  a.m = M;
  a.n = N;
  a.k = K;
  a.fmt = fmt;
  a.y = Y;
  a.out_dtype = out_dtype;
  a.ws = workspace;
  const cudaError_t e = fp4q::run_gemm_dequant(a, (cudaStream_t)stream);
  if (e == cudaErrorNotSupported) return FP4Q_ENOTSUP;
  return e == cudaSuccess ? FP4Q_OK : FP4Q_ECUDA;
}

int fp4q_code_histogram(const fp4q_qtensor* q, int64_t rows, int64_t cols, unsigned long long* counts,
                        void* stream) {
  if (!q || !counts || !aligned(counts, 8)) return FP4Q_EINVAL;
  if (rows < 0 || cols < 0 || (cols & 1)) return FP4Q_EINVAL;
  if (rows && cols > (int64_t(1) << 46) / rows) return FP4Q_EINVAL;
  const int64_t nbytes = rows * (cols / 2);
  if (nbytes && (!q->codes || !aligned(q->codes, 16))) return FP4Q_EINVAL;
  return fp4q::run_code_histogram(q->codes, nbytes, counts, (cudaStream_t)stream) == cudaSuccess ? FP4Q_OK
                                                                                                  : FP4Q_ECUDA;
}

double fp4q_effective_bucket_ratio(const unsigned long long* counts) {
  if (!counts) return 0.0;
  double m[8], tot = 0.0;
  for (int l = 0; l < 8; ++l) {
    m[l] = (double)counts[l] + (double)counts[l + 8];
    tot += m[l];
  }
  if (tot == 0.0) return 0.0;
  double h = 0.0;
  for (int l = 0; l < 8; ++l) {
    if (m[l] > 0.0) {
      const double p = m[l] / tot;
      h -= p * std::log(p);
    }
  }
  return std::exp(h) / 8.0;
}

int fp4q_stats(const void* workspace, fp4q_stats_t* row_stats, fp4q_stats_t* col_stats,
               void* stream) {
  if (!workspace) return FP4Q_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  const fp4q::Workspace* ws = static_cast<const fp4q::Workspace*>(workspace);
  // the header fields, then the per-CTA partials of each copy, summed here in FP64
  constexpr size_t kHead = offsetof(fp4q::Workspace, amax_part);
  unsigned char head[kHead];
  if (cudaMemcpyAsync(head, ws, kHead, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FP4Q_ECUDA;
  struct {
    unsigned int stat_nparts, copies;
    float tensor_scale[2], qmax;
    double n;
  } h;
  std::memcpy(&h.stat_nparts, head + offsetof(fp4q::Workspace, stat_nparts), sizeof(unsigned int));
  std::memcpy(&h.copies, head + offsetof(fp4q::Workspace, copies), sizeof(unsigned int));
  std::memcpy(h.tensor_scale, head + offsetof(fp4q::Workspace, tensor_scale), 2 * sizeof(float));
  std::memcpy(&h.qmax, head + offsetof(fp4q::Workspace, qmax), sizeof(float));
  std::memcpy(&h.n, head + offsetof(fp4q::Workspace, n), sizeof(double));
  const unsigned int np = h.stat_nparts < (unsigned)fp4q::kMaxCtas ? h.stat_nparts : (unsigned)fp4q::kMaxCtas;
  std::vector<double> part((size_t)np * 3);
  fp4q_stats_t* out[2] = {row_stats, col_stats};
  for (int c = 0; c < 2; ++c) {
    if (!out[c]) continue;
    fp4q_stats_t st{};
    if (h.copies & (1u << c)) {
      double sum[3] = {0.0, 0.0, 0.0};
      if (np) {
        for (int k = 0; k < 3; ++k) {
          if (cudaMemcpyAsync(part.data() + (size_t)k * np, &ws->stat_part[c][k][0], np * sizeof(double),
                              cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return FP4Q_ECUDA;
        }
        if (cudaStreamSynchronize(s) != cudaSuccess) return FP4Q_ECUDA;
        for (int k = 0; k < 3; ++k)
          for (unsigned int i = 0; i < np; ++i) sum[k] += part[(size_t)k * np + i];
      }
      const double g = (double)h.tensor_scale[c];
      st.sum_bias = sum[0];
      st.sum_sig2 = sum[1] * g * g;
      st.sum_err2 = sum[2] * g * g;
      st.n = (int64_t)h.n;
      const double qmax = (double)h.qmax;
      st.shrink_bias = st.n ? st.sum_bias / (qmax * (double)st.n) : 0.0;
      if (st.sum_err2 == 0.0) st.snr_db = INFINITY;
      else if (st.sum_sig2 == 0.0) st.snr_db = -INFINITY;
      else st.snr_db = 10.0 * std::log10(st.sum_sig2 / st.sum_err2);
    }
    *out[c] = st;
  }
  return FP4Q_OK;
}

int fp4q_status(void* workspace, void* stream) {
  if (!workspace) return FP4Q_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  fp4q::Workspace* ws = static_cast<fp4q::Workspace*>(workspace);
  unsigned int st = 0;
  if (cudaMemcpyAsync(&st, &ws->status, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(&ws->status, 0, sizeof(st), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FP4Q_ECUDA;
  if (st & fp4q::kStatusTimeout) return FP4Q_ETIMEOUT;
  if (st & fp4q::kStatusNonfinite) return FP4Q_ENONFINITE;
  return FP4Q_OK;
}

namespace {

int gemm_common(const fp4q_qtensor* A, const fp4q_qtensor* B, int64_t M, int64_t N, int64_t K, int fmt,
                void* Y, int out_dtype, void* workspace, size_t ws_bytes, uint64_t timeout_ns, int skip,
                void* stream) {
  if (fmt < FP4Q_NVFP4 || fmt > FP4Q_HIF4) return FP4Q_EINVAL;
  // UFP4 and HiF4 have no FP4 tensor-core type: their block values go through the 16-bit MMA
  if (fmt == FP4Q_UFP4 || fmt == FP4Q_HIF4) {
    if (skip) return FP4Q_ENOTSUP;
    return fp4q_gemm_dequant(A, B, M, N, K, fmt, Y, out_dtype, workspace, ws_bytes, stream);
  }
  // per-128 scales: their own kernel, without the bounded-wait self-test
  if (outer_scaled(fmt) && skip) return FP4Q_ENOTSUP;
  int rc;
  if ((rc = check_qtensor(A)) || (rc = check_qtensor(B))) return rc;
  if (A->scale_layout != FP4Q_SCALES_MMA || B->scale_layout != FP4Q_SCALES_MMA) return FP4Q_EINVAL;
  if (out_dtype != FP4Q_BF16 && out_dtype != FP4Q_F32) return FP4Q_EINVAL;
  if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % 256) return FP4Q_EINVAL;
  if (M > (int64_t(1) << 20) || N > (int64_t(1) << 20) || K > (int64_t(1) << 20)) return FP4Q_EINVAL;
  if (!Y || !aligned(Y, 16)) return FP4Q_EINVAL;
  if (!workspace || !aligned(workspace, 16) || ws_bytes < fp4q_workspace_size()) return FP4Q_EINVAL;
  if (outer_scaled(fmt) && (!aligned(A->tensor_scale, 16) || !aligned(B->tensor_scale, 16))) return FP4Q_EINVAL;
  fp4q::GemmArgs a{};
  a.a = to_qout(A);
  a.b = to_qout(B);
  a.m = M;
  a.n = N;
  a.k = K;
  a.fmt = fmt;
  a.y = Y;
  a.out_dtype = out_dtype;
  a.ws = workspace;
  if (outer_scaled(fmt)) {
    const cudaError_t e = fp4q::run_gemm_outer(a, (cudaStream_t)stream);
    return e == cudaSuccess ? FP4Q_OK : FP4Q_ECUDA;
  }
  const cudaError_t e = timeout_ns ? fp4q::run_gemm_ex(a, timeout_ns, skip, (cudaStream_t)stream)
                                   : fp4q::run_gemm(a, (cudaStream_t)stream);
  if (e == cudaErrorNotSupported) return FP4Q_ENOTSUP;
  return e == cudaSuccess ? FP4Q_OK : FP4Q_ECUDA;
}

}  // namespace

int fp4q_gemm(const fp4q_qtensor* A, const fp4q_qtensor* B, int64_t M, int64_t N, int64_t K,
              int fmt, void* Y, int out_dtype, void* workspace, size_t ws_bytes, void* stream) {
  return gemm_common(A, B, M, N, K, fmt, Y, out_dtype, workspace, ws_bytes, 0, 0, stream);
}

int fp4q_gemm_selftest_timeout(const fp4q_qtensor* A, const fp4q_qtensor* B, int64_t M, int64_t N,
                               int64_t K, int fmt, void* Y, int out_dtype, void* workspace,
                               size_t ws_bytes, uint64_t timeout_ns, void* stream) {
  if (timeout_ns < 1000000ull || timeout_ns > 10000000000ull) return FP4Q_EINVAL;
  return gemm_common(A, B, M, N, K, fmt, Y, out_dtype, workspace, ws_bytes, timeout_ns, 1, stream);
}

const char* fp4q_strerror(int code) {
  switch (code) {
    case FP4Q_OK: return "ok";
    case FP4Q_EINVAL: return "invalid argument";
    case FP4Q_ENOTSUP: return "not supported";
    case FP4Q_ECUDA: return "CUDA error";
    case FP4Q_ENONFINITE: return "non-finite input";
    case FP4Q_ETIMEOUT: return "bounded wait timed out";
    default: return "unknown error";
  }
}

int fp4q_version(void) { return 100; }

}  // extern "C"
