// Host-side plumbing shared between the C ABI and the kernel launchers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp4q {

struct QOut {
  uint8_t* codes;
  uint8_t* scales;
  float* tensor_scale;
  int scale_layout;
};

struct QuantArgs {
  const void* src;
  int dtype;          // 0 BF16, 1 FP32
  int64_t rows, cols;
  int fmt;            // 0 NVFP4, 1 MXFP4, 2 UFP4
  int rht, rounding;  // rounding 0 RTNE, 1 SR
  uint64_t seed;
  int axis;           // bit 0 row-wise, bit 1 column-wise
  QOut row, col;
  void* ws;
  int amax_ready;     // 1: the tensor amax already sits in the workspace (skip K1)
};

struct DequantArgs {
  QOut q;
  int64_t rows, cols;
  int fmt;
  int inverse_rht;
  uint64_t seed;
  void* dst;
  int dst_dtype;
};

struct GemmArgs {
  QOut a, b;
  int64_t m, n, k;
  int fmt;
  void* y;
  int out_dtype;      // 0 BF16, 1 FP32
  void* ws;
};

// Number of SMs of the current device (cached per device).
int sm_count();
// Resident CTAs per SM of `kernel` at `threads` threads and `smem` dynamic bytes (cached).
int cached_occupancy(const void* kernel, int threads, int smem);
// A 2-D TMA map (128-byte swizzle, zero fill outside the tensor) over `outer`
// rows of `inner` elements of type `dt`, rows `pitch_bytes` apart, with a box
// of box_inner x box_outer elements. False if the driver's encoder is missing
// or rejects the arguments.
bool encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                     uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer);

cudaError_t run_quantize(const QuantArgs& a, cudaStream_t s);
// K1 alone: the tensor amax of the requested copies, recorded in the workspace.
cudaError_t run_amax(const QuantArgs& a, cudaStream_t s);
// Flat-stream kernels of the row-wise copy (fp4q_rows.cu): the amax pass when
// there is no RHT or only the row-wise copy is wanted, and the quantisation
// pass of a row-wise-only request.
cudaError_t run_amax_rows(const QuantArgs& a, cudaStream_t s);
// grid_out (optional): the number of CTAs launched, i.e. of statistics partials.
cudaError_t run_quant_rows(const QuantArgs& a, cudaStream_t s, int* grid_out = nullptr);
// The column-wise copy of two-level NVFP4 and MBS (rows % 128 == 0): 128-row
// tiles, outer blocks down the columns. row_np: CTAs of the row kernel that
// ran before it for the row-wise copy of the same call (0 if none).
cudaError_t run_quant_cols_outer(const QuantArgs& a, int row_np, cudaStream_t s);
// Requests with the column-wise copy (rows and cols multiples of 16).
cudaError_t run_amax_tiles(const QuantArgs& a, cudaStream_t s);
cudaError_t run_quant_tiles(const QuantArgs& a, cudaStream_t s);
// Both passes of a row-wise NVFP4/UFP4 request in one cooperative launch.
cudaError_t run_quant_fused(const QuantArgs& a, cudaStream_t s);
cudaError_t run_dequantize(const DequantArgs& a, cudaStream_t s);
// Block-scaled operands dequantised in shared memory to exact 16-bit block
// values, multiplied by tcgen05 kind::f16 MMAs with FP32 accumulation, scaled
// by g_A * g_B (UFP4, NVFP4, the E8M0 formats; K % 64 == 0, N % 8 == 0).
cudaError_t run_gemm_dequant(const GemmArgs& a, cudaStream_t s);
// The GEMM on operands with an FP32 scale per 128 elements along K (two-level
// NVFP4, MBS), per-128 scales column-major (K/128 x rows).
cudaError_t run_gemm_outer(const GemmArgs& a, cudaStream_t s);
// Counts of the 16 four-bit codes in `nbytes` bytes of packed codes (zeroes `counts` first).
cudaError_t run_code_histogram(const uint8_t* codes, int64_t nbytes, unsigned long long* counts,
                               cudaStream_t s);
// Returns cudaErrorNotSupported when no GEMM kernel covers the request.
cudaError_t run_gemm(const GemmArgs& a, cudaStream_t s);
// run_gemm with an explicit bound on every wait and, when `skip_first_stage`,
// the producer withholding the first stage of its first tile (so that the
// bounded waits run out): the path that exercises the timeout handling.
cudaError_t run_gemm_ex(const GemmArgs& a, uint64_t timeout_ns, int skip_first_stage, cudaStream_t s);

}  // namespace fp4q
