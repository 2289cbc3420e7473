// Dispatch of the block-scaled 4-bit quantisation (sm_103a): which kernels one
// fp4q_amax / fp4q_quantize call launches.
//
// Method: "Replanteamiento del Sesgo de Contraccion en el Preentrenamiento de
// LLM en FP4" (Metodologia §1-2: E2M1 / uniform E1M2 grids, RTNE, stochastic
// rounding, RHT; Eficiencia: RHT fused into the quantisation pass);
// "TetraJet-v2 ..." (Riepilogo Tecnico §2A: NVFP4 16-element groups with an
// 8-bit scale under a per-tensor scale, the transposed copy, SR); "Unveiling
// the Potential of Quantization with MXFP4 ..." (Resume technique §2: MXFP4
// 32-element E8M0 blocks, NVFP4 16-element E4M3 blocks).
//
// Paths (all kernels in fp4q_rows.cu):
//  * row-wise copy only: the tensor is a flat stream of 8192-element chunks
//    (amax_rows_kernel, quant_rows_kernel), or one cooperative launch of both
//    passes for NVFP4 / UFP4 tensors below 2^20 elements (quant_fused_kernel);
//  * any request with the column-wise copy: 64 x 128 tiles through a shared-
//    memory ring, one read of the source serving both copies
//    (amax_tiles_kernel when the RHT makes the two copies' amax differ,
//    quant_tiles_kernel).
// The E8M0 formats (MXFP4 on 32- or 16-element blocks, its overflow-aware
// variant, MBS with its 128-element macro scale), two-level NVFP4 (a scale
// per 128-element outer block) and HiF4 (a scale per 64-element block) have no
// tensor scale, so they skip the amax pass (HiF4: "Unleashing Low-Bit
// Inference on Ascend NPUs ...", Resumen tecnico §2).
#include <cstdint>

#include <cuda_runtime.h>

#include "fp4q_device.cuh"
#include "fp4q_internal.h"

namespace fp4q {

namespace {

// Empty input: write the tensor scales and empty statistics, nothing else.
__global__ void quantize_empty_kernel(int fmt, int axis, float* ts_row, float* ts_col, Workspace* ws) {
  const float g = (fmt == 0 || fmt == 2) ? 0.f : 1.f;       // 1.0 for the E8M0 formats
  if (fmt == 3 || fmt == 6) ts_row = ts_col = nullptr;     // per-128-element scales: the array is empty
  ws->stat_nparts = 0u;
  ws->copies = (unsigned)axis;
  ws->tensor_scale[0] = g;
  ws->tensor_scale[1] = g;
  ws->qmax = (fmt == 2 || fmt == 7) ? 7.f : 6.f;
  ws->n = 0.0;
  if ((axis & 1) && ts_row) *ts_row = g;
  if ((axis & 2) && ts_col) *ts_col = g;
}

// Empty input: a zero amax for both copies.
__global__ void amax_empty_kernel(Workspace* ws) {
  ws->amax_part[0][0] = 0u;
  ws->amax_part[1][0] = 0u;
  ws->amax_nparts = 1u;
}

}  // namespace

cudaError_t run_amax(const QuantArgs& a, cudaStream_t s) {
  Workspace* ws = static_cast<Workspace*>(a.ws);
  if (a.rows == 0 || a.cols == 0) {
    amax_empty_kernel<<<1, 1, 0, s>>>(ws);
    return cudaGetLastError();
  }
  // without the RHT both copies hold the same values, so one flat pass serves both
  if (!a.rht || a.axis == 1) return run_amax_rows(a, s);
  return run_amax_tiles(a, s);
}

cudaError_t run_quantize(const QuantArgs& a, cudaStream_t s) {
  if (a.rows == 0 || a.cols == 0) {
    quantize_empty_kernel<<<1, 1, 0, s>>>(a.fmt, a.axis, a.row.tensor_scale, a.col.tensor_scale,
                                          static_cast<Workspace*>(a.ws));
    return cudaGetLastError();
  }
  // Both passes in one launch pays only for small tensors: measured on B300
  // (one call, median, L2 flushed / not flushed), 256 x 4096: 15.6 / 16.0 us
  // one launch against 12.4 / 18.0 us two; from 1024 x 4096 up the two
  // launches win both ways (22.2 / 18.6 against 16.4 / 18.0 us; 4096 x 4096:
  // 33.9 / 28.6 against 27.4 / 23.3 us), since the second launch's grid
  // restarts on the chunks the amax pass left in L2 and its warps run ahead of
  // one another, which the one-launch kernel's grid barrier and per-chunk CTA
  // barriers do not allow.
  // the E8M0 formats and two-level NVFP4 have no tensor amax: one pass
  const bool tensor_scaled = a.fmt == 0 || a.fmt == 2;
  if (tensor_scaled && !a.amax_ready && a.axis == 1 && a.rows * a.cols < (int64_t(1) << 20)) {
    // the two-launch path if a co-resident grid cannot be had
    const cudaError_t e = run_quant_fused(a, s);
    if (e == cudaSuccess) return e;
    cudaGetLastError();
  }
  if (tensor_scaled && !a.amax_ready) {
    const cudaError_t e = run_amax(a, s);
    if (e != cudaSuccess) return e;
  }
  if ((a.fmt == 3 || a.fmt == 6 || a.fmt == 7) && (a.axis & 2)) {
    // scales per 128 (or, HiF4, 64) elements: the column-wise copy on 128-row
    // tiles (blocks down the columns), the row-wise copy, if wanted, from the
    // row kernel
    int row_np = 0;
    if (a.axis & 1) {
      const cudaError_t e = run_quant_rows(a, s, &row_np);
      if (e != cudaSuccess) return e;
    }
    return run_quant_cols_outer(a, row_np, s);
  }
  return a.axis == 1 ? run_quant_rows(a, s) : run_quant_tiles(a, s);
}

}  // namespace fp4q
