// fp4q_quantize_noalloc: fp4q_quantize for callers that cannot allocate
// device memory. The scratch the quantisation kernels need (tensor amaxes,
// per-CTA partial sums, completion counters, status word) lives in one
// file-scope device array instead of a caller-provided workspace.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fp4q.h"
#include "fp4q_device.cuh"

namespace {

// Fixed capacity of the library-owned scratch. Every GPU that loads the
// library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(128) << 10;   // 128 KiB
static_assert(sizeof(fp4q::Workspace) <= kNoAllocScratchBytes, "scratch too small");

// Host code must not use this name as a device address: on the host it is a
// stand-in symbol. Its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (the first call on each device does this set-up).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4Q_ECUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FP4Q_ECUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FP4Q_OK;
}

}  // namespace

extern "C" int fp4q_quantize_noalloc(const void* src, int dtype, int64_t rows, int64_t cols,
                                     int fmt, int block, int rht, int rounding, uint64_t seed,
                                     int axis, const fp4q_qtensor* row_out,
                                     const fp4q_qtensor* col_out, void* stream) {
  if (fp4q_workspace_size() > kNoAllocScratchBytes) return FP4Q_EINVAL;
  // the amax of an earlier fp4q_amax call cannot be handed over: no workspace
  if (axis & FP4Q_AMAX_READY) return FP4Q_EINVAL;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc) return rc;
  // the header (status word, partial counts, grid-barrier state) must start
  // at zero; everything else in the scratch is written before it is read
  // within one call
  const size_t head = offsetof(fp4q::Workspace, amax_part);
  if (cudaMemsetAsync(scratch, 0, head, (cudaStream_t)stream) != cudaSuccess) return FP4Q_ECUDA;
  return fp4q_quantize(src, dtype, rows, cols, fmt, block, rht, rounding, seed, axis, row_out,
                       col_out, scratch, kNoAllocScratchBytes, stream);
}

extern "C" int fp4q_status_noalloc(void* stream) {
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc) return rc;
  return fp4q_status(scratch, stream);
}
