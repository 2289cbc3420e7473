// Block-scaled operands on a BF16 contraction: "Replanteamiento del Sesgo de
// Contraccion en el Preentrenamiento de LLM en FP4", Metodologia §2 and
// Resultados (UFP4, the uniform grid, with the RHT on every training GEMM).
// UFP4 has no tensor-core format, and this build has no native MXFP4 GEMM, so
// each operand is dequantised (our kernel) to the BF16 block values
// level * s_b, which BF16 holds exactly (at most 3 + 4 significant bits, in
// range), and a plain BF16 GEMM with FP32 accumulation (cuBLAS) multiplies
// them, scaled by g_A * g_B read on the device. NVFP4 operands take the same
// path too (for comparison with the native block-scaled GEMM).
#include <cstdint>
#include <unordered_map>

#include <cublas_v2.h>
#include <cuda_runtime.h>

#include "fp4q_internal.h"

namespace fp4q {
namespace {

constexpr size_t kCublasWorkspace = size_t(32) << 20;

// alpha = g_A * g_B (FP32, as the native GEMM's epilogue forms it), the unit
// tensor scale the dequantisations use, and beta = 0.
__global__ void gemm_bf16_scalars(const float* ga, const float* gb, float* out) {
  out[0] = __fmul_rn(*ga, *gb);
  out[1] = 1.f;
  out[2] = 0.f;
}

// One cuBLAS handle per host thread and device (a handle must not be used by
// two threads at once).
cublasHandle_t handle_for_device() {
  thread_local std::unordered_map<int, cublasHandle_t> handles;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  auto it = handles.find(dev);
  if (it != handles.end()) return it->second;
  cublasHandle_t h = nullptr;
  if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return nullptr;
  handles[dev] = h;
  return h;
}

}  // namespace

size_t gemm_bf16_scratch_bytes(int64_t m, int64_t n, int64_t k) {
  return 256 + (size_t)(m + n) * (size_t)k * 2 + kCublasWorkspace;
}

cudaError_t run_gemm_bf16(const GemmArgs& a, void* scratch, cudaStream_t s) {
  uint8_t* base = static_cast<uint8_t*>(scratch);
  float* scal = reinterpret_cast<float*>(base);
  uint8_t* abf = base + 256;
  uint8_t* bbf = abf + (size_t)a.m * (size_t)a.k * 2;
  uint8_t* cws = bbf + (size_t)a.n * (size_t)a.k * 2;
  gemm_bf16_scalars<<<1, 1, 0, s>>>(static_cast<const float*>(a.a.tensor_scale),
                                    static_cast<const float*>(a.b.tensor_scale), scal);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  for (int w = 0; w < 2; ++w) {
    DequantArgs d{};
    d.q = w ? a.b : a.a;
    d.q.tensor_scale = scal + 1;      // level * s_b only: the tensor scales go into alpha
    d.rows = w ? a.n : a.m;
    d.cols = a.k;
    d.fmt = a.fmt;
    d.inverse_rht = 0;
    d.seed = 0;
    d.dst = w ? bbf : abf;
    d.dst_dtype = 0;
    if ((e = run_dequantize(d, s)) != cudaSuccess) return e;
  }
  cublasHandle_t h = handle_for_device();
  if (!h) return cudaErrorUnknown;
  if (cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS ||
      cublasSetPointerMode(h, CUBLAS_POINTER_MODE_DEVICE) != CUBLAS_STATUS_SUCCESS ||
      cublasSetWorkspace(h, cws, kCublasWorkspace) != CUBLAS_STATUS_SUCCESS)
    return cudaErrorUnknown;
  // Row-major Y (M x N) = A (M x K) B^T (N x K)^T is column-major Y^T = B A^T:
  // B read as a K x N column-major matrix (transposed), A as K x M (not).
  const cublasStatus_t st = cublasGemmEx(h, CUBLAS_OP_T, CUBLAS_OP_N, (int)a.n, (int)a.m, (int)a.k, scal,
                                         bbf, CUDA_R_16BF, (int)a.k, abf, CUDA_R_16BF, (int)a.k, scal + 2, a.y,
                                         a.out_dtype ? CUDA_R_32F : CUDA_R_16BF, (int)a.n, CUBLAS_COMPUTE_32F,
                                         CUBLAS_GEMM_DEFAULT);
  return st == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

}  // namespace fp4q
