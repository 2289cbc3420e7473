// Block-scaled FP4 GEMM (placeholder until the tcgen05 kernel lands).
#include "fp4q_internal.h"
namespace fp4q {
cudaError_t run_gemm(const GemmArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fp4q
