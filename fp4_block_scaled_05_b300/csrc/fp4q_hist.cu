// Code utilisation of a quantised copy (sm_103a): how many elements carry each
// of the 16 four-bit codes. "Replanteamiento del Sesgo de Contraccion en el
// Preentrenamiento de LLM en FP4", Resultados: the RHT raises the effective
// bucket ratio of both grids; this histogram is what that ratio is read from.
//
// The copy's code bytes are read once as 16-byte vectors (grid-stride). For
// each 32-bit word (8 codes) the four bit planes of its nibbles are taken
// once; for each code value v, the AND of each plane or its complement (per
// v's bits) leaves one bit per matching nibble, and a popcount gives the count. Per-thread counts are summed by warp shuffles and
// shared memory, then added to the 16 global counters (one atomic each per CTA).
#include <cstdint>

#include <cuda_runtime.h>

#include "fp4q_internal.h"

namespace fp4q {
namespace {

constexpr int HT = 256;

// Bit planes of the 8 nibbles of a word: plane k holds bit k of every nibble
// at the nibble's bit 0.
struct Planes {
  uint32_t b0, b1, b2, b3;
};

__device__ __forceinline__ Planes planes_of(uint32_t w) {
  return Planes{w & 0x11111111u, (w >> 1) & 0x11111111u, (w >> 2) & 0x11111111u, (w >> 3) & 0x11111111u};
}

// Number of nibbles equal to V: each plane or its complement, per V's bits.
template <uint32_t V>
__device__ __forceinline__ uint32_t nibbles_equal(const Planes& p) {
  const uint32_t m = ((V & 1u) ? p.b0 : ~p.b0) & ((V & 2u) ? p.b1 : ~p.b1) & ((V & 4u) ? p.b2 : ~p.b2) &
                     ((V & 8u) ? p.b3 : ~p.b3) & 0x11111111u;
  return __popc(m);
}

template <uint32_t V>
__device__ __forceinline__ void count_all(const Planes& p, uint32_t (&cnt)[16]) {
  cnt[V] += nibbles_equal<V>(p);
  if constexpr (V < 15u) count_all<V + 1u>(p, cnt);
}

__global__ void __launch_bounds__(HT) code_hist_kernel(const uint8_t* __restrict__ codes, int64_t nbytes,
                                                       unsigned long long* __restrict__ out) {
  uint32_t cnt[16];
#pragma unroll
  for (int v = 0; v < 16; ++v) cnt[v] = 0u;
  const int64_t nvec = nbytes / 16;
  const uint4* p = reinterpret_cast<const uint4*>(codes);
  const int64_t stride = (int64_t)gridDim.x * HT;
  for (int64_t i = (int64_t)blockIdx.x * HT + threadIdx.x; i < nvec; i += stride) {
    const uint4 u = __ldg(p + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) count_all<0u>(planes_of(w[k]), cnt);
  }
  // the last nbytes % 16 bytes, one per thread of CTA 0
  const int64_t tail = nbytes - nvec * 16;
  if (blockIdx.x == 0 && (int64_t)threadIdx.x < tail) {
    const uint32_t b = codes[nvec * 16 + threadIdx.x];
#pragma unroll
    for (int v = 0; v < 16; ++v) cnt[v] += ((b & 15u) == (uint32_t)v) + ((b >> 4) == (uint32_t)v);
  }
  __shared__ uint32_t sh[HT / 32][16];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int v = 0; v < 16; ++v) {
    uint32_t c = cnt[v];
#pragma unroll
    for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
    if (lane == 0) sh[warp][v] = c;
  }
  __syncthreads();
  if (threadIdx.x < 16) {
    unsigned long long t = 0ull;
#pragma unroll
    for (int w = 0; w < HT / 32; ++w) t += sh[w][threadIdx.x];
    if (t) atomicAdd(out + threadIdx.x, t);
  }
}

}  // namespace

cudaError_t run_code_histogram(const uint8_t* codes, int64_t nbytes, unsigned long long* counts,
                               cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(counts, 0, 16 * sizeof(unsigned long long), s);
  if (e != cudaSuccess || nbytes == 0) return e;
  const int64_t nvec = nbytes / 16;
  int64_t grid = (nvec + HT - 1) / HT;
  const int64_t gmax = (int64_t)sm_count() * 8;
  if (grid > gmax) grid = gmax;
  if (grid < 1) grid = 1;
  code_hist_kernel<<<(int)grid, HT, 0, s>>>(codes, nbytes, counts);
  return cudaGetLastError();
}

}  // namespace fp4q
