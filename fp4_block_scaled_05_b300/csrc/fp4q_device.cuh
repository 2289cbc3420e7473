// Device helpers for the fp4q kernels (sm_103a).
//
// Exact-path rule: every FP32 operation that decides a code or a scale is an
// explicit round-to-nearest intrinsic (__fadd_rn, __fmul_rn, __fdiv_rn,
// __frcp_rn), the translation units are built with -fmad=false, and no
// flush-to-zero is enabled, so each step is one IEEE operation in a fixed order.
#pragma once

#include <cstdint>
#include <cfloat>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace fp4q {

// ---- workspace shared by every call ------------------------------------------
constexpr int kMaxCtas = 2048;   // upper bound on the persistent grid of a quantise kernel

constexpr uint32_t kStatusNonfinite = 1u;
constexpr uint32_t kStatusTimeout = 2u;

// The passes hand their results on through per-CTA partials, so no kernel
// ends in a serial fold: the amax pass leaves one partial maximum per CTA,
// which every CTA of the quantisation pass folds at its start; the
// quantisation pass leaves one partial per CTA of each statistic, which
// fp4q_stats sums on the host in FP64.
struct Workspace {
  unsigned int status;          // sticky FP4Q status bits, cleared by fp4q_status
  unsigned int amax_nparts;     // CTAs of the last amax pass (entries of amax_part)
  unsigned int stat_nparts;     // CTAs of the last quantisation pass (entries of stat_part)
  unsigned int copies;          // axis bits produced by the last quantisation pass
  float tensor_scale[2];        // g of its row / column copy
  float qmax;                   // its Qmax
  unsigned int gbar_count;      // grid barrier of the one-launch quantiser: arrivals (wraps to 0;
                                // zeroed before each launch)
  double n;                     // its elements per copy
  unsigned int gbar_gen;        // grid barrier: generation, bumped by the last arrival
  unsigned int reserved;
  unsigned int amax_part[2][kMaxCtas];   // per-CTA max |v| (FP32 bits) of the row / column copy
  double stat_part[2][3][kMaxCtas];      // per-CTA sums: bias (grid units); signal, error
                                         // (grid units x s^2; MXFP4: absolute)
};

// ---- Philox4x32-10 (Salmon et al., SC'11) -----------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    if (i) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// The ten round keys of one seed: round i uses (k0 + i * 0x9E3779B9,
// k1 + i * 0xBB67AE85) mod 2^32. Computed once on the host and passed as a
// kernel argument, they sit in the constant bank, so a round costs only its
// two multiplies and two XORs.
struct PhiloxKey {
  uint32_t k0[10], k1[10];
};

inline PhiloxKey philox_key(uint64_t seed) {
  PhiloxKey k;
  uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    k.k0[i] = a;
    k.k1[i] = b;
    a += 0x9E3779B9u;
    b += 0xBB67AE85u;
  }
  return k;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKey& k) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.k0[i], lo1, hi0 ^ c.w ^ k.k1[i], lo0);
  }
  return c;
}

// 16-bit RHT sign mask: bit j set <=> sigma_j = -1.
__device__ __forceinline__ uint32_t rht_sign_mask(uint64_t seed) {
  const uint4 w = philox4x32_10(make_uint4(0u, 0u, 0u, 0xFFFFFFFFu), (uint32_t)seed,
                                (uint32_t)(seed >> 32));
  return w.x & 0xFFFFu;
}

// ---- number formats ------------------------------------------------------------
// E4M3 code of t >= 0: nearest-even, saturating at 448 (hardware cvt).
__device__ __forceinline__ uint32_t f32_to_e4m3(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(t));
  return r & 0xFFu;
}

// Value of an E4M3 code 0..126 (exact): subnormal m * 2^-9, else (1 + m/8) 2^(e-7).
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const uint32_t e = c >> 3, m = c & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20))
           : __fmul_rn((float)m, 0.001953125f);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Byte offset of scale (row r, block kb) in the tensor-core tiled layout
// (128 rows x 4 blocks per 512-byte tile, block index fastest between tiles).
__device__ __forceinline__ int64_t mma_scale_offset(int64_t r, int64_t kb, int64_t nkb_p) {
  return ((r >> 7) * (nkb_p >> 2) + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 +
         (kb & 3);
}

// Kahan-compensated FP32 running sum.
struct Kahan {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = __fsub_rn(x, c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
  }
  __device__ __forceinline__ double value() const { return (double)s - (double)c; }
};

// ---- quantisation plumbing shared by the kernel families ---------------------

struct CopyOut {
  uint8_t* codes;
  uint8_t* scales;
  float* tensor_scale;
  int mma;          // scale layout: 1 = tensor-core tiled
  int64_t ld;       // bytes per row of codes = (elements per row of the copy) / 2
  int64_t nkb;      // blocks per row of the copy
  int64_t nkb_p;    // blocks per row padded to 4 (tiled layout)
  int64_t rows;     // rows of the copy (per-128 scales in the tiled layout are column-major)
};


// Per-copy scale constants derived from the tensor amax (NVFP4 / UFP4).
struct Ctx {
  float g;       // tensor scale A / (Qmax * 448)
  float d;       // Qmax * g
  float inv_g;   // 1 / g (statistics of blocks whose scale rounds to 0)
};

__device__ __forceinline__ Ctx make_ctx(uint32_t amax_bits, float qmax, float qmax448) {
  Ctx c;
  const float a = __uint_as_float(amax_bits);
  c.g = __fdiv_rn(a, qmax448);
  c.d = __fmul_rn(qmax, c.g);
  c.inv_g = (c.g > 0.f) ? __frcp_rn(c.g) : 0.f;
  return c;
}


// ---------------------------------------------------------------------------
// CTA reductions and the last-CTA handshake.
// ---------------------------------------------------------------------------
template <int kNT>
__device__ __forceinline__ double cta_sum(double v, double* sh) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  double r = 0.0;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kNT / 32; ++w) r += sh[w];
  }
  __syncthreads();
  return r;   // meaningful in thread 0
}

template <int kNT>
__device__ __forceinline__ uint32_t cta_max(uint32_t v, uint32_t* sh) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  uint32_t r = 0;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kNT / 32; ++w) r = max(r, sh[w]);
  }
  __syncthreads();
  return r;
}

// SR uniform of one Philox word: its top 24 bits times 2^-24 (exact in FP32).
__device__ __forceinline__ float sr_u(uint32_t w) { return __uint2float_rz(w >> 8) * 5.9604644775390625e-08f; }

// Tensor amax (FP32 bits) of copy c, folded from the amax pass's per-CTA
// partials; every thread of the CTA gets it.
template <int kNT>
__device__ __forceinline__ uint32_t fold_amax(const Workspace* ws, int c, uint32_t* sh) {
  const uint32_t np = __ldcg(&ws->amax_nparts);
  uint32_t m = 0u;
  for (uint32_t i = threadIdx.x; i < np; i += kNT) m = max(m, __ldcg(&ws->amax_part[c][i]));
#pragma unroll
  for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = m;
  __syncthreads();
  uint32_t r = 0u;
#pragma unroll
  for (int w = 0; w < kNT / 32; ++w) r = max(r, sh[w]);
  __syncthreads();
  return r;
}

// FP32 sums of K values over the CTA; the results are meaningful in thread 0.
template <int kNT, int K>
__device__ __forceinline__ void cta_sums_f32(float (&v)[K], float (*sh)[kNT / 32]) {
#pragma unroll
  for (int k = 0; k < K; ++k) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v[k] += __shfl_xor_sync(0xFFFFFFFFu, v[k], o);
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) sh[k][threadIdx.x >> 5] = v[k];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      float r = 0.f;
      for (int w = 0; w < kNT / 32; ++w) r += sh[k][w];
      v[k] = r;
    }
  }
  __syncthreads();
}


// Barrier over every CTA of a co-resident (cooperatively launched) grid,
// through the workspace: the last CTA to arrive bumps the generation the
// others poll. Bounded: returns false (every thread) if the wait ran out.
__device__ __forceinline__ bool grid_barrier(Workspace* ws, uint64_t timeout_ns) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    volatile unsigned int* gen = &ws->gbar_gen;
    const unsigned int g0 = *gen;
    __threadfence();
    const unsigned int prev = atomicInc(&ws->gbar_count, gridDim.x - 1);
    if (prev == gridDim.x - 1) {
      __threadfence();
      atomicAdd(&ws->gbar_gen, 1u);
    } else {
      uint64_t t0 = 0;
      for (uint32_t i = 1; *gen == g0; ++i) {
        if ((i & 255u) == 0u) {
          uint64_t now;
          asm volatile("mov.u64 %0, %globaltimer;" : "=l"(now));
          if (t0 == 0) t0 = now;
          else if (now - t0 > timeout_ns) { ok = 0; break; }
        }
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

}  // namespace fp4q
