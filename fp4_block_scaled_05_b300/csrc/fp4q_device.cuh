// Device helpers for the fp4q kernels (sm_103a).
//
// Exact-path rule: every FP32 operation that decides a code or a scale is an
// explicit round-to-nearest intrinsic (__fadd_rn, __fmul_rn, __fdiv_rn,
// __frcp_rn), the translation units are built with -fmad=false, and no
// flush-to-zero is enabled, so each step is one IEEE operation in a fixed order.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace fp4q {

// ---- workspace shared by every call ------------------------------------------
constexpr int kMaxCtas = 2048;   // upper bound on the persistent grid of a quantise kernel

constexpr uint32_t kStatusNonfinite = 1u;
constexpr uint32_t kStatusTimeout = 2u;

struct Workspace {
  unsigned int status;          // sticky FP4Q status bits, cleared by fp4q_status
  unsigned int cnt_amax;        // last-CTA counters (wrap back to 0 by atomicInc)
  unsigned int cnt_quant;
  unsigned int copies;          // axis bits produced by the last quantise call
  unsigned int amax_bits[2];    // tensor amax (FP32 bits) of the row / column copy
  float tensor_scale[2];        // g of the row / column copy
  double sums[2][5];            // per copy: sum_bias, sum_sig2, sum_err2, n, Qmax
  unsigned int amax_part[2][kMaxCtas];
  double stat_part[2][3][kMaxCtas];
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

// Two FP32 values -> one byte of E2M1 codes (nearest-even, saturating at 6):
// `lo` lands in bits 0-3, `hi` in bits 4-7.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// One byte of E2M1 codes -> the two magnitudes (bits 0-3 -> lo, bits 4-7 -> hi).
__device__ __forceinline__ void e2m1x2_abs(uint32_t byte, float& lo, float& hi) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2) : "r"(byte));
  lo = fabsf(__half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))));
  hi = fabsf(__half2float(__ushort_as_half((unsigned short)(h2 >> 16))));
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// In-place 16-point RHT of w (already sign-flipped): stages h = 1, 2, 4, 8 of
// (a + b, a - b), then * 0.25, every step one FP32 rounding.
__device__ __forceinline__ void fwht16_quarter(float* w) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float a = w[i], b = w[i + h];
        w[i] = __fadd_rn(a, b);
        w[i + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = __fmul_rn(w[i], 0.25f);
}

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

}  // namespace fp4q
