// Block-scaled 4-bit quantisation kernels (sm_103a): the tensor-amax pass and
// the quantisation pass, as a flat stream for row-wise copies and as a tile
// stream for requests with the transposed copy; the one-launch quantiser for
// small row-wise tensors; the dequantiser.
//
// Method: "Replanteamiento del Sesgo de Contraccion en el Preentrenamiento de
// LLM en FP4" (Metodologia §1-2: E2M1 / uniform E1M2 grids, RTNE, stochastic
// rounding, RHT; Eficiencia: RHT fused into the quantisation pass);
// "TetraJet-v2 ..." (Riepilogo Tecnico §2A: NVFP4 16-element groups with an
// 8-bit scale under a per-tensor scale, SR); "Unveiling the Potential of
// Quantization with MXFP4 ..." (Resume technique §2: MXFP4 32-element E8M0
// blocks, NVFP4 16-element E4M3 blocks).
//
// Blocks of the row-wise copy never straddle a row (cols is a multiple of the
// block), so the copy is a flat stream of blocks: element e of the row-major
// source is element e of the copy, its codes sit at byte e/2 and its linear
// scale at e/b. Each CTA of a persistent grid walks chunks of 8192 elements;
// one thread keeps a ring of bulk (TMA) copies of the CTA's next chunks in
// flight into shared memory (16 KiB per BF16 chunk, 4 deep), so the loads
// overlap the arithmetic. A thread quantises 32 consecutive elements of a
// chunk (two 16-blocks, or one MXFP4 32-block) in registers, using packed
// FP32x2 operations where the lanes are independent; every value-deciding step
// is one IEEE round-to-nearest-even operation in the order of the method.
//
// Requests with the transposed copy (TetraJet-v2, Riepilogo Tecnico §2A) walk
// 64 x 128 tiles instead, brought in by 2-D TMA with the 128-byte swizzle, so
// that one read of the source serves the row-wise and the column-wise copy
// (see the tile section below).
#include <cfloat>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fp4q_device.cuh"
#include "fp4q_internal.h"
#include "fp4q_ptx.cuh"

namespace fp4q {
namespace {

constexpr int RT = 256;            // threads per CTA
constexpr int EPT = 32;            // elements per thread per chunk
constexpr int CH = RT * EPT;       // elements per chunk
constexpr uint64_t kRingTimeoutNs = 2000000000ull;

template <bool F32>
struct Ring {
  static constexpr int kChunkBytes = CH * (F32 ? 4 : 2);
  static constexpr int kStages = F32 ? 3 : 4;
  static constexpr int kSmem = kStages * kChunkBytes;
};

// Division by a fixed divisor d >= 1 for 32-bit numerators (round-up method
// of Granlund and Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994): q = (t + ((n - t) >> 1)) >> s, t = mulhi(m, n).
struct FastDiv {
  uint32_t d, m, s;
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    if (d == 1) return n;
    const uint32_t t = __umulhi(m, n);
    return (t + ((n - t) >> 1)) >> s;
  }
};

FastDiv make_fastdiv(uint32_t d) {
  FastDiv f{d, 0, 0};
  if (d <= 1) return f;
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  f.m = (uint32_t)(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
  f.s = l - 1;
  return f;
}

struct Flat {
  const uint8_t* src;
  int64_t n;          // elements
  int64_t nchunks;
  FastDiv nkb;        // blocks per row (tiled scale layout)
  int small;          // 1 when every block index fits in 32 bits
};

// ---- the ring ------------------------------------------------------------------
template <bool F32>
__device__ __forceinline__ void ring_issue(const Flat& f, int64_t chunk, uint8_t* ring, int slot,
                                           uint32_t bar) {
  constexpr int es = F32 ? 4 : 2;
  const int64_t e0 = chunk * CH;
  const int64_t ne = (f.n - e0 < CH) ? (f.n - e0) : CH;
  const uint32_t bytes = (uint32_t)(ne * es);        // a multiple of 32: blocks are whole
  mbar_arrive_expect_tx(bar, bytes);
  bulk_load(smem_u32(ring + slot * Ring<F32>::kChunkBytes), f.src + e0 * es, bytes, bar);
}

// The same ring with warps decoupled: empty[s] collects one arrival per warp
// once the warp is done with slot s, and only warp 0, which refills the slot,
// waits for the slowest; warps run ahead of one another by up to kStages - 1
// chunks. Every wait is bounded.
struct FlatPipe {
  uint64_t* full;
  uint64_t* empty;
  int64_t next_it;     // thread 0: the next iteration whose chunk is to be issued
};

template <bool F32>
__device__ __forceinline__ void flat_ring_start(const Flat& f, uint8_t* ring, FlatPipe& p, bool reverse) {
  constexpr int S = Ring<F32>::kStages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&p.full[s]), 1);
      mbar_init(smem_u32(&p.empty[s]), RT / 32);
    }
    fence_mbarrier_init();
  }
  __syncthreads();
  p.next_it = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      const int64_t c = blockIdx.x + (int64_t)s * gridDim.x;
      if (c >= f.nchunks) break;
      ring_issue<F32>(f, reverse ? f.nchunks - 1 - c : c, ring, s, smem_u32(&p.full[s]));
      p.next_it = s + 1;
    }
  }
}

// The calling warp is done with iteration `it` (chunk c of the CTA's walk).
// False if warp 0's wait for the other warps ran out.
template <bool F32>
__device__ __forceinline__ bool flat_ring_release(const Flat& f, uint8_t* ring, FlatPipe& p, int64_t it,
                                                  int64_t c, bool reverse, uint64_t timeout_ns) {
  constexpr int S = Ring<F32>::kStages;
  const int s = (int)(it % S);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&p.empty[s]));
  if (threadIdx.x < 32) {
    const int64_t nx = c + (int64_t)S * gridDim.x;
    if (nx < f.nchunks) {
      if (!mbar_wait_bounded(smem_u32(&p.empty[s]), (uint32_t)((it / S) & 1), timeout_ns)) return false;
      if (threadIdx.x == 0) {
        ring_issue<F32>(f, reverse ? f.nchunks - 1 - nx : nx, ring, s, smem_u32(&p.full[s]));
        p.next_it = it + S + 1;
      }
    }
  }
  return true;
}

// After a wait ran out: thread 0 waits (50 ms at most) for the copies that may
// still be in flight, the last kStages issued.
template <int S>
__device__ __forceinline__ void pipe_drain(const uint64_t* full, int64_t next_it) {
  if (threadIdx.x != 0) return;
  const uint64_t t0 = globaltimer();
  for (int64_t j = max((int64_t)0, next_it - S); j < next_it; ++j) {
    const uint32_t bar = smem_u32(&full[j % S]);
    while (!mbar_try_wait(bar, (uint32_t)((j / S) & 1)) && globaltimer() - t0 < 50000000ull) {
    }
  }
}

// ---- loading a thread's 32 elements as FP32 pairs -------------------------------
// Q[j] = {v[2j], v[2j+1]}, v the (transformed) values of elements 32t .. 32t+31
// of the chunk. With the RHT, each 16-block is sign-flipped by sigma, run
// through the butterfly stages 1, 2, 4, 8 and scaled by 1/4. Stages 1, 2, 4
// run on lanes {x_i, x_{i+8}} with packed adds; stage 8 pairs the two lanes.
__device__ __forceinline__ void rht16_pairs(float (&x)[16], f2* Q) {
  f2 P[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) P[i] = f2_make(x[i], x[i + 8]);
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((i & h) == 0) {
        const f2 a = P[i], b = P[i + h];
        P[i] = f2_add(a, b);
        P[i + h] = f2_sub(a, b);
      }
    }
  }
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float lo, hi;
    f2_split(P[i], lo, hi);
    v[i] = __fadd_rn(lo, hi);
    v[i + 8] = __fsub_rn(lo, hi);
  }
  const f2 quarter = f2_make(0.25f, 0.25f);
#pragma unroll
  for (int j = 0; j < 8; ++j) Q[j] = f2_mul(f2_make(v[2 * j], v[2 * j + 1]), quarter);
}

// Same butterfly without the final 1/4 and with plain scalar outputs (amax pass:
// max |round(w/4)| = round(max |w| / 4), since the scaling is monotone).
__device__ __forceinline__ void rht16_unscaled(float (&x)[16]) {
  f2 P[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) P[i] = f2_make(x[i], x[i + 8]);
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((i & h) == 0) {
        const f2 a = P[i], b = P[i + h];
        P[i] = f2_add(a, b);
        P[i + h] = f2_sub(a, b);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float lo, hi;
    f2_split(P[i], lo, hi);
    x[i] = __fadd_rn(lo, hi);
    x[i + 8] = __fsub_rn(lo, hi);
  }
}

// A thread's 32-element segment in shared memory, read as 16-byte chunks
// (4 for BF16, 8 for FP32). LinearSeg: the chunks are contiguous. SwzSeg: one
// row of a TMA box written with the 128-byte swizzle, where chunk c of row r
// sits at position c ^ (r & 7); `y` holds 16 * (first chunk ^ (r & 7)).
struct LinearSeg {
  const uint8_t* p;
  __device__ __forceinline__ uint4 chunk(int k) const { return *reinterpret_cast<const uint4*>(p + 16 * k); }
};
struct SwzSeg {
  const uint8_t* row;
  uint32_t y;
  __device__ __forceinline__ uint4 chunk(int k) const {
    return *reinterpret_cast<const uint4*>(row + ((16u * (uint32_t)k) ^ y));
  }
};

// Widen the 16 elements starting at chunk k0 of `sg` to FP32, flipping signs
// by `sign` when RHT (BF16: sign words hold sigma at bits 15 and 31; FP32: one
// bit per value).
template <bool F32, bool RHT, class Seg>
__device__ __forceinline__ void widen16(const Seg& sg, int k0, const uint32_t (&sgn)[16], float (&x)[16]) {
  if constexpr (F32) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 u = sg.chunk(k0 + k);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) x[4 * k + i] = __uint_as_float(RHT ? (w[i] ^ sgn[4 * k + i]) : w[i]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4 u = sg.chunk(k0 + k);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t s = RHT ? (w[i] ^ sgn[4 * k + i]) : w[i];
        x[8 * k + 2 * i] = __uint_as_float(s << 16);
        x[8 * k + 2 * i + 1] = __uint_as_float(s & 0xFFFF0000u);
      }
    }
  }
}

template <bool F32, bool RHT, class Seg>
__device__ __forceinline__ void load_block16(const Seg& sg, int k0, const uint32_t (&sgn)[16], f2* Q) {
  float x[16];
  widen16<F32, RHT>(sg, k0, sgn, x);
  if constexpr (RHT) {
    rht16_pairs(x, Q);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) Q[j] = f2_make(x[2 * j], x[2 * j + 1]);
  }
}

// Sign words: BF16 -> word i of a 16-block covers elements 2i, 2i+1 (bits 15,
// 31); FP32 -> one word per element (bit 31).
template <bool F32>
__device__ __forceinline__ void make_sign_words(uint32_t smask, uint32_t (&sgn)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if constexpr (F32) {
      sgn[i] = ((smask >> i) & 1u) << 31;
    } else {
      sgn[i] = (i < 8) ? ((((smask >> (2 * i)) & 1u) << 15) | (((smask >> (2 * i + 1)) & 1u) << 31)) : 0u;
    }
  }
}

// ---- per-block quantisation --------------------------------------------------------
// Formats (template argument FMT): 0 NVFP4, 1 MXFP4 (32-element blocks),
// 2 UFP4, 3 two-level NVFP4, 4 MXFP4 on 16-element blocks, 5 the same with the
// overflow-aware exponent rule, 6 MBS-static (16-element E8M0 blocks under a
// 128-element macro scale), 7 HiF4 (an E6M2 scale per 64 elements with
// halving bits per 8 and per 4 elements, uniform levels 0..7).
template <int FMT> constexpr bool kE8M0 = FMT == 1 || FMT == 4 || FMT == 5 || FMT == 6;
// formats with a per-tensor FP32 scale (and so an amax pass)
template <int FMT> constexpr bool kTensorScaled = FMT == 0 || FMT == 2;
// formats whose "tensor scale" array holds one FP32 scale per 128 elements
template <int FMT> constexpr bool kOuterScaled = FMT == 3 || FMT == 6;

struct Sums {        // per-thread running sums of one copy
  Kahan bias, sig, err;
  double sig64 = 0.0, err64 = 0.0;
  int e_ref = 0;     // per-block scales: sig / err are in units of 2^(2 (e_ref - 127)); 0 = not set yet
};

// Two-level NVFP4 and the E8M0 formats: add a thread's signal and error sums,
// in units of g^2 (g the outer scale, or the block's scale), to its running
// sums. FP32 Kahan sums in units of a power of two fixed by the first scale the
// thread meets (the exact power-of-two rescaling keeps them far from overflow
// and underflow); a scale more than 2^60 away from it, or subnormal, goes to
// the FP64 sums instead (FP64 arithmetic is slow on this GPU: the common case
// stays in FP32).
__device__ __forceinline__ void add_outer_stats(Sums& acc, float g, float ss, float es) {
  const int E = (int)((__float_as_uint(g) >> 23) & 0xFFu);
  if (acc.e_ref == 0 && E != 0 && E != 255) acc.e_ref = E;
  const int dE = E - acc.e_ref;
  if (E != 0 && E != 255 && dE >= -60 && dE <= 60) {
    const float w = __uint_as_float((uint32_t)((int)__float_as_uint(g) - (acc.e_ref - 127) * (1 << 23)));
    const float w2 = __fmul_rn(w, w);
    acc.sig.add(__fmul_rn(ss, w2));
    acc.err.add(__fmul_rn(es, w2));
  } else if (g != 0.f) {
    const double g2 = (double)g * (double)g;
    acc.sig64 += (double)ss * g2;
    acc.err64 += (double)es * g2;
  }
}

// The running sums of add_outer_stats in absolute units (FP64).
__device__ __forceinline__ void outer_stats_value(const Sums& acc, double& sig, double& err) {
  sig = acc.sig64;
  err = acc.err64;
  if (acc.e_ref != 0) {
    const double u = __longlong_as_double((long long)(1023 + 2 * (acc.e_ref - 127)) << 52);
    sig += acc.sig.value() * u;
    err += acc.err.value() * u;
  }
}

// Two plain FP32 sums, one per lane of a pair. The row-wise quantisation pass
// adds one partial per chunk to them (about 9 per thread at 2^25 elements, 300
// at 2^30): the relative error stays below that count times 2^-24 of the sum
// of magnitudes (typically its square root), and the compensation of Kahan2
// would cost that kernel register spills.
struct Sum2 {
  f2 s = 0ull;
  __device__ __forceinline__ void add(f2 x) { s = f2_add(s, x); }
  __device__ __forceinline__ float value_f() const {   // both lanes together
    float s0, s1;
    f2_split(s, s0, s1);
    return __fadd_rn(s0, s1);
  }
};

// Two independent Kahan-compensated FP32 sums, one per lane of a pair.
struct Kahan2 {
  f2 s = 0ull, c = 0ull;
  __device__ __forceinline__ void add(f2 x) {
    const f2 y = f2_sub(x, c);
    const f2 t = f2_add(s, y);
    c = f2_sub(f2_sub(t, s), y);
    s = t;
  }
  __device__ __forceinline__ float value_f() const {   // both lanes together
    float s0, s1, c0, c1;
    f2_split(s, s0, s1);
    f2_split(c, c0, c1);
    return __fadd_rn(__fsub_rn(s0, c0), __fsub_rn(s1, c1));
  }
};

// max(m, |a|, |b|), NaN-propagating.
__device__ __forceinline__ float max3_abs_nan(float m, float a, float b) {
  float d;
  asm("{\n\t.reg .f32 x, y;\n\tabs.f32 x, %2;\n\tabs.f32 y, %3;\n\tmax.NaN.f32 %0, %1, x, y;\n\t}"
      : "=f"(d) : "f"(m), "f"(a), "f"(b));
  return d;
}

// Per-CTA constants of the E4M3 block scales (NVFP4/UFP4), for each of the
// 128 codes: r = 1 / RN(s * g) rounded to nearest (0 when the product is 0,
// FLT_MAX when it overflows; the NaN code 127 maps to 0) and s^2, s the
// code's value. A block's normaliser and statistics weight are then one table
// read instead of a decode, a product and a reciprocal per block.
__device__ __forceinline__ float2 scale_entry(uint32_t c, float g) {
  const float s = (c < 127) ? e4m3_to_f32(c) : 0.f;
  const float p = __fmul_rn(s, g);
  float r = (p == 0.f) ? 0.f : __frcp_rn(p);
  if (r > FLT_MAX) r = FLT_MAX;
  return make_float2(r, __fmul_rn(s, s));
}

__device__ __forceinline__ void fill_scale_table(float2* tab, float g) {
  for (int c = threadIdx.x; c < 128; c += blockDim.x) tab[c] = scale_entry((uint32_t)c, g);
}

// t = RN(m / d) for both lanes. With y = RN(1/d) two correction steps
// q <- RN(q + RN(m - q d) y) give the correctly rounded quotient (Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990); used only when d lies in
// [2^-38, 2^50], where no step underflows or overflows.
struct Divider {
  int fast;
  float d;
  f2 nd2, y2;
  __device__ __forceinline__ void init(float dd) {
    d = dd;
    fast = (dd >= 3.637978807091713e-12f && dd <= 1.125899906842624e15f) ? 1 : 0;
    const float y = fast ? __frcp_rn(dd) : 0.f;
    nd2 = f2_make(-dd, -dd);
    y2 = f2_make(y, y);
  }
  __device__ __forceinline__ f2 div(f2 m) const {
    if (fast) {
      const f2 q0 = f2_mul(m, y2);
      const f2 q1 = f2_fma(f2_fma(nd2, q0, m), y2, q0);
      return f2_fma(f2_fma(nd2, q1, m), y2, q1);
    }
    float a, b;
    f2_split(m, a, b);
    return f2_make(__fdiv_rn(a, d), __fdiv_rn(b, d));
  }
};

// One E2M1 byte (nearest-even, saturating) of the pair Y and the rounding
// errors |q| - |y| of its two lanes.
__device__ __forceinline__ uint32_t e2m1_pair(f2 Y, f2& D) {
  float y0, y1;
  f2_split(Y, y0, y1);
  uint32_t byte, hq;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %3, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t"
      "and.b32 %1, %0, 0x77;\n\t"
      "cvt.u8.u32 t, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, t;\n\t}"
      : "=r"(byte), "=r"(hq) : "f"(y0), "f"(y1));
  D = f2_make(sub_f16_f32((uint16_t)(hq & 0xFFFFu), fabsf(y0)),
              sub_f16_f32((uint16_t)(hq >> 16), fabsf(y1)));
  return byte;
}

// One UFP4 byte: |y| clamped to 7 and rounded to the nearest integer, ties to
// even (adding 2^23 rounds to an integer in FP32), sign kept in bit 3.
__device__ __forceinline__ uint32_t ufp4_pair(f2 Y, f2& D) {
  float y0, y1;
  f2_split(Y, y0, y1);
  const float a0 = fabsf(y0), a1 = fabsf(y1);
  const f2 magic = f2_make(8388608.f, 8388608.f);
  const f2 T = f2_add(f2_make(fminf(a0, 7.f), fminf(a1, 7.f)), magic);
  const f2 Qv = f2_sub(T, magic);
  D = f2_sub(Qv, f2_make(a0, a1));
  float t0, t1;
  f2_split(T, t0, t1);
  return (__float_as_uint(t0) & 7u) | ((__float_as_uint(t1) & 7u) << 4) |
         ((__float_as_uint(y0) >> 31) << 3) | ((__float_as_uint(y1) >> 31) << 7);
}

// ---- stochastic rounding of a pair, without branches ------------------------------
// The level goes up iff u < f, f = (|y| - lo) / step the exact fraction of the
// way from the level below to the one above and u = (w >> 8) 2^-24 the
// element's uniform. Both grids have power-of-two steps, so f is exact; floor
// is an addition of 2^23 rounded toward zero (exact below 2^23).
__device__ __forceinline__ f2 f2_add_rz(f2 a, f2 b) {
  f2 d;
  asm("add.rz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// E2M1: with a = min(|y|, 6) and E = max(floor(log2 a), 0) the neighbouring
// levels are lo and lo + step, step = 2^(E-1) (0.5 below 2, then 1, then 2):
// t = a / step, lo = floor(t) step. The grid value q is exact and its code
// (sign of y kept) comes from the nearest-even conversion of the signed q.
__device__ __forceinline__ uint32_t sr_pair_e2m1(f2 Y, uint32_t w0, uint32_t w1, f2& D) {
  float y0, y1;
  f2_split(Y, y0, y1);
  const float a0 = fminf(fabsf(y0), 6.f), a1 = fminf(fabsf(y1), 6.f);
  const uint32_t m0 = max(__float_as_uint(a0) >> 23, 127u), m1 = max(__float_as_uint(a1) >> 23, 127u);
  const f2 T = f2_mul(f2_make(a0, a1),
                      f2_make(__uint_as_float((255u - m0) << 23), __uint_as_float((255u - m1) << 23)));
  const f2 magic = f2_make(8388608.f, 8388608.f);
  const f2 FL = f2_sub(f2_add_rz(T, magic), magic);
  float t0, t1, l0, l1;
  f2_split(T, t0, t1);
  f2_split(FL, l0, l1);
  const float v0 = (sr_u(w0) < __fsub_rn(t0, l0)) ? __fadd_rn(l0, 1.f) : l0;
  const float v1 = (sr_u(w1) < __fsub_rn(t1, l1)) ? __fadd_rn(l1, 1.f) : l1;
  const f2 Q = f2_mul(f2_make(v0, v1),
                      f2_make(__uint_as_float((m0 - 1u) << 23), __uint_as_float((m1 - 1u) << 23)));
  D = f2_sub(Q, f2_make(fabsf(y0), fabsf(y1)));
  float q0, q1;
  f2_split(Q, q0, q1);
  uint32_t byte;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(byte) : "f"(copysignf(q0, y0)), "f"(copysignf(q1, y1)));
  return byte;
}

// UFP4: integer levels 0..7; with a = min(|y|, 7), lo = floor(a), whose low
// three bits sit in the mantissa of a + 2^23 (rounded toward zero).
__device__ __forceinline__ uint32_t sr_pair_ufp4(f2 Y, uint32_t w0, uint32_t w1, f2& D) {
  float y0, y1;
  f2_split(Y, y0, y1);
  const f2 A = f2_make(fminf(fabsf(y0), 7.f), fminf(fabsf(y1), 7.f));
  const f2 magic = f2_make(8388608.f, 8388608.f);
  const f2 T = f2_add_rz(A, magic);
  const f2 L = f2_sub(T, magic);
  const f2 F = f2_sub(A, L);
  float l0, l1, f0, f1, t0, t1;
  f2_split(L, l0, l1);
  f2_split(F, f0, f1);
  f2_split(T, t0, t1);
  const uint32_t u0 = (sr_u(w0) < f0) ? 1u : 0u, u1 = (sr_u(w1) < f1) ? 1u : 0u;
  D = f2_sub(f2_make(__fadd_rn(l0, (float)u0), __fadd_rn(l1, (float)u1)), f2_make(fabsf(y0), fabsf(y1)));
  const uint32_t k0 = (__float_as_uint(t0) & 7u) + u0, k1 = (__float_as_uint(t1) & 7u) + u1;
  return (k0 | ((__float_as_uint(y0) >> 31) << 3)) | ((k1 | ((__float_as_uint(y1) >> 31) << 3)) << 4);
}

template <int FMT>
__device__ __forceinline__ uint32_t sr_pair(f2 Y, uint32_t w0, uint32_t w1, f2& D) {
  if constexpr (FMT == 2) return sr_pair_ufp4(Y, w0, w1, D);
  else return sr_pair_e2m1(Y, w0, w1, D);
}

// MBS-static macro scale: alpha / 6 rounded to nearest, ties to even, on
// FP32's grid with 8 fraction bits (the low 15 bits of the FP32 encoding zero).
// The quotient q is correctly rounded and alpha - 6 q is exact (fma), so when
// q falls on a tie of the 8-bit grid the remainder's sign says on which side
// the exact quotient lies.
__device__ __forceinline__ float mbs_macro_scale(float alpha) {
  const float q = __fdiv_rn(alpha, 6.f);
  const float rem = __fmaf_rn(-6.f, q, alpha);
  const uint32_t b = __float_as_uint(q);
  const uint32_t low = b & 0x7FFFu, base = b - low;
  const bool up = low > 0x4000u || (low == 0x4000u && (rem > 0.f || (rem == 0.f && (base & 0x8000u))));
  return __uint_as_float(base + (up ? 0x8000u : 0u));
}

// HiF4's block scale: an unsigned E6M2 value (6 exponent bits with bias 31,
// 2 mantissa bits, subnormals below 2^-30 in steps of 2^-32, every code
// finite). t >= 0 is rounded to the nearest value, ties to the even code, and
// saturates at 1.75 * 2^32. In the normal range the rounding keeps 2 of
// FP32's 23 fraction bits (a carry into the exponent is the correct result);
// below it, t * 2^32 (exact) is rounded to an integer, ties to even.
__device__ __forceinline__ float e6m2_rne_sat(float t, uint32_t& code) {
  if (t >= 9.313225746154785e-10f) {                         // 2^-30
    const uint32_t b = __float_as_uint(t);
    uint32_t u = (b + 0x000FFFFFu + ((b >> 21) & 1u)) & ~0x001FFFFFu;
    if (u > 0x4FE00000u) u = 0x4FE00000u;                    // 1.75 * 2^32 (and +inf)
    code = (((u >> 23) - 96u) << 2) | ((u >> 21) & 3u);     // E = FP32 exponent - 127 + 31
    return __uint_as_float(u);
  }
  const float k = rintf(__fmul_rn(t, 4294967296.f));         // 0 .. 4 (4 is 2^-30, code 4)
  code = (uint32_t)k;
  return __fmul_rn(k, 2.3283064365386963e-10f);              // k * 2^-32
}

// HiF4's codes and statistics for one half block (see hif4_half), with the
// halving bits decided from the micro-block maxima a4. The signal and error
// sums are FP32 in units of a power of two times S^2 (add_outer_stats):
//   MODE 0  y and y - q as they are, units S^2;
//   MODE 1  a scale saturated so far below the values that sums of y^2 could
//           overflow FP32: y 2^-64 and (q - y) 2^-64, units (S 2^64)^2;
//   MODE 2  a scale that rounded to 0: every value becomes 0 and its error is
//           v itself; v 2^64 for both sums, units 2^-128.
// Every scaling is by a power of two, exact but for what underflows next to
// the block's largest terms.
template <bool SR, int MODE>
__device__ __forceinline__ void hif4_codes(const f2 (&Q)[16], const float (&a4)[8], float S, float r,
                                           uint64_t e0, const PhiloxKey& pk, uint32_t axis, uint32_t (&cw)[4],
                                           uint32_t& mine, Sums& acc) {
  const f2 R = f2_make(r, r);
  const float k = MODE == 1 ? 5.421010862427522e-20f : 1.8446744073709552e19f;     // 2^-64, 2^64
  const f2 K = f2_make(k, k);
  float bsum = 0.f, ss = 0.f, es = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t d8 = (__fmul_rn(fmaxf(a4[2 * j], a4[2 * j + 1]), r) <= 3.5f) ? 1u : 0u;
    mine |= d8 << j;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = 2 * j + h;
      const uint32_t d4 = (__fmul_rn(a4[i], r) <= (d8 ? 1.75f : 3.5f)) ? 1u : 0u;
      mine |= d4 << (4 + i);
      const uint32_t sh = d8 + d4;
      const f2 M = f2_make(__uint_as_float((127u + sh) << 23), __uint_as_float((127u + sh) << 23));
      uint4 rw = make_uint4(0u, 0u, 0u, 0u);
      if constexpr (SR) {   // the micro-block's four uniforms: one Philox call
        const uint64_t q = (e0 >> 2) + (uint64_t)i;
        rw = philox4x32_10(make_uint4((uint32_t)q, (uint32_t)(q >> 32), axis, 0u), pk);
      }
      f2 B2 = f2_make(0.f, 0.f), E2 = B2, S2 = B2;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const f2 Y = f2_mul(f2_mul(Q[2 * i + t], R), M);
        f2 D;
        uint32_t byte;
        if constexpr (SR) {
          byte = (t == 0) ? sr_pair<2>(Y, rw.x, rw.y, D) : sr_pair<2>(Y, rw.z, rw.w, D);
        } else {
          byte = ufp4_pair(Y, D);
        }
        cw[i >> 1] |= byte << (8 * ((2 * i + t) & 3));
        B2 = f2_add(B2, D);
        if constexpr (MODE == 0) {
          E2 = f2_fma(D, D, E2);
          S2 = f2_fma(Y, Y, S2);
        } else if constexpr (MODE == 1) {
          const f2 Dk = f2_mul(D, K), Yk = f2_mul(Y, K);
          E2 = f2_fma(Dk, Dk, E2);
          S2 = f2_fma(Yk, Yk, S2);
        } else {
          const f2 Vk = f2_mul(Q[2 * i + t], K);
          S2 = f2_fma(Vk, Vk, S2);
        }
      }
      float x0, x1;
      f2_split(B2, x0, x1);
      bsum = __fadd_rn(bsum, __fadd_rn(x0, x1));
      const float wt = MODE == 2 ? 1.f : __uint_as_float((127u - 2u * sh) << 23);   // 4^-shift
      f2_split(S2, x0, x1);
      ss = __fmaf_rn(__fadd_rn(x0, x1), wt, ss);
      if constexpr (MODE != 2) {
        f2_split(E2, x0, x1);
        es = __fmaf_rn(__fadd_rn(x0, x1), wt, es);
      }
    }
  }
  acc.bias.add(bsum);
  if constexpr (MODE == 0) {
    add_outer_stats(acc, S, ss, es);
  } else if constexpr (MODE == 1) {
    add_outer_stats(acc, __fmul_rn(S, 1.8446744073709552e19f), ss, es);
  } else {
    add_outer_stats(acc, 5.421010862427522e-20f, ss, ss);
  }
}

// HiF4 ("Unleashing Low-Bit Inference on Ascend NPUs: A Comprehensive
// Evaluation of HiFloat Formats", Resumen tecnico §2 Metodologia): quantise the
// calling thread's half of a 64-element block; the other half is held by the
// lane whose index differs in bit 0. The two share the block's amax a, which
// sets the E6M2 scale S = RN_E6M2(a / 7). Each thread then decides, for its
// four 8-element sub-blocks and eight 4-element micro-blocks, whether the
// group's step can be halved without a value clamping at 7 (w = RN(a_group /
// S) <= 3.5, and <= 1.75 for a micro-block whose sub-block already halved),
// and rounds y = RN(v / S) 2^shift onto the levels 0..7.
//   Q      the half's 32 values in order (16 pairs); read only when `valid`
//   e0     index of the half's first element in the copy (SR counters)
// Writes the half's four code words; returns the block's scale word (E6M2
// code, the eight sub-block bits, the sixteen micro-block bits) to the lane
// with bit 0 clear. Every lane of the warp must call it (two shuffles).
template <bool SR>
__device__ __forceinline__ uint32_t hif4_half(const f2 (&Q)[16], bool valid, uint64_t e0, const PhiloxKey& pk,
                                              uint32_t axis, uint32_t (&cw)[4], Sums& acc, uint32_t& nonfinite) {
  float a4[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a = 0.f, b = 0.f, c = 0.f, d = 0.f;
    if (valid) {
      f2_split(Q[2 * i], a, b);
      f2_split(Q[2 * i + 1], c, d);
    }
    a4[i] = max3_abs_nan(max3_abs_nan(0.f, a, b), c, d);
  }
  float m = max_abs_nan(max_abs_nan(max_abs_nan(a4[0], a4[1]), max_abs_nan(a4[2], a4[3])),
                        max_abs_nan(max_abs_nan(a4[4], a4[5]), max_abs_nan(a4[6], a4[7])));
  m = max_abs_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  uint32_t mine = 0u, scode = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j) cw[j] = 0u;
  if (valid) {
    nonfinite |= (__float_as_uint(m) >= 0x7F800000u) ? 1u : 0u;
    const float S = e6m2_rne_sat(__fdiv_rn(m, 7.f), scode);
    const float r = (S == 0.f) ? 0.f : __frcp_rn(S);
    // y <= 4 RN(a r): past 1e17 the FP32 sums of y^2 could overflow (NaN lands there too)
    if (S == 0.f) {
      hif4_codes<SR, 2>(Q, a4, S, r, e0, pk, axis, cw, mine, acc);
    } else if (__fmul_rn(m, r) <= 1.0e17f) {
      hif4_codes<SR, 0>(Q, a4, S, r, e0, pk, axis, cw, mine, acc);
    } else {
      hif4_codes<SR, 1>(Q, a4, S, r, e0, pk, axis, cw, mine, acc);
    }
  }
  // the block's word: E6M2 code, the eight sub-block bits, then the sixteen
  // micro-block bits (the lower half's first)
  const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, mine, 1);
  return scode | ((mine & 0xFu) << 8) | ((other & 0xFu) << 12) | (((mine >> 4) & 0xFFu) << 16) |
         (((other >> 4) & 0xFFu) << 24);
}

// Quantise one block of NP pairs (NP = 8: a 16-block, NP = 16: an MXFP4
// 32-block) whose first element has index e0 in the copy. Writes NP/4 code
// words and returns the scale code; adds the block's sums to bsum/ssum/esum
// (NVFP4/UFP4: grid units times s^2; MXFP4: FP64 absolute in sig64/err64).
template <int FMT, bool SR, int NP>
__device__ __forceinline__ uint32_t quant_block(const f2* Q, const Ctx& cx, uint64_t e0, const PhiloxKey& pk,
                                                uint32_t* cw, float& bsum, float& ssum, float& esum,
                                                Sums& acc, uint32_t& nonfinite, uint32_t axis = 0u,
                                                float s_macro = 1.f) {
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    float a, b;
    f2_split(Q[j], a, b);
    m = max_abs_nan(m, a);
    m = max_abs_nan(m, b);
  }
  nonfinite |= (__float_as_uint(m) >= 0x7F800000u) ? 1u : 0u;
  uint32_t scode;
  float r, s2 = 0.f;
  if constexpr (kE8M0<FMT>) {
    // OCP rule: e = floor(log2 m) - 2 puts m / 2^e in [4, 8); the overflow-aware
    // rule (FMT 5) adds one when m's significand is above 1.75, which puts
    // m / 2^e in (3.5, 7]
    const uint32_t mb = __float_as_uint(m);
    const uint32_t E = mb >> 23;
    const int msb = mb ? 31 - __clz((int)mb) : 0;
    int fl = E ? (int)E - 127 : (mb ? msb - 149 : -200);
    if constexpr (FMT == 5) {
      const uint32_t frac = E ? (mb & 0x7FFFFFu) : ((mb << (23 - msb)) & 0x7FFFFFu);
      if (frac > 0x600000u) ++fl;
    }
    const int e = max(-127, min(127, fl - 2));
    scode = (uint32_t)(e + 127);
    r = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e, e in [-127, 126]
  } else {
    if (cx.g == 0.f) {
      scode = 0;
      r = 0.f;
    } else {
      scode = f32_to_e4m3(__fdiv_rn(m, cx.d));
      const float p = __fmul_rn(e4m3_to_f32(scode), cx.g);
      r = (p == 0.f) ? 0.f : __frcp_rn(p);
      if (r > FLT_MAX) r = FLT_MAX;
    }
    const float s = e4m3_to_f32(scode);
    s2 = __fmul_rn(s, s);
  }

  const f2 R = f2_make(r, r);
  f2 B2 = f2_make(0.f, 0.f), E2 = B2, S2 = B2;
#pragma unroll
  for (int j = 0; j < NP / 4; ++j) cw[j] = 0u;
#pragma unroll
  for (int j0 = 0; j0 < NP; j0 += 2) {
    uint4 rw = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (SR) {   // one Philox call per 4 elements (e0 is a multiple of 16)
      const uint64_t q = (e0 >> 2) + (uint64_t)(j0 >> 1);
      rw = philox4x32_10(make_uint4((uint32_t)q, (uint32_t)(q >> 32), axis, 0u), pk);
    }
#pragma unroll
    for (int j = j0; j < j0 + 2; ++j) {
      const f2 Y = f2_mul(Q[j], R);
      f2 D;
      uint32_t byte;
      if constexpr (SR) {
        byte = (j == j0) ? sr_pair<FMT>(Y, rw.x, rw.y, D) : sr_pair<FMT>(Y, rw.z, rw.w, D);
      } else if constexpr (FMT == 2) {
        byte = ufp4_pair(Y, D);
      } else {
        byte = e2m1_pair(Y, D);
      }
      cw[j >> 2] |= byte << (8 * (j & 3));
      B2 = f2_add(B2, D);
      E2 = f2_fma(D, D, E2);
      S2 = f2_fma(Y, Y, S2);
    }
  }
  float b0, b1, e0f, e1f, s0, s1;
  f2_split(B2, b0, b1);
  f2_split(E2, e0f, e1f);
  f2_split(S2, s0, s1);
  const float bs = __fadd_rn(b0, b1), es = __fadd_rn(e0f, e1f), ys = __fadd_rn(s0, s1);
  bsum = __fadd_rn(bsum, bs);
  if constexpr (kE8M0<FMT>) {
    // in units of the block's scale squared: 2^e (2^-127 for code 0), times S
    // under a macro scale (exact unless it underflows; then in FP64)
    const float sv = scode ? __uint_as_float(scode << 23) : __uint_as_float(0x00400000u);
    const float g = (FMT == 6) ? __fmul_rn(sv, s_macro) : sv;
    if (FMT == 6 && g < FLT_MIN && s_macro != 0.f) {
      const double w = (double)sv * (double)s_macro;
      acc.sig64 += (double)ys * w * w;
      acc.err64 += (double)es * w * w;
    } else {
      add_outer_stats(acc, g, ys, es);
    }
  } else if (scode == 0 && cx.g > 0.f) {
    // the scale rounded to 0: every element becomes 0 and its error is v itself
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      float a, b;
      f2_split(Q[j], a, b);
      const float wa = __fmul_rn(a, cx.inv_g), wb = __fmul_rn(b, cx.inv_g);
      z = __fmaf_rn(wa, wa, __fmaf_rn(wb, wb, z));
    }
    ssum = __fadd_rn(ssum, z);
    esum = __fadd_rn(esum, z);
  } else {
    ssum = __fadd_rn(ssum, __fmul_rn(ys, s2));
    esum = __fadd_rn(esum, __fmul_rn(es, s2));
  }
  return scode;
}

// Quantise the thread's two consecutive 16-blocks (NVFP4 or UFP4) at `p`,
// elements e .. e+31 of the copy. The scalar steps of both blocks run in the
// two lanes of FP32 pairs. Writes four code words and two scale codes; adds
// the blocks' bias / signal / error sums (grid units, signal and error times
// s^2) to the lanes of bias2 / sig2 / err2.
template <int FMT, bool SR, bool TAB = true>
__device__ __forceinline__ void quant_two16_vals(const f2* Q, float m0, float m1, const Ctx& cx,
                                                 const Divider& dv, const float2* tab, uint64_t e0,
                                                 uint64_t e1, const PhiloxKey& pk, uint32_t axis,
                                                 uint32_t (&cw)[4], uint32_t (&sc)[2], f2& bias2,
                                                 f2& sig2, f2& err2, uint32_t& nonfinite);

template <int FMT, bool F32, bool RHT, bool SR, class Seg>
__device__ __forceinline__ void quant_two16(const Seg& sg, const uint32_t (&sgn)[16], const Ctx& cx,
                                            const Divider& dv, const float2* tab, uint64_t e,
                                            const PhiloxKey& pk, uint32_t (&cw)[4], uint32_t (&sc)[2],
                                            f2& bias2, f2& sig2, f2& err2, uint32_t& nonfinite) {
  f2 Q[16];
  float m0 = 0.f, m1 = 0.f;
  if constexpr (!F32 && !RHT) {
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 u = sg.chunk(k);
      w[4 * k] = u.x; w[4 * k + 1] = u.y; w[4 * k + 2] = u.z; w[4 * k + 3] = u.w;
    }
    uint32_t a0 = 0u, a1 = 0u;     // block maxima on the BF16 pairs
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      a0 = max_abs_nan_bf16x2(a0, w[k]);
      a1 = max_abs_nan_bf16x2(a1, w[k + 8]);
    }
    m0 = max3_abs_nan(0.f, bf16lo(a0), bf16hi(a0));
    m1 = max3_abs_nan(0.f, bf16lo(a1), bf16hi(a1));
#pragma unroll
    for (int j = 0; j < 16; ++j) Q[j] = f2_make(bf16lo(w[j]), bf16hi(w[j]));
  } else {
    load_block16<F32, RHT>(sg, 0, sgn, Q);
    load_block16<F32, RHT>(sg, F32 ? 4 : 2, sgn, Q + 8);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float a, b;
      f2_split(Q[j], a, b);
      m0 = max3_abs_nan(m0, a, b);
      f2_split(Q[j + 8], a, b);
      m1 = max3_abs_nan(m1, a, b);
    }
  }
  quant_two16_vals<FMT, SR>(Q, m0, m1, cx, dv, tab, e, e + 16, pk, 0u, cw, sc, bias2, sig2, err2,
                            nonfinite);
}

// Quantise two 16-blocks given as FP32 pairs (block 0 in Q[0..7], block 1 in
// Q[8..15], pair j holding elements 2j and 2j+1) with their maxima |v| m0, m1;
// e0, e1 are the blocks' first element indices in the copy, `axis` the copy
// (0 row-wise, 1 column-wise) for the SR counter. TAB: the normaliser and s^2
// of a scale code come from the CTA's table `tab`; else they are computed from
// cx.g, as the table computes them (the scale g differs between threads).
template <int FMT, bool SR, bool TAB>
__device__ __forceinline__ void quant_two16_vals(const f2* Q, float m0, float m1, const Ctx& cx,
                                                 const Divider& dv, const float2* tab, uint64_t e0,
                                                 uint64_t e1, const PhiloxKey& pk, uint32_t axis,
                                                 uint32_t (&cw)[4], uint32_t (&sc)[2], f2& bias2,
                                                 f2& sig2, f2& err2, uint32_t& nonfinite) {
  nonfinite |= (max(__float_as_uint(m0), __float_as_uint(m1)) >= 0x7F800000u) ? 1u : 0u;

  sc[0] = sc[1] = 0u;
  if (cx.g > 0.f) {
    float t0, t1;
    f2_split(dv.div(f2_make(m0, m1)), t0, t1);
    uint16_t c2;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c2) : "f"(t1), "f"(t0));
    sc[0] = c2 & 0xFFu;
    sc[1] = (uint32_t)c2 >> 8;
  }
  float2 T0, T1;
  if constexpr (TAB) {
    T0 = tab[sc[0]];
    T1 = tab[sc[1]];
  } else {
    T0 = scale_entry(sc[0], cx.g);
    T1 = scale_entry(sc[1], cx.g);
  }

  float bs[2], ys[2], es[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const f2 R = b ? f2_make(T1.x, T1.x) : f2_make(T0.x, T0.x);
    f2 B2 = 0ull, E2 = 0ull, S2 = 0ull;
    cw[2 * b] = 0u;
    cw[2 * b + 1] = 0u;
#pragma unroll
    for (int j0 = 0; j0 < 8; j0 += 2) {
      uint4 rw = make_uint4(0u, 0u, 0u, 0u);
      if constexpr (SR) {   // one Philox call per 4 elements
        const uint64_t q = ((b ? e1 : e0) >> 2) + (uint64_t)(j0 >> 1);
        rw = philox4x32_10(make_uint4((uint32_t)q, (uint32_t)(q >> 32), axis, 0u), pk);
      }
#pragma unroll
      for (int j = j0; j < j0 + 2; ++j) {
        const f2 Y = f2_mul(Q[8 * b + j], R);
        f2 D;
        uint32_t byte;
        if constexpr (SR) {
          byte = (j == j0) ? sr_pair<FMT>(Y, rw.x, rw.y, D) : sr_pair<FMT>(Y, rw.z, rw.w, D);
        } else if constexpr (FMT == 2) {
          byte = ufp4_pair(Y, D);
        } else {
          byte = e2m1_pair(Y, D);
        }
        cw[2 * b + (j >> 2)] += byte << (8 * (j & 3));
        B2 = f2_add(B2, D);
        E2 = f2_fma(D, D, E2);
        S2 = f2_fma(Y, Y, S2);
      }
    }
    float x0, x1;
    f2_split(B2, x0, x1);
    bs[b] = __fadd_rn(x0, x1);
    f2_split(E2, x0, x1);
    es[b] = __fadd_rn(x0, x1);
    f2_split(S2, x0, x1);
    ys[b] = __fadd_rn(x0, x1);
  }
  bias2 = f2_add(bias2, f2_make(bs[0], bs[1]));
  const f2 W = f2_make(T0.y, T1.y);
  sig2 = f2_fma(f2_make(ys[0], ys[1]), W, sig2);
  err2 = f2_fma(f2_make(es[0], es[1]), W, err2);
  if (cx.g > 0.f && (sc[0] == 0u || sc[1] == 0u)) {
    // a scale that rounded to 0: its block's elements become 0 and their
    // error is the value itself
    float z[2] = {0.f, 0.f};
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      if (sc[b] == 0u) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float a, c;
          f2_split(Q[8 * b + j], a, c);
          const float wa = __fmul_rn(a, cx.inv_g), wc = __fmul_rn(c, cx.inv_g);
          z[b] = __fmaf_rn(wa, wa, __fmaf_rn(wc, wc, z[b]));
        }
      }
    }
    const f2 Z = f2_make(z[0], z[1]);
    sig2 = f2_add(sig2, Z);
    err2 = f2_add(err2, Z);
  }
}

// The tensor cores read one scale per 16 elements along K: in the MMA layout a
// 32-element block's scale (DUP) is written for both of its halves, as one
// 2-byte store (the pair starts on an even byte).
template <bool DUP = false>
__device__ __forceinline__ void put_scale(const CopyOut& o, const Flat& f, uint64_t blk, uint32_t sc) {
  if (!o.mma) {
    o.scales[blk] = (uint8_t)sc;
    return;
  }
  uint64_t r;
  if (f.small) {
    r = f.nkb.div((uint32_t)blk);
  } else {
    r = blk / f.nkb.d;
  }
  const uint64_t kb = blk - r * f.nkb.d;
  if constexpr (DUP) {
    *reinterpret_cast<uint16_t*>(o.scales + mma_scale_offset((int64_t)r, (int64_t)(2 * kb), o.nkb_p)) =
        (uint16_t)(sc | (sc << 8));
  } else {
    o.scales[mma_scale_offset((int64_t)r, (int64_t)kb, o.nkb_p)] = (uint8_t)sc;
  }
}

// Index of the FP32 scale of element e's 128-element outer (or macro) block:
// rows x cols/128 row-major, or, with the tiled scale layout, column-major
// (cols/128 x rows), so that the scales of one 128-element K chunk of
// consecutive rows are contiguous for the GEMM.
__device__ __forceinline__ int64_t outer_index(const CopyOut& o, const Flat& f, int64_t e) {
  if (!o.mma) return e / 128;
  const uint64_t blk = (uint64_t)e / 16;
  const uint64_t r = f.small ? (uint64_t)f.nkb.div((uint32_t)blk) : blk / f.nkb.d;
  const uint64_t kc = (blk - r * f.nkb.d) / 8;
  return (int64_t)(kc * (uint64_t)o.rows + r);
}

// ---- per-thread work on its 32 elements of a ring slot ---------------------------------
// Running max |v| of the (up to two) 16-blocks at p: `m` (FP32 values; |w| = 4|v|
// with the RHT) or `m2` (BF16 pairs, no RHT).
template <bool F32, bool RHT, class Seg>
__device__ __forceinline__ void amax_segment(const Seg& sg, int nb, const uint32_t (&sgn)[16], float& m,
                                             uint32_t& m2) {
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    if (b < nb) {
      const int kb = b * (F32 ? 4 : 2);
      if constexpr (!RHT && !F32) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint4 u = sg.chunk(kb + k);
          m2 = max_abs_nan_bf16x2(m2, u.x);
          m2 = max_abs_nan_bf16x2(m2, u.y);
          m2 = max_abs_nan_bf16x2(m2, u.z);
          m2 = max_abs_nan_bf16x2(m2, u.w);
        }
      } else {
        float x[16];
        widen16<F32, RHT>(sg, kb, sgn, x);
        if (RHT) rht16_unscaled(x);
#pragma unroll
        for (int i = 0; i < 16; i += 2) m = max3_abs_nan(m, x[i], x[i + 1]);
      }
    }
  }
}

// The thread's max |v| from its running maxima. With the RHT the maxima are of
// |w| = 4 |v|: scaling the maximum once is exact (or monotone) and gives max |v|.
template <bool F32, bool RHT>
__device__ __forceinline__ float amax_result(float m, uint32_t m2) {
  if constexpr (!RHT && !F32) {
    m = fmaxf(fabsf(__uint_as_float(m2 << 16)), fabsf(__uint_as_float(m2 & 0xFFFF0000u)));
    if ((m2 & 0x7FFFu) > 0x7F80u || (m2 >> 16 & 0x7FFFu) > 0x7F80u) m = __uint_as_float(0x7FFFFFFFu);
  }
  return RHT ? __fmul_rn(m, 0.25f) : m;
}

// Quantise the thread's 32 elements at p (elements e .. e+31 of the copy) and
// add their statistics to the running sums.
template <int FMT, bool F32, bool RHT, bool SR, class Acc2>
__device__ __forceinline__ void quant_segment(const uint8_t* p, int64_t e, const Flat& f, const CopyOut& o,
                                              const uint32_t (&sgn)[16], const Ctx& cx, const Divider& dv,
                                              const float2* tab, const PhiloxKey& pk, Sums& acc, Acc2& kb,
                                              Acc2& ks, Acc2& ke, uint32_t& nonfinite) {
  const int nb16 = (f.n - e >= 32) ? 2 : (f.n - e >= 16 ? 1 : 0);
  if constexpr (FMT == 1) {
    if (nb16 == 2) {
      float bsum = 0.f, ssum = 0.f, esum = 0.f;
      f2 Q[16];
      load_block16<F32, RHT>(LinearSeg{p}, 0, sgn, Q);
      load_block16<F32, RHT>(LinearSeg{p}, F32 ? 4 : 2, sgn, Q + 8);
      uint32_t cw[4];
      const uint32_t sc = quant_block<FMT, SR, 16>(Q, cx, (uint64_t)e, pk, cw, bsum, ssum, esum,
                                                    acc, nonfinite);
      *reinterpret_cast<uint4*>(o.codes + e / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      put_scale<true>(o, f, (uint64_t)e / 32, sc);
      acc.bias.add(bsum);
    }
  } else if constexpr (FMT == 4 || FMT == 5) {
    // E8M0 scales on 16-element blocks
    float bsum = 0.f, ssum = 0.f, esum = 0.f;
    f2 Q[16];
    if (nb16 >= 1) load_block16<F32, RHT>(LinearSeg{p}, 0, sgn, Q);
    if (nb16 == 2) load_block16<F32, RHT>(LinearSeg{p}, F32 ? 4 : 2, sgn, Q + 8);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (h < nb16) {
        uint32_t cw[2];
        const uint32_t sc = quant_block<FMT, SR, 8>(Q + 8 * h, cx, (uint64_t)(e + 16 * h), pk, cw, bsum, ssum,
                                                     esum, acc, nonfinite);
        *reinterpret_cast<uint2*>(o.codes + (e + 16 * h) / 2) = make_uint2(cw[0], cw[1]);
        put_scale(o, f, (uint64_t)e / 16 + h, sc);
      }
    }
    acc.bias.add(bsum);
  } else if constexpr (FMT == 6) {
    // MBS-static ("Unveiling the Potential of Quantization with MXFP4 ...",
    // Resume technique §2B): the four threads of a 128-element macro block
    // (lanes 4k .. 4k+3; rows hold whole macro blocks) share its amax, which
    // sets the macro scale S (8 mantissa bits); the values are taken to units
    // of S (w = v * (1/S)) and quantised as 16-element E8M0 blocks. Every lane
    // takes part in the shuffles.
    f2 Q[16];
    float m = 0.f;
    if (nb16 == 2) {
      load_block16<F32, RHT>(LinearSeg{p}, 0, sgn, Q);
      load_block16<F32, RHT>(LinearSeg{p}, F32 ? 4 : 2, sgn, Q + 8);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float a, b;
        f2_split(Q[j], a, b);
        m = max3_abs_nan(m, a, b);
      }
    }
    m = max_abs_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max_abs_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    if (nb16 == 2) {
      const float S = mbs_macro_scale(m);
      float rs = (S == 0.f) ? 0.f : __frcp_rn(S);
      if (rs > FLT_MAX) rs = FLT_MAX;
      const f2 RS = f2_make(rs, rs);
#pragma unroll
      for (int j = 0; j < 16; ++j) Q[j] = f2_mul(Q[j], RS);
      float bsum = 0.f, ssum = 0.f, esum = 0.f;
      uint32_t cw[4];
      const uint32_t s0 = quant_block<FMT, SR, 8>(Q, cx, (uint64_t)e, pk, cw, bsum, ssum, esum, acc, nonfinite,
                                                   0u, S);
      const uint32_t s1 = quant_block<FMT, SR, 8>(Q + 8, cx, (uint64_t)e + 16, pk, cw + 2, bsum, ssum, esum, acc,
                                                   nonfinite, 0u, S);
      *reinterpret_cast<uint4*>(o.codes + e / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      put_scale(o, f, (uint64_t)e / 16, s0);
      put_scale(o, f, (uint64_t)e / 16 + 1, s1);
      acc.bias.add(bsum);
      if ((threadIdx.x & 3u) == 0u) o.tensor_scale[outer_index(o, f, e)] = S;
    }
  } else if constexpr (FMT == 7) {
    // HiF4: the two threads of a 64-element block are lanes 2k, 2k+1 (rows
    // hold whole blocks); every lane takes part in the shuffles
    f2 Q[16];
    if (nb16 == 2) {
      load_block16<F32, RHT>(LinearSeg{p}, 0, sgn, Q);
      load_block16<F32, RHT>(LinearSeg{p}, F32 ? 4 : 2, sgn, Q + 8);
    }
    uint32_t cw[4];
    const uint32_t w = hif4_half<SR>(Q, nb16 == 2, (uint64_t)e, pk, 0u, cw, acc, nonfinite);
    if (nb16 == 2) {
      *reinterpret_cast<uint4*>(o.codes + e / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      if ((threadIdx.x & 1u) == 0u) reinterpret_cast<uint32_t*>(o.scales)[(uint64_t)e >> 6] = w;
    }
  } else if constexpr (FMT == 3) {
    // Two-level NVFP4 (TetraJet-v2, Riepilogo Tecnico §2A): the four threads of
    // a 128-element outer block (lanes 4k .. 4k+3; rows hold whole outer
    // blocks) share its amax, which sets the block's own scale g_o in place
    // of the tensor scale. Every lane takes part in the shuffles.
    f2 Q[16];
    float m0 = 0.f, m1 = 0.f;
    if (nb16 == 2) {
      load_block16<F32, RHT>(LinearSeg{p}, 0, sgn, Q);
      load_block16<F32, RHT>(LinearSeg{p}, F32 ? 4 : 2, sgn, Q + 8);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float a, b;
        f2_split(Q[j], a, b);
        m0 = max3_abs_nan(m0, a, b);
        f2_split(Q[j + 8], a, b);
        m1 = max3_abs_nan(m1, a, b);
      }
    }
    float m = max_abs_nan(m0, m1);
    m = max_abs_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max_abs_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    if (nb16 == 2) {
      const Ctx co = make_ctx(__float_as_uint(m), 6.f, 2688.f);
      Divider dvo;
      dvo.init(co.d);
      uint32_t cw[4], sc[2];
      f2 b2 = 0ull, s2 = 0ull, e2 = 0ull;
      quant_two16_vals<0, SR, false>(Q, m0, m1, co, dvo, nullptr, (uint64_t)e, (uint64_t)e + 16, pk, 0u, cw, sc,
                                     b2, s2, e2, nonfinite);
      *reinterpret_cast<uint4*>(o.codes + e / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      put_scale(o, f, (uint64_t)e / 16, sc[0]);
      put_scale(o, f, (uint64_t)e / 16 + 1, sc[1]);
      float x0, x1, y0, y1;
      f2_split(b2, x0, x1);
      acc.bias.add(__fadd_rn(x0, x1));
      f2_split(s2, x0, x1);
      f2_split(e2, y0, y1);
      add_outer_stats(acc, co.g, __fadd_rn(x0, x1), __fadd_rn(y0, y1));
      if ((threadIdx.x & 3u) == 0u) o.tensor_scale[outer_index(o, f, e)] = co.g;
    }
  } else if (nb16 == 2) {
    uint32_t cw[4], sc[2];
    f2 b2 = 0ull, s2 = 0ull, e2 = 0ull;
    quant_two16<FMT, F32, RHT, SR>(LinearSeg{p}, sgn, cx, dv, tab, (uint64_t)e, pk, cw, sc, b2, s2, e2,
                                   nonfinite);
    *reinterpret_cast<uint4*>(o.codes + e / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    put_scale(o, f, (uint64_t)e / 16, sc[0]);
    put_scale(o, f, (uint64_t)e / 16 + 1, sc[1]);
    kb.add(b2);
    ks.add(s2);
    ke.add(e2);
  } else if (nb16 == 1) {
    // a lone 16-block at the very end of the copy
    float bsum = 0.f, ssum = 0.f, esum = 0.f;
    f2 Q[8];
    load_block16<F32, RHT>(LinearSeg{p}, 0, sgn, Q);
    uint32_t cw[2];
    const uint32_t sc = quant_block<FMT, SR, 8>(Q, cx, (uint64_t)e, pk, cw, bsum, ssum, esum,
                                                 acc, nonfinite);
    *reinterpret_cast<uint2*>(o.codes + e / 2) = make_uint2(cw[0], cw[1]);
    put_scale(o, f, (uint64_t)e / 16, sc);
    kb.add(f2_make(bsum, 0.f));
    ks.add(f2_make(ssum, 0.f));
    ke.add(f2_make(esum, 0.f));
  }
}

// ---- K1: tensor amax of the row-wise copy ----------------------------------------
template <bool F32, bool RHT>
__global__ void __launch_bounds__(RT, 2) amax_rows_kernel(Flat f, uint64_t seed, Workspace* ws,
                                                          uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[Ring<F32>::kStages], empty[Ring<F32>::kStages];
  __shared__ uint32_t sh_max[RT / 32];
  constexpr int S = Ring<F32>::kStages;
  const int tid = threadIdx.x;
  uint32_t sgn[16];
  make_sign_words<F32>(RHT ? rht_sign_mask(seed) : 0u, sgn);
  // chunks are visited from the end of the tensor, so that the quantisation
  // pass (which walks forward) starts on the chunks this pass left in L2
  FlatPipe pipe{full, empty, 0};
  flat_ring_start<F32>(f, ring, pipe, true);

  float m = 0.f;
  uint32_t m2 = 0u;      // BF16 pairs without the RHT
  bool timed_out = false;
  int64_t it = 0;
  for (int64_t c = blockIdx.x; c < f.nchunks; ++it, c += gridDim.x) {
    // the CTA's last chunk: the next kernel on the stream may start its prologue
    if (c + gridDim.x >= f.nchunks) grid_launch_dependents();
    const int s = (int)(it % S);
    if (!mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((it / S) & 1), timeout_ns)) {
      timed_out = true;
      break;
    }
    const int64_t e = (f.nchunks - 1 - c) * CH + (int64_t)tid * EPT;
    const int nb = (f.n - e >= 32) ? 2 : (f.n - e >= 16 ? 1 : 0);
    amax_segment<F32, RHT>(LinearSeg{ring + s * Ring<F32>::kChunkBytes + tid * EPT * (F32 ? 4 : 2)}, nb, sgn, m,
                           m2);
    if (!flat_ring_release<F32>(f, ring, pipe, it, c, true, timeout_ns)) {
      timed_out = true;
      break;
    }
  }
  grid_launch_dependents();     // a CTA that left the loop early
  // the workspace may still be read by the kernel before this one (its
  // quantisation pass): write only once that kernel has completed
  grid_dependency_wait();
  if (__syncthreads_or(timed_out)) {
    pipe_drain<S>(full, pipe.next_it);
    if (tid == 0) atomicOr(&ws->status, kStatusTimeout);
  }
  const uint32_t cm = cta_max<RT>(__float_as_uint(amax_result<F32, RHT>(m, m2)), sh_max);
  if (tid == 0) {
    ws->amax_part[0][blockIdx.x] = cm;
    ws->amax_part[1][blockIdx.x] = cm;
    if (blockIdx.x == 0) ws->amax_nparts = gridDim.x;
  }
}

// ---- K2: quantise the row-wise copy --------------------------------------------------
template <int FMT, bool F32, bool RHT, bool SR>
__global__ void __launch_bounds__(RT, SR ? 2 : 3) quant_rows_kernel(Flat f, uint64_t seed, PhiloxKey pk, CopyOut o,
                                                           Workspace* ws, uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[Ring<F32>::kStages], empty[Ring<F32>::kStages];
  __shared__ float2 tab[128];
  __shared__ double sh_sum[RT / 32];
  __shared__ float sh_f[3][RT / 32];
  __shared__ uint32_t sh_max[RT / 32];
  constexpr int S = Ring<F32>::kStages;
  constexpr int ES = F32 ? 4 : 2;
  constexpr float kQmax = (FMT == 2 || FMT == 7) ? 7.f : 6.f;
  constexpr float kQmax448 = (FMT == 2) ? 3136.f : 2688.f;
  const int tid = threadIdx.x;
  uint32_t sgn[16];
  make_sign_words<F32>(RHT ? rht_sign_mask(seed) : 0u, sgn);
  FlatPipe pipe{full, empty, 0};
  flat_ring_start<F32>(f, ring, pipe, false);     // the first copies fly while the scales are set up
  // Launched as a programmatic dependent of the amax pass: everything above
  // only reads the source; the amax partials are read after this wait.
  grid_dependency_wait();
  // The tensor scale's constants stay in shared memory and are read where
  // used: held in registers through the loop they made the kernel spill.
  __shared__ Ctx s_cx;
  __shared__ Divider s_dv;
  if (tid == 0) {
    s_cx = Ctx{1.f, 0.f, 0.f};
    s_dv = Divider{};
  }
  if constexpr (FMT == 0 || FMT == 2) {
    const Ctx c = make_ctx(fold_amax<RT>(ws, 0, sh_max), kQmax, kQmax448);
    if (tid == 0) {
      s_cx = c;
      s_dv.init(c.d);
    }
    fill_scale_table(tab, c.g);
  }
  __syncthreads();
  const Ctx& cx = s_cx;
  const Divider& dv = s_dv;

  Sums acc;
  Sum2 kb, ks, ke;
  uint32_t nonfinite = 0;
  bool timed_out = false;
  int64_t it = 0;
  // Warps run ahead of one another by up to kStages - 1 chunks, each
  // releasing a slot on its own (per-slot empty barriers, as the amax pass):
  // measured 6-7% faster than one CTA barrier per chunk on 8192 x 4096.
  for (int64_t c = blockIdx.x; c < f.nchunks; ++it, c += gridDim.x) {
    const int s = (int)(it % S);
    if (!mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((it / S) & 1), timeout_ns)) {
      timed_out = true;
      break;
    }
    const int64_t e = c * CH + (int64_t)tid * EPT;
    quant_segment<FMT, F32, RHT, SR>(ring + s * Ring<F32>::kChunkBytes + tid * EPT * ES, e, f, o, sgn, cx, dv,
                                     tab, pk, acc, kb, ks, ke, nonfinite);
    if (!flat_ring_release<F32>(f, ring, pipe, it, c, false, timeout_ns)) {
      timed_out = true;
      break;
    }
  }
  // the CTA's last chunk is done: the next kernel on the stream may start
  grid_launch_dependents();
  if (__syncthreads_or(timed_out)) {
    pipe_drain<S>(full, pipe.next_it);
    if (tid == 0) atomicOr(&ws->status, kStatusTimeout);
  }

  // ---- statistics: one partial per CTA (summed on the host by fp4q_stats) ----
  if (__syncthreads_or((int)nonfinite) && tid == 0) atomicOr(&ws->status, kStatusNonfinite);
  if constexpr (!kTensorScaled<FMT>) {   // FP64 sums (absolute units)
    double p[3] = {acc.bias.value(), acc.sig64, acc.err64};
    outer_stats_value(acc, p[1], p[2]);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const double v = cta_sum<RT>(p[k], sh_sum);
      if (tid == 0) ws->stat_part[0][k][blockIdx.x] = v;
    }
  } else {
    float v[3] = {kb.value_f(), ks.value_f(), ke.value_f()};
    cta_sums_f32<RT, 3>(v, sh_f);
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 3; ++k) ws->stat_part[0][k][blockIdx.x] = (double)v[k];
    }
  }
  if (blockIdx.x == 0 && tid == 0) {
    ws->stat_nparts = gridDim.x;
    ws->copies = 1u;
    ws->tensor_scale[0] = kTensorScaled<FMT> ? cx.g : 1.f;
    ws->qmax = kQmax;
    ws->n = (double)f.n;
    if (!kOuterScaled<FMT> && o.tensor_scale) *o.tensor_scale = kTensorScaled<FMT> ? cx.g : 1.f;
  }
}

// ---- requests with the transposed (column-wise) copy: tiles through a ring ------------
// The source is walked in 64 x 128 tiles. Warp 0 brings each tile into a ring
// slot with 2-D TMA loads, as boxes of 64 rows x 128 bytes (two per tile for
// BF16, four for FP32) written with the 128-byte swizzle: chunk c (16 bytes)
// of row r lands at chunk position c ^ (r & 7). With that layout both reading
// patterns are free of bank conflicts: the row-wise pass (each thread 32
// consecutive elements of one row, the 8 lanes of a quarter-warp on 8
// consecutive rows) and the column-wise pass (each thread two adjacent columns
// x 16 rows, a warp covering one 128-byte box row at a time). One read of the
// source serves both copies. Rows and cols are multiples of 16; TMA fills the
// parts of a box outside the tensor with zeros, which no thread reads.
constexpr int TTR = 64;     // tile rows
constexpr int TTC = 128;    // tile cols
constexpr int kBoxBytes = TTR * 128;

// TR: tile rows (64; 128 for the column-wise copies of the formats with a
// scale per 128 elements, whose outer blocks then run down a tile's columns).
template <bool F32, int TR = TTR>
struct TileRing {
  static constexpr int kBoxes = F32 ? 4 : 2;
  static constexpr int kBoxCols = F32 ? 32 : 64;
  static constexpr int kBoxBytes = TR * 128;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kStages = TR == TTR ? (F32 ? 3 : 4) : (F32 ? 2 : 3);
  static constexpr int kSmem = kStages * kTileBytes + 1024;    // + slack to align the ring to 1024
};

struct TileGeom {
  int64_t rows, cols;
  int64_t ntc;        // tiles along the columns
  int64_t ntiles;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// Lane 0 of warp 0 fills `slot` with tile t: the byte count (whole boxes, the
// zero fill included), then one load per box.
template <bool F32, int TR = TTR>
__device__ __forceinline__ void tile_issue(const CUtensorMap* map, const TileGeom& g, int64_t t, uint8_t* slot,
                                           uint32_t bar) {
  using TRg = TileRing<F32, TR>;
  if ((threadIdx.x & 31) != 0) return;
  const int32_t r0 = (int32_t)((t / g.ntc) * TR), c0 = (int32_t)((t % g.ntc) * TTC);
  mbar_arrive_expect_tx(bar, (uint32_t)TRg::kTileBytes);
#pragma unroll
  for (int b = 0; b < TRg::kBoxes; ++b)
    tma_load_2d(smem_u32(slot + b * TRg::kBoxBytes), map, bar, c0 + b * TRg::kBoxCols, r0);
}

// Ring protocol. full[s]: the slot's loads have landed (one arrival with the
// byte count, then the loads' transactions). empty[s]: every warp is done
// reading the slot (one arrival per warp). Warps run ahead of one another by
// up to kStages - 1 tiles; only warp 0, which refills the slots, waits for the
// slowest. Every wait is bounded.
struct TilePipe {
  uint64_t* full;
  uint64_t* empty;
  int64_t next_it;     // warp 0: the next iteration whose tile is to be issued
};

template <bool F32, int TR = TTR>
__device__ __forceinline__ void tile_ring_start(const CUtensorMap* map, const TileGeom& g, uint8_t* ring,
                                                TilePipe& p) {
  constexpr int S = TileRing<F32, TR>::kStages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&p.full[s]), 1);
      mbar_init(smem_u32(&p.empty[s]), RT / 32);
    }
    fence_mbarrier_init();
  }
  __syncthreads();
  p.next_it = 0;
  if (threadIdx.x < 32) {
    for (int s = 0; s < S; ++s) {
      const int64_t t = blockIdx.x + (int64_t)s * gridDim.x;
      if (t >= g.ntiles) break;
      tile_issue<F32, TR>(map, g, t, ring + s * TileRing<F32, TR>::kTileBytes, smem_u32(&p.full[s]));
      p.next_it = s + 1;
    }
  }
}

// The calling warp is done with iteration `it` (tile t). Warp 0 then waits for
// the other warps to be done with the slot too and refills it with the tile
// kStages iterations later. False if that wait ran out.
template <bool F32, int TR = TTR>
__device__ __forceinline__ bool tile_ring_release(const CUtensorMap* map, const TileGeom& g, uint8_t* ring,
                                                  TilePipe& p, int64_t it, int64_t t, uint64_t timeout_ns) {
  constexpr int S = TileRing<F32, TR>::kStages;
  const int s = (int)(it % S);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&p.empty[s]));
  if (threadIdx.x < 32) {
    const int64_t nx = t + (int64_t)S * gridDim.x;
    if (nx < g.ntiles) {
      if (!mbar_wait_bounded(smem_u32(&p.empty[s]), (uint32_t)((it / S) & 1), timeout_ns)) return false;
      tile_issue<F32, TR>(map, g, nx, ring + s * TileRing<F32, TR>::kTileBytes, smem_u32(&p.full[s]));
      p.next_it = it + S + 1;
    }
  }
  return true;
}

// The row-wise pass's thread layout: row r of the tile, 32-element segment
// `seg` of that row (a warp covers 8 rows; a quarter-warp, 8 rows at one seg).
__device__ __forceinline__ int tile_row_of(int tid) { return (tid & 7) + 8 * (tid >> 5); }
__device__ __forceinline__ int tile_seg_of(int tid) { return (tid >> 3) & 3; }

// The thread's row segment in a slot: its box and its chunks.
template <bool F32>
__device__ __forceinline__ SwzSeg tile_row_seg(const uint8_t* slot, int r, int seg) {
  const int box = F32 ? seg : (seg >> 1);
  const uint32_t first = F32 ? 0u : (uint32_t)(seg & 1) * 4u;
  return SwzSeg{slot + box * kBoxBytes + r * 128, 16u * (first ^ (uint32_t)(r & 7))};
}

// Byte offset, within a slot of TR-row tiles, of the byte at `b` (0 .. row
// bytes - 1) of tile row r, for r = r0 + i with r0 a multiple of 8.
template <int TR = TTR>
__device__ __forceinline__ uint32_t tile_byte(int r, uint32_t b, int i) {
  return (b >> 7) * (uint32_t)(TR * 128) + (uint32_t)r * 128u + ((b & 127u) ^ (16u * (uint32_t)(i & 7)));
}

// Two adjacent columns x 16 rows of a slot as FP32 (sign-flipped by sigma
// along the column when RHT): a[i] = column 2*pair, b[i] = column 2*pair+1.
template <bool F32, bool RHT, int TR = TTR>
__device__ __forceinline__ void load_col_pair(const uint8_t* slot, int row0, int pair, uint32_t smask,
                                              float (&a)[16], float (&b)[16]) {
  const uint32_t bo = (uint32_t)pair * (F32 ? 8u : 4u);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint8_t* q = slot + tile_byte<TR>(row0 + i, bo, i);
    const uint32_t sg = RHT ? (((smask >> i) & 1u) << 31) : 0u;
    if constexpr (F32) {
      const uint2 w = *reinterpret_cast<const uint2*>(q);
      a[i] = __uint_as_float(w.x ^ sg);
      b[i] = __uint_as_float(w.y ^ sg);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(q);
      a[i] = __uint_as_float((w << 16) ^ sg);
      b[i] = __uint_as_float((w & 0xFFFF0000u) ^ sg);
    }
  }
}

// One column x 32 rows (MXFP4 column blocks) as FP32 pairs of consecutive rows.
template <bool F32, bool RHT>
__device__ __forceinline__ void load_col32(const uint8_t* slot, int row0, int col, uint32_t smask, f2* Q) {
  const uint32_t bo = (uint32_t)col * (F32 ? 4u : 2u);
  float x[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint8_t* q = slot + tile_byte(row0 + i, bo, i);
    const uint32_t sg = RHT ? (((smask >> (i & 15)) & 1u) << 31) : 0u;
    if constexpr (F32) {
      x[i] = __uint_as_float(*reinterpret_cast<const uint32_t*>(q) ^ sg);
    } else {
      x[i] = __uint_as_float(((uint32_t)*reinterpret_cast<const uint16_t*>(q) << 16) ^ sg);
    }
  }
  if constexpr (RHT) {
    float h0[16], h1[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) { h0[i] = x[i]; h1[i] = x[i + 16]; }
    rht16_pairs(h0, Q);
    rht16_pairs(h1, Q + 8);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) Q[j] = f2_make(x[2 * j], x[2 * j + 1]);
  }
}

template <bool DUP = false>
__device__ __forceinline__ void put_scale_rk(const CopyOut& o, int64_t row, int64_t kb, uint32_t sc) {
  if (DUP && o.mma) {
    *reinterpret_cast<uint16_t*>(o.scales + mma_scale_offset(row, 2 * kb, o.nkb_p)) = (uint16_t)(sc | (sc << 8));
  } else {
    o.scales[o.mma ? mma_scale_offset(row, kb, o.nkb_p) : row * o.nkb + kb] = (uint8_t)sc;
  }
}

// 16 code bytes of one row of a copy. A row starts on an 8-byte boundary (its
// length is a multiple of 16 elements); the bytes go out as one 16-byte store
// where the address allows, else as two 8-byte stores.
__device__ __forceinline__ void store_codes16(uint8_t* p, const uint32_t (&cw)[4]) {
  if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
    *reinterpret_cast<uint4*>(p) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  } else {
    *reinterpret_cast<uint2*>(p) = make_uint2(cw[0], cw[1]);
    *reinterpret_cast<uint2*>(p + 8) = make_uint2(cw[2], cw[3]);
  }
}

// Per-copy state of the quantisation pass.
struct CopyState {
  Ctx cx;
  Divider dv;
  Sums acc;
  Kahan2 kb, ks, ke;
};

// ---- K1 for tiles: tensor amax of the row-wise and the column-wise copy (RHT) --------
template <bool F32, bool ROWS>
__global__ void __launch_bounds__(RT, 2) amax_tiles_kernel(const __grid_constant__ CUtensorMap tmap, TileGeom g,
                                                           uint64_t seed, Workspace* ws, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[TileRing<F32>::kStages], empty[TileRing<F32>::kStages];
  __shared__ uint32_t sh_max[RT / 32];
  constexpr int S = TileRing<F32>::kStages;
  uint8_t* ring = align1024(smem_raw);
  const int tid = threadIdx.x;
  const uint32_t smask = rht_sign_mask(seed);
  uint32_t sgn[16];
  make_sign_words<F32>(smask, sgn);
  TilePipe pipe{full, empty, 0};
  tile_ring_start<F32>(&tmap, g, ring, pipe);
  const int rr = tile_row_of(tid), seg = tile_seg_of(tid);   // row-wise pass
  const int pair = tid & 63, cb = tid >> 6;                    // column-wise pass
  float mr = 0.f, mc = 0.f;
  bool timed_out = false;
  int64_t it = 0;
  for (int64_t t = blockIdx.x; t < g.ntiles; ++it, t += gridDim.x) {
    // the CTA's last tile: the next kernel on the stream may start its prologue
    if (t + gridDim.x >= g.ntiles) grid_launch_dependents();
    const int s = (int)(it % S);
    if (!mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((it / S) & 1), timeout_ns)) {
      timed_out = true;
      break;
    }
    {
      const uint8_t* slot = ring + s * TileRing<F32>::kTileBytes;
      const int64_t r0 = (t / g.ntc) * TTR, c0 = (t % g.ntc) * TTC;
      const int vr = (int)min((int64_t)TTR, g.rows - r0), vc = (int)min((int64_t)TTC, g.cols - c0);
      if constexpr (ROWS) {
        if (rr < vr && 32 * seg < vc) {
          uint32_t m2 = 0u;
          amax_segment<F32, true>(tile_row_seg<F32>(slot, rr, seg), min(2, (vc - 32 * seg) / 16), sgn, mr, m2);
        }
      }
      if (16 * cb < vr && 2 * pair < vc) {
        float a[16], b[16];
        load_col_pair<F32, true>(slot, 16 * cb, pair, smask, a, b);
        rht16_unscaled(a);
        rht16_unscaled(b);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          mc = max3_abs_nan(mc, a[i], a[i + 1]);
          mc = max3_abs_nan(mc, b[i], b[i + 1]);
        }
      }
    }
    if (!tile_ring_release<F32>(&tmap, g, ring, pipe, it, t, timeout_ns)) {
      timed_out = true;
      break;
    }
  }
  grid_launch_dependents();     // a CTA that left the loop early
  // the workspace may still be read by the kernel before this one (its
  // quantisation pass): write only once that kernel has completed
  grid_dependency_wait();
  if (__syncthreads_or(timed_out)) {
    pipe_drain<TileRing<F32>::kStages>(pipe.full, pipe.next_it);
    if (tid == 0) atomicOr(&ws->status, kStatusTimeout);
  }
  // maxima of |w| = 4 |v|: one exact (or monotone) scaling gives max |v|
  const uint32_t cr = cta_max<RT>(__float_as_uint(__fmul_rn(mr, 0.25f)), sh_max);
  const uint32_t cc = cta_max<RT>(__float_as_uint(__fmul_rn(mc, 0.25f)), sh_max);
  if (tid == 0) {
    ws->amax_part[0][blockIdx.x] = cr;
    ws->amax_part[1][blockIdx.x] = cc;
    if (blockIdx.x == 0) ws->amax_nparts = gridDim.x;
  }
}

// ---- K2 for tiles: quantise the row-wise and/or the column-wise copy ------------------
template <int FMT, bool F32, bool RHT, bool SR, bool ROWS>
__global__ void __launch_bounds__(RT, 2) quant_tiles_kernel(const __grid_constant__ CUtensorMap tmap, TileGeom g,
                                                            uint64_t seed, PhiloxKey pk, CopyOut orow, CopyOut ocol,
                                                            Workspace* ws, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[TileRing<F32>::kStages], empty[TileRing<F32>::kStages];
  __shared__ float2 tab[2][128];
  __shared__ double sh_sum[RT / 32];
  __shared__ float sh_f[6][RT / 32];
  __shared__ uint32_t sh_max[RT / 32];
  constexpr int S = TileRing<F32>::kStages;
  constexpr float kQmax = (FMT == 2) ? 7.f : 6.f;
  constexpr float kQmax448 = (FMT == 2) ? 3136.f : 2688.f;
  uint8_t* ring = align1024(smem_raw);
  const int tid = threadIdx.x;
  const uint32_t smask = RHT ? rht_sign_mask(seed) : 0u;
  uint32_t sgn[16];
  make_sign_words<F32>(smask, sgn);
  TilePipe pipe{full, empty, 0};
  tile_ring_start<F32>(&tmap, g, ring, pipe);   // the first loads fly while the scales are set up
  // Launched as a programmatic dependent of the amax pass: everything above
  // only reads the source; the amax partials are read after this wait.
  grid_dependency_wait();
  CopyState cr, cc;
  cr.cx = Ctx{1.f, 0.f, 0.f};
  cc.cx = Ctx{1.f, 0.f, 0.f};
  cr.dv = Divider{};
  cc.dv = Divider{};
  if constexpr (kTensorScaled<FMT>) {
    if (ROWS) {
      cr.cx = make_ctx(fold_amax<RT>(ws, 0, sh_max), kQmax, kQmax448);
      cr.dv.init(cr.cx.d);
      fill_scale_table(tab[0], cr.cx.g);
    }
    cc.cx = make_ctx(fold_amax<RT>(ws, 1, sh_max), kQmax, kQmax448);
    cc.dv.init(cc.cx.d);
    fill_scale_table(tab[1], cc.cx.g);
    __syncthreads();
  }
  const int rr = tile_row_of(tid), seg = tile_seg_of(tid);
  uint32_t nonfinite = 0;
  bool timed_out = false;
  int64_t it = 0;
  for (int64_t t = blockIdx.x; t < g.ntiles; ++it, t += gridDim.x) {
    const int s = (int)(it % S);
    if (!mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((it / S) & 1), timeout_ns)) {
      timed_out = true;
      break;
    }
    {
      const uint8_t* slot = ring + s * TileRing<F32>::kTileBytes;
      const int64_t r0 = (t / g.ntc) * TTR, c0 = (t % g.ntc) * TTC;
      const int vr = (int)min((int64_t)TTR, g.rows - r0), vc = (int)min((int64_t)TTC, g.cols - c0);
      // ---- row-wise copy: 32 consecutive elements of one tile row per thread ----
      if constexpr (ROWS) {
        const int nb16 = (rr < vr) ? max(0, min(2, (vc - 32 * seg) / 16)) : 0;
        const SwzSeg sg = tile_row_seg<F32>(slot, rr, seg);
        const int64_t row = r0 + rr, col = c0 + 32 * seg;
        const int64_t e = row * g.cols + col;
        if constexpr (FMT == 1) {
          if (nb16 == 2) {
            float bsum = 0.f, ssum = 0.f, esum = 0.f;
            f2 Q[16];
            load_block16<F32, RHT>(sg, 0, sgn, Q);
            load_block16<F32, RHT>(sg, F32 ? 4 : 2, sgn, Q + 8);
            uint32_t cw[4];
            const uint32_t sc = quant_block<FMT, SR, 16>(Q, cr.cx, (uint64_t)e, pk, cw, bsum, ssum, esum,
                                                          cr.acc, nonfinite, 0u);
            store_codes16(orow.codes + row * orow.ld + col / 2, cw);
            put_scale_rk<true>(orow, row, col / 32, sc);
            cr.acc.bias.add(bsum);
          }
        } else if constexpr (FMT == 4 || FMT == 5) {
          float bsum = 0.f, ssum = 0.f, esum = 0.f;
          f2 Q[16];
          if (nb16 >= 1) load_block16<F32, RHT>(sg, 0, sgn, Q);
          if (nb16 == 2) load_block16<F32, RHT>(sg, F32 ? 4 : 2, sgn, Q + 8);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h < nb16) {
              uint32_t cw[2];
              const uint32_t sc = quant_block<FMT, SR, 8>(Q + 8 * h, cr.cx, (uint64_t)(e + 16 * h), pk, cw, bsum,
                                                           ssum, esum, cr.acc, nonfinite, 0u);
              *reinterpret_cast<uint2*>(orow.codes + row * orow.ld + col / 2 + 8 * h) = make_uint2(cw[0], cw[1]);
              put_scale_rk(orow, row, col / 16 + h, sc);
            }
          }
          cr.acc.bias.add(bsum);
        } else if (nb16 == 2) {
          uint32_t cw[4], sc[2];
          f2 b2 = 0ull, s2 = 0ull, e2 = 0ull;
          quant_two16<FMT, F32, RHT, SR>(sg, sgn, cr.cx, cr.dv, tab[0], (uint64_t)e, pk, cw, sc, b2, s2, e2,
                                         nonfinite);
          store_codes16(orow.codes + row * orow.ld + col / 2, cw);
          put_scale_rk(orow, row, col / 16, sc[0]);
          put_scale_rk(orow, row, col / 16 + 1, sc[1]);
          cr.kb.add(b2);
          cr.ks.add(s2);
          cr.ke.add(e2);
        } else if (nb16 == 1) {
          float bsum = 0.f, ssum = 0.f, esum = 0.f;
          f2 Q[8];
          load_block16<F32, RHT>(sg, 0, sgn, Q);
          uint32_t cw[2];
          const uint32_t sc = quant_block<FMT, SR, 8>(Q, cr.cx, (uint64_t)e, pk, cw, bsum, ssum, esum,
                                                       cr.acc, nonfinite, 0u);
          *reinterpret_cast<uint2*>(orow.codes + row * orow.ld + col / 2) = make_uint2(cw[0], cw[1]);
          put_scale_rk(orow, row, col / 16, sc);
          cr.kb.add(f2_make(bsum, 0.f));
          cr.ks.add(f2_make(ssum, 0.f));
          cr.ke.add(f2_make(esum, 0.f));
        }
      }
      // ---- column-wise copy: blocks run down the columns; copy row = source column ----
      if constexpr (FMT == 1) {
        const int col = tid & 127, cb = tid >> 7;        // one column x 32 rows
        if (32 * cb < vr && col < vc) {
          float bsum = 0.f, ssum = 0.f, esum = 0.f;
          f2 Q[16];
          load_col32<F32, RHT>(slot, 32 * cb, col, smask, Q);
          const int64_t crow = c0 + col, ccol = r0 + 32 * cb;
          uint32_t cw[4];
          const uint32_t sc = quant_block<FMT, SR, 16>(Q, cc.cx, (uint64_t)(crow * g.rows + ccol), pk, cw,
                                                        bsum, ssum, esum, cc.acc, nonfinite, 1u);
          *reinterpret_cast<uint4*>(ocol.codes + crow * ocol.ld + ccol / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
          put_scale_rk<true>(ocol, crow, ccol / 32, sc);
          cc.acc.bias.add(bsum);
        }
      } else if constexpr (FMT == 4 || FMT == 5) {
        const int pair = tid & 63, cb = tid >> 6;         // two columns x 16 rows, a block each
        if (16 * cb < vr && 2 * pair < vc) {
          float a[16], b[16];
          load_col_pair<F32, RHT>(slot, 16 * cb, pair, smask, a, b);
          f2 Q[16];
          if constexpr (RHT) {
            rht16_pairs(a, Q);
            rht16_pairs(b, Q + 8);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              Q[j] = f2_make(a[2 * j], a[2 * j + 1]);
              Q[j + 8] = f2_make(b[2 * j], b[2 * j + 1]);
            }
          }
          const int64_t ca = c0 + 2 * pair, rw = r0 + 16 * cb;
          float bsum = 0.f, ssum = 0.f, esum = 0.f;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t cw[2];
            const uint32_t sc = quant_block<FMT, SR, 8>(Q + 8 * h, cc.cx, (uint64_t)((ca + h) * g.rows + rw), pk,
                                                         cw, bsum, ssum, esum, cc.acc, nonfinite, 1u);
            *reinterpret_cast<uint2*>(ocol.codes + (ca + h) * ocol.ld + rw / 2) = make_uint2(cw[0], cw[1]);
            put_scale_rk(ocol, ca + h, rw / 16, sc);
          }
          cc.acc.bias.add(bsum);
        }
      } else {
        const int pair = tid & 63, cb = tid >> 6;         // two columns x 16 rows
        if (16 * cb < vr && 2 * pair < vc) {
          float a[16], b[16];
          load_col_pair<F32, RHT>(slot, 16 * cb, pair, smask, a, b);
          f2 Q[16];
          float m0 = 0.f, m1 = 0.f;
          if constexpr (RHT) {
            rht16_pairs(a, Q);
            rht16_pairs(b, Q + 8);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              Q[j] = f2_make(a[2 * j], a[2 * j + 1]);
              Q[j + 8] = f2_make(b[2 * j], b[2 * j + 1]);
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float x0, x1;
            f2_split(Q[j], x0, x1);
            m0 = max3_abs_nan(m0, x0, x1);
            f2_split(Q[j + 8], x0, x1);
            m1 = max3_abs_nan(m1, x0, x1);
          }
          const int64_t ca = c0 + 2 * pair, rw = r0 + 16 * cb;
          uint32_t cw[4], sc[2];
          f2 b2 = 0ull, s2 = 0ull, e2 = 0ull;
          quant_two16_vals<FMT, SR>(Q, m0, m1, cc.cx, cc.dv, tab[1], (uint64_t)(ca * g.rows + rw),
                                    (uint64_t)((ca + 1) * g.rows + rw), pk, 1u, cw, sc, b2, s2, e2, nonfinite);
          *reinterpret_cast<uint2*>(ocol.codes + ca * ocol.ld + rw / 2) = make_uint2(cw[0], cw[1]);
          *reinterpret_cast<uint2*>(ocol.codes + (ca + 1) * ocol.ld + rw / 2) = make_uint2(cw[2], cw[3]);
          put_scale_rk(ocol, ca, rw / 16, sc[0]);
          put_scale_rk(ocol, ca + 1, rw / 16, sc[1]);
          cc.kb.add(b2);
          cc.ks.add(s2);
          cc.ke.add(e2);
        }
      }
    }
    if (!tile_ring_release<F32>(&tmap, g, ring, pipe, it, t, timeout_ns)) {
      timed_out = true;
      break;
    }
  }
  // the CTA's last tile is done: the next kernel on the stream may start
  grid_launch_dependents();
  if (__syncthreads_or(timed_out)) {
    pipe_drain<TileRing<F32>::kStages>(pipe.full, pipe.next_it);
    if (tid == 0) atomicOr(&ws->status, kStatusTimeout);
  }

  // ---- statistics: one partial per CTA and copy (summed on the host) ----
  if (__syncthreads_or((int)nonfinite) && tid == 0) atomicOr(&ws->status, kStatusNonfinite);
  if constexpr (kE8M0<FMT>) {
    double p[2][3] = {{cr.acc.bias.value(), cr.acc.sig64, cr.acc.err64},
                      {cc.acc.bias.value(), cc.acc.sig64, cc.acc.err64}};
    outer_stats_value(cr.acc, p[0][1], p[0][2]);
    outer_stats_value(cc.acc, p[1][1], p[1][2]);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const double v = cta_sum<RT>(p[c][k], sh_sum);
        if (tid == 0) ws->stat_part[c][k][blockIdx.x] = v;
      }
    }
  } else {
    float v[6] = {cr.kb.value_f(), cr.ks.value_f(), cr.ke.value_f(),
                  cc.kb.value_f(), cc.ks.value_f(), cc.ke.value_f()};
    cta_sums_f32<RT, 6>(v, sh_f);
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 6; ++k) ws->stat_part[k / 3][k % 3][blockIdx.x] = (double)v[k];
    }
  }
  if (blockIdx.x == 0 && tid == 0) {
    ws->stat_nparts = gridDim.x;
    ws->copies = (ROWS ? 1u : 0u) | 2u;
    ws->tensor_scale[0] = kE8M0<FMT> ? 1.f : cr.cx.g;
    ws->tensor_scale[1] = kE8M0<FMT> ? 1.f : cc.cx.g;
    ws->qmax = kQmax;
    ws->n = (double)g.rows * (double)g.cols;
    if (ROWS && orow.tensor_scale) *orow.tensor_scale = kE8M0<FMT> ? 1.f : cr.cx.g;
    if (ocol.tensor_scale) *ocol.tensor_scale = kE8M0<FMT> ? 1.f : cc.cx.g;
  }
}

// ---- the column-wise copy of the formats with a scale per 128 elements -----------------
// Two-level NVFP4 ("TetraJet-v2 ...", Riepilogo Tecnico §2A: the transposed
// copy for the weight gradient, the double-block scale) and MBS-static
// ("Unveiling the Potential of Quantization with MXFP4 ...", Resume technique
// §2B): in the column-wise copy the 16-element blocks and the 128-element outer
// (macro) blocks run down the source's columns. The source is walked in
// 128 x 128 tiles, so each tile column holds exactly one outer block. Thread t
// takes the column pair p = t / 4 (columns 2p, 2p + 1) and the quarter q = t % 4
// (rows 32q .. 32q + 31: two 16-row blocks per column); the four quarters of a
// pair are lanes 4k .. 4k + 3, which share the outer maxima by two shuffles.
// Each column then has its own outer scale, so its blocks go through
// quant_block one at a time. Rows are a multiple of 128 (whole outer blocks);
// the row-wise copy, when requested too, comes from the row kernel.
constexpr int TOR = 128;    // tile rows of this pass

template <int FMT, bool F32, bool RHT, bool SR>
__global__ void __launch_bounds__(RT, F32 ? 1 : 2) quant_cols_outer_kernel(
    const __grid_constant__ CUtensorMap tmap, TileGeom g, uint64_t seed, PhiloxKey pk, CopyOut ocol,
    Workspace* ws, uint64_t timeout_ns, int row_nparts) {
  static_assert(kOuterScaled<FMT> || FMT == 7, "formats with a scale per 128 elements, or HiF4");
  using TRg = TileRing<F32, TOR>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[TRg::kStages], empty[TRg::kStages];
  __shared__ double sh_sum[RT / 32];
  constexpr int S = TRg::kStages;
  uint8_t* ring = align1024(smem_raw);
  const int tid = threadIdx.x;
  const uint32_t smask = RHT ? rht_sign_mask(seed) : 0u;
  TilePipe pipe{full, empty, 0};
  tile_ring_start<F32, TOR>(&tmap, g, ring, pipe);
  grid_dependency_wait();      // the workspace's statistics slots may still be read before this
  const int pair = tid >> 2, qr = tid & 3;
  const Ctx unit{1.f, 0.f, 0.f};
  Sums acc;
  uint32_t nonfinite = 0;
  bool timed_out = false;
  int64_t it = 0;
  for (int64_t t = blockIdx.x; t < g.ntiles; ++it, t += gridDim.x) {
    const int s = (int)(it % S);
    if (!mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((it / S) & 1), timeout_ns)) {
      timed_out = true;
      break;
    }
    {
      const uint8_t* slot = ring + s * TRg::kTileBytes;
      const int64_t r0 = (t / g.ntc) * TOR, c0 = (t % g.ntc) * TTC;
      const int vc = (int)min((int64_t)TTC, g.cols - c0);
      const bool valid = 2 * pair < vc;       // vc is a multiple of 16: pairs are whole
      // the two 16-row blocks of each column of the pair, transformed
      f2 Qa[2][8], Qb[2][8];
      float ma[2] = {0.f, 0.f}, mb[2] = {0.f, 0.f};
      if (valid) {
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
          float a[16], b[16];
          load_col_pair<F32, RHT, TOR>(slot, 32 * qr + 16 * gi, pair, smask, a, b);
          if constexpr (RHT) {
            rht16_pairs(a, Qa[gi]);
            rht16_pairs(b, Qb[gi]);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              Qa[gi][j] = f2_make(a[2 * j], a[2 * j + 1]);
              Qb[gi][j] = f2_make(b[2 * j], b[2 * j + 1]);
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float x0, x1;
            f2_split(Qa[gi][j], x0, x1);
            ma[gi] = max3_abs_nan(ma[gi], x0, x1);
            f2_split(Qb[gi][j], x0, x1);
            mb[gi] = max3_abs_nan(mb[gi], x0, x1);
          }
        }
      }
      if constexpr (FMT == 7) {
        // HiF4: a 64-row block of a column is held by the threads qr = 2k,
        // 2k + 1 (lanes differing in bit 0); rows are whole 64-row blocks, so
        // the block is in the tensor for both or for neither
        const bool in = valid && r0 + 32 * qr < g.rows;
#pragma unroll
        for (int k = 0; k < 2; ++k) {           // column 2p + k: one row of the copy
          const f2 (&Q)[16] = *reinterpret_cast<const f2(*)[16]>(k ? &Qb[0][0] : &Qa[0][0]);
          const int64_t crow = c0 + 2 * pair + k, ccol = r0 + 32 * qr;
          uint32_t cw[4];
          const uint32_t w = hif4_half<SR>(Q, in, (uint64_t)(crow * g.rows + ccol), pk, 1u, cw, acc, nonfinite);
          if (in) {
            *reinterpret_cast<uint4*>(ocol.codes + crow * ocol.ld + ccol / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            if ((qr & 1) == 0) reinterpret_cast<uint32_t*>(ocol.scales)[crow * (g.rows / 64) + ccol / 64] = w;
          }
        }
      } else {
      // outer maxima of both columns over the pair's four quarters (every lane shuffles)
      float Ma = max_abs_nan(ma[0], ma[1]), Mb = max_abs_nan(mb[0], mb[1]);
      Ma = max_abs_nan(Ma, __shfl_xor_sync(0xFFFFFFFFu, Ma, 1));
      Ma = max_abs_nan(Ma, __shfl_xor_sync(0xFFFFFFFFu, Ma, 2));
      Mb = max_abs_nan(Mb, __shfl_xor_sync(0xFFFFFFFFu, Mb, 1));
      Mb = max_abs_nan(Mb, __shfl_xor_sync(0xFFFFFFFFu, Mb, 2));
      if (valid) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {           // column 2p + k: one row of the copy
          f2 (*Q)[8] = k ? Qb : Qa;
          const float M = k ? Mb : Ma;
          const int64_t crow = c0 + 2 * pair + k, ccol = r0 + 32 * qr;
          uint32_t cw[4];
          float bsum = 0.f, ssum = 0.f, esum = 0.f;
          float outer;
          if constexpr (FMT == 3) {
            // the outer block's own scale g_o in place of the tensor scale
            const Ctx co = make_ctx(__float_as_uint(M), 6.f, 2688.f);
#pragma unroll
            for (int gi = 0; gi < 2; ++gi) {
              const uint32_t sc = quant_block<0, SR, 8>(Q[gi], co, (uint64_t)(crow * g.rows + ccol + 16 * gi), pk,
                                                        cw + 2 * gi, bsum, ssum, esum, acc, nonfinite, 1u);
              put_scale_rk(ocol, crow, ccol / 16 + gi, sc);
            }
            add_outer_stats(acc, co.g, ssum, esum);
            outer = co.g;
          } else {
            // MBS: values in units of the macro scale S, then E8M0 blocks
            const float Sm = mbs_macro_scale(M);
            float rs = (Sm == 0.f) ? 0.f : __frcp_rn(Sm);
            if (rs > FLT_MAX) rs = FLT_MAX;
            const f2 RS = f2_make(rs, rs);
#pragma unroll
            for (int gi = 0; gi < 2; ++gi) {
#pragma unroll
              for (int j = 0; j < 8; ++j) Q[gi][j] = f2_mul(Q[gi][j], RS);
              const uint32_t sc = quant_block<6, SR, 8>(Q[gi], unit, (uint64_t)(crow * g.rows + ccol + 16 * gi), pk,
                                                        cw + 2 * gi, bsum, ssum, esum, acc, nonfinite, 1u, Sm);
              put_scale_rk(ocol, crow, ccol / 16 + gi, sc);
            }
            outer = Sm;
          }
          acc.bias.add(bsum);
          *reinterpret_cast<uint4*>(ocol.codes + crow * ocol.ld + ccol / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
          if (qr == 0) {
            const int64_t kc = r0 / 128;       // the outer block along the copy's row
            ocol.tensor_scale[ocol.mma ? kc * ocol.rows + crow : crow * (g.rows / 128) + kc] = outer;
          }
        }
      }
      }
    }
    if (!tile_ring_release<F32, TOR>(&tmap, g, ring, pipe, it, t, timeout_ns)) {
      timed_out = true;
      break;
    }
  }
  grid_launch_dependents();
  if (__syncthreads_or(timed_out)) {
    pipe_drain<S>(pipe.full, pipe.next_it);
    if (tid == 0) atomicOr(&ws->status, kStatusTimeout);
  }
  // ---- statistics of the column-wise copy: one partial per CTA ----
  if (__syncthreads_or((int)nonfinite) && tid == 0) atomicOr(&ws->status, kStatusNonfinite);
  double p[3] = {acc.bias.value(), acc.sig64, acc.err64};
  outer_stats_value(acc, p[1], p[2]);
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const double v = cta_sum<RT>(p[k], sh_sum);
    if (tid == 0) ws->stat_part[1][k][blockIdx.x] = v;
  }
  // The statistics header covers both copies: when the row kernel ran before
  // this one (row_nparts CTAs), each copy's partials past its own grid are zero.
  const int np = max((int)gridDim.x, row_nparts);
  if (blockIdx.x == 0) {
    for (int i = tid; i < np; i += RT) {
      if (i >= (int)gridDim.x) {
#pragma unroll
        for (int k = 0; k < 3; ++k) ws->stat_part[1][k][i] = 0.0;
      }
      if (row_nparts > 0 && i >= row_nparts) {
#pragma unroll
        for (int k = 0; k < 3; ++k) ws->stat_part[0][k][i] = 0.0;
      }
    }
    if (tid == 0) {
      ws->stat_nparts = (unsigned)np;
      ws->copies = (row_nparts > 0 ? 1u : 0u) | 2u;
      ws->tensor_scale[1] = 1.f;
      ws->qmax = FMT == 7 ? 7.f : 6.f;
      ws->n = (double)g.rows * (double)g.cols;
      if (FMT == 7 && ocol.tensor_scale) *ocol.tensor_scale = 1.f;
    }
  }
}

// ---- one launch for both passes (NVFP4 / UFP4 row-wise) ------------------------------
// A cooperatively launched (co-resident) grid streams its chunks twice through
// one ring: the amax pass, a grid barrier, the fold of the per-CTA maxima, then
// the quantisation pass. The ring runs on across the barrier, so the second
// pass's first chunks are already in flight while the first pass finishes.
template <int FMT, bool F32, bool RHT, bool SR>
__global__ void __launch_bounds__(RT, SR ? 2 : 3) quant_fused_kernel(Flat f, uint64_t seed, PhiloxKey pk, CopyOut o,
                                                                     Workspace* ws, uint64_t timeout_ns) {
  static_assert(FMT != 1, "MXFP4 has no tensor amax");
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[Ring<F32>::kStages];
  __shared__ float2 tab[128];
  __shared__ float sh_f[3][RT / 32];
  __shared__ uint32_t sh_max[RT / 32];
  constexpr int S = Ring<F32>::kStages;
  constexpr int ES = F32 ? 4 : 2;
  constexpr float kQmax = (FMT == 2) ? 7.f : 6.f;
  constexpr float kQmax448 = (FMT == 2) ? 3136.f : 2688.f;
  const int tid = threadIdx.x;
  uint32_t sgn[16];
  make_sign_words<F32>(RHT ? rht_sign_mask(seed) : 0u, sgn);
  // this CTA's chunks: bid, bid + grid, ...; visited once per pass
  const int64_t n1 = (f.nchunks - (int64_t)blockIdx.x + gridDim.x - 1) / gridDim.x;
  const int64_t total = 2 * n1;
  auto chunk_of = [&](int64_t it) { return (int64_t)blockIdx.x + (it < n1 ? it : it - n1) * gridDim.x; };
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < S && s < total; ++s) ring_issue<F32>(f, chunk_of(s), ring, s, smem_u32(&full[s]));
  }

  bool timed_out = false;
  int64_t it = 0;
  // ---- pass 1: tensor amax ----
  float m = 0.f;
  uint32_t m2 = 0u;
  for (; it < n1; ++it) {
    const int s = (int)(it % S);
    const bool ok = mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((it / S) & 1), timeout_ns);
    if (ok) {
      const int64_t e = chunk_of(it) * CH + (int64_t)tid * EPT;
      const int nb = (f.n - e >= 32) ? 2 : (f.n - e >= 16 ? 1 : 0);
      amax_segment<F32, RHT>(LinearSeg{ring + s * Ring<F32>::kChunkBytes + tid * EPT * ES}, nb, sgn, m, m2);
    }
    timed_out = __syncthreads_or(!ok);
    if (timed_out) break;
    if (tid == 0 && it + S < total) ring_issue<F32>(f, chunk_of(it + S), ring, s, smem_u32(&full[s]));
  }

  Sums acc;
  Sum2 kb, ks, ke;      // plain sums: see Sum2 (compensation made the kernel spill)
  uint32_t nonfinite = 0;
  // the tensor scale's constants in shared memory, read where used (see quant_rows_kernel)
  __shared__ Ctx s_cx;
  __shared__ Divider s_dv;
  if (tid == 0) s_cx = Ctx{1.f, 0.f, 0.f};
  if (!timed_out) {
    const uint32_t cm = cta_max<RT>(__float_as_uint(amax_result<F32, RHT>(m, m2)), sh_max);
    if (tid == 0) {
      ws->amax_part[0][blockIdx.x] = cm;
      ws->amax_part[1][blockIdx.x] = cm;
      if (blockIdx.x == 0) ws->amax_nparts = gridDim.x;
    }
    timed_out = !grid_barrier(ws, timeout_ns);
  }
  if (!timed_out) {
    const Ctx c = make_ctx(fold_amax<RT>(ws, 0, sh_max), kQmax, kQmax448);
    if (tid == 0) {
      s_cx = c;
      s_dv.init(c.d);
    }
    fill_scale_table(tab, c.g);
    __syncthreads();
    const Ctx& cx = s_cx;
    const Divider& dv = s_dv;
    // ---- pass 2: quantise ----
    for (; it < total; ++it) {
      const int s = (int)(it % S);
      const bool ok = mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((it / S) & 1), timeout_ns);
      if (ok) {
        const int64_t e = chunk_of(it) * CH + (int64_t)tid * EPT;
        quant_segment<FMT, F32, RHT, SR>(ring + s * Ring<F32>::kChunkBytes + tid * EPT * ES, e, f, o, sgn, cx,
                                         dv, tab, pk, acc, kb, ks, ke, nonfinite);
      }
      timed_out = __syncthreads_or(!ok);
      if (timed_out) break;
      if (tid == 0 && it + S < total) ring_issue<F32>(f, chunk_of(it + S), ring, s, smem_u32(&full[s]));
    }
  }
  if (timed_out) {
    // let the copies still in flight land before the CTA exits
    if (tid == 0) {
      const uint64_t t0 = globaltimer();
      for (int64_t j = it; j < it + S && j < total; ++j) {
        const uint32_t bar = smem_u32(&full[j % S]);
        while (!mbar_try_wait(bar, (uint32_t)((j / S) & 1)) && globaltimer() - t0 < 50000000ull) {
        }
      }
      atomicOr(&ws->status, kStatusTimeout);
    }
  }

  // ---- statistics: one partial per CTA (summed on the host by fp4q_stats) ----
  if (__syncthreads_or((int)nonfinite) && tid == 0) atomicOr(&ws->status, kStatusNonfinite);
  float v[3] = {kb.value_f(), ks.value_f(), ke.value_f()};
  cta_sums_f32<RT, 3>(v, sh_f);
  if (tid == 0) {
#pragma unroll
    for (int k = 0; k < 3; ++k) ws->stat_part[0][k][blockIdx.x] = (double)v[k];
  }
  if (blockIdx.x == 0 && tid == 0) {
    ws->stat_nparts = gridDim.x;
    ws->copies = 1u;
    ws->tensor_scale[0] = s_cx.g;
    ws->qmax = kQmax;
    ws->n = (double)f.n;
    if (o.tensor_scale) *o.tensor_scale = s_cx.g;
  }
}

// ---- dequantisation of a row-wise copy -------------------------------------------------
// v_hat = (level * s_b) * g (MXFP4: level * 2^e_b), two round-to-nearest
// products in that order; optionally the inverse transform (1/4) diag(sigma)
// H16 on every 16-block: butterfly stages 1, 2, 4, 8, then * 1/4, then the sign
// flip. A thread converts 32 consecutive elements (one 16-byte load of codes),
// grid-stride over the copy.

// Two signed levels of one code byte (bits 0-3 -> lo, bits 4-7 -> hi) as FP32.
template <int FMT>
__device__ __forceinline__ void levels2(uint32_t byte, float& lo, float& hi) {
  if constexpr (FMT == 2) {   // UFP4: integer levels, via the 2^23 offset trick (exact)
    const uint32_t l = byte & 0xFu, h = (byte >> 4) & 0xFu;
    const f2 m = f2_sub(f2_make(__uint_as_float(0x4B000000u | (l & 7u)), __uint_as_float(0x4B000000u | (h & 7u))),
                        f2_make(8388608.f, 8388608.f));
    float a, b;
    f2_split(m, a, b);
    lo = __uint_as_float(__float_as_uint(a) ^ ((l & 8u) << 28));
    hi = __uint_as_float(__float_as_uint(b) ^ ((h & 8u) << 28));
  } else {                    // E2M1 through the hardware conversion (exact in FP16)
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
    lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
    hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
  }
}

template <int FMT>
__device__ __forceinline__ float block_scale_value(uint32_t sc) {
  if constexpr (kE8M0<FMT>) {   // E8M0: 2^(sc - 127); code 0 is 2^-127 (subnormal)
    return sc ? __uint_as_float(sc << 23) : __uint_as_float(0x00400000u);
  } else {
    return e4m3_to_f32(sc);
  }
}

// 16 dequantised values to `out` (BF16 or FP32), after R^T when IRHT.
template <bool OUT_F32, bool IRHT>
__device__ __forceinline__ void store16(float (&v)[16], const uint32_t (&sgn)[16], void* out) {
  if constexpr (IRHT) {
    // R^T = (1/4) diag(sigma) H16: the forward butterfly (stages 1, 2, 4, 8, then
    // * 1/4) without its sign flip, then the sign flip
    f2 Q[8];
    rht16_pairs(v, Q);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float a, b;
      f2_split(Q[j], a, b);
      v[2 * j] = __uint_as_float(__float_as_uint(a) ^ sgn[2 * j]);
      v[2 * j + 1] = __uint_as_float(__float_as_uint(b) ^ sgn[2 * j + 1]);
    }
  }
  if constexpr (OUT_F32) {
    float4* o = reinterpret_cast<float4*>(out);
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  } else {
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
      h[k] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    uint4* o = reinterpret_cast<uint4*>(out);
    o[0] = make_uint4(h[0], h[1], h[2], h[3]);
    o[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// Byte b of x in the low byte and its sign bit replicated over the high byte
// (prmt, default mode: a selector nibble with bit 3 set copies the sign of the
// byte it names into every bit).
__device__ __forceinline__ uint32_t prmt_sign(uint32_t x, uint32_t b) {
  uint32_t d;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(x), "r"(b | ((8u | b) << 12)));
  return d;
}

// Dequantise one 16-block: `w0`, `w1` its code words, `sv` its scale value.
// Writes 16 values at `out` (BF16 or FP32).
template <int FMT, bool OUT_F32, bool IRHT>
__device__ __forceinline__ void deq16(uint32_t w0, uint32_t w1, float sv, float g, const uint32_t (&sgn)[16],
                                      void* out) {
  float v[16];
  const f2 G = f2_make(g, g);
  if constexpr (FMT == 2 && !OUT_F32) {
    // UFP4 to BF16 without per-nibble extraction: one prmt puts a code's magnitude
    // (bits 4-6 of a byte of w << 4 for the low code, of w for the high one)
    // into the low byte and its sign, replicated, into the high byte; the
    // magnitude under the FP32 pattern of 2^23 gives 2^23 + 16 k, and
    // fma(2^23 + 16 k, s / 16, -2^19 s) = k s exactly (k s has at most 7
    // significant bits; s / 16 and 2^19 s are exact for every E4M3 value).
    // The sign goes on afterwards, so code 8 still gives -0. Measured on the
    // 8192 x 4096 activation with the inverse RHT: 24.7 against 26.0 us; the
    // FP32 output kept the look-up path (71.7 against 79.9 us this way).
    const f2 S16 = f2_make(__fmul_rn(sv, 0.0625f), __fmul_rn(sv, 0.0625f));
    const f2 C = f2_make(__fmul_rn(sv, -524288.f), __fmul_rn(sv, -524288.f));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t w = j < 4 ? w0 : w1, b = (uint32_t)(j & 3);
      const uint32_t xl = prmt_sign(w << 4, b), xh = prmt_sign(w, b);
      const f2 A = f2_make(__uint_as_float((xl & 0x70u) | 0x4B000000u), __uint_as_float((xh & 0x70u) | 0x4B000000u));
      float r0, r1;
      f2_split(f2_mul(f2_fma(A, S16, C), G), r0, r1);
      v[2 * j] = __uint_as_float(__float_as_uint(r0) ^ (xl & 0x80000000u));
      v[2 * j + 1] = __uint_as_float(__float_as_uint(r1) ^ (xh & 0x80000000u));
    }
  } else {
    float q[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) levels2<FMT>(((j < 4 ? w0 : w1) >> (8 * (j & 3))) & 0xFFu, q[2 * j], q[2 * j + 1]);
    const f2 S = f2_make(sv, sv);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      f2 r = f2_mul(f2_make(q[2 * j], q[2 * j + 1]), S);
      if (FMT != 1 && FMT != 4 && FMT != 5) r = f2_mul(r, G);
      f2_split(r, v[2 * j], v[2 * j + 1]);
    }
  }
  store16<OUT_F32, IRHT>(v, sgn, out);
}

// Value of a HiF4 E6M2 scale code (bias 31; exponent field 0 is subnormal).
__device__ __forceinline__ float e6m2_value(uint32_t c) {
  const uint32_t E = c >> 2, m = c & 3u;
  return E ? __uint_as_float(((E + 96u) << 23) | (m << 21)) : __fmul_rn((float)m, 2.3283064365386963e-10f);
}

// Dequantise 16 HiF4 elements, the `hb`-th 16 (0..3) of the block whose scale
// word is `word`: level * S * 2^-(d_8 + d_4) per 4-element micro-block, exact
// in FP32 (at most 6 significant bits, exponent within range).
template <bool OUT_F32, bool IRHT>
__device__ __forceinline__ void deq16_hif4(uint32_t w0, uint32_t w1, uint32_t word, int hb,
                                           const uint32_t (&sgn)[16], void* out) {
  float q[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) levels2<2>(((j < 4 ? w0 : w1) >> (8 * (j & 3))) & 0xFFu, q[2 * j], q[2 * j + 1]);
  const float S = e6m2_value(word & 0xFFu);
  float v[16];
#pragma unroll
  for (int qd = 0; qd < 4; ++qd) {
    const int i = 4 * hb + qd;                       // micro-block in the block
    const uint32_t sh = ((word >> (8 + (i >> 1))) & 1u) + ((word >> (16 + i)) & 1u);
    const float st = __fmul_rn(S, __uint_as_float((127u - sh) << 23));
    const f2 ST = f2_make(st, st);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int j = 2 * qd + t;
      f2_split(f2_mul(f2_make(q[2 * j], q[2 * j + 1]), ST), v[2 * j], v[2 * j + 1]);
    }
  }
  store16<OUT_F32, IRHT>(v, sgn, out);
}

// DUP: a 32-element block, whose scale the MMA layout holds for both halves
template <bool DUP = false>
__device__ __forceinline__ uint32_t get_scale(const CopyOut& q, const Flat& f, uint64_t blk) {
  if (!q.mma) return __ldg(q.scales + blk);
  const uint64_t r = f.small ? (uint64_t)f.nkb.div((uint32_t)blk) : blk / f.nkb.d;
  const uint64_t kb = blk - r * f.nkb.d;
  return __ldg(q.scales + mma_scale_offset((int64_t)r, (int64_t)(DUP ? 2 * kb : kb), q.nkb_p));
}

template <int FMT, bool OUT_F32, bool IRHT>
__global__ void __launch_bounds__(256) dequant_rows_kernel(Flat f, CopyOut q, uint64_t seed, void* dst) {
  // launched as a programmatic dependent: the codes may come from the kernel
  // just before this one
  grid_dependency_wait();
  uint32_t sgn[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) sgn[i] = 0u;
  if constexpr (IRHT) {
    const uint32_t m = rht_sign_mask(seed);
#pragma unroll
    for (int i = 0; i < 16; ++i) sgn[i] = ((m >> i) & 1u) << 31;
  }
  constexpr int B = (FMT == 1) ? 32 : 16;
  constexpr int ES = OUT_F32 ? 4 : 2;
  const float g = kTensorScaled<FMT> ? __ldg(q.tensor_scale) : 1.f;
  const int64_t nseg = (f.n + 31) / 32;
  uint8_t* out = static_cast<uint8_t*>(dst);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t sgi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; sgi < nseg; sgi += stride) {
    const int64_t e = sgi * 32;
    // the next segment's codes are loaded ahead, so two loads are in flight
    const int64_t e2 = e + stride * 32;
    if (e2 + 32 <= f.n) asm volatile("prefetch.global.L2 [%0];" ::"l"(q.codes + e2 / 2));
    if (f.n - e >= 32) {
      const uint4 cw = __ldg(reinterpret_cast<const uint4*>(q.codes + e / 2));
      if constexpr (FMT == 7) {   // rows hold whole 64-element blocks
        const uint32_t word = __ldg(reinterpret_cast<const uint32_t*>(q.scales) + (e >> 6));
        const int hb = (int)((e >> 4) & 3);
        deq16_hif4<OUT_F32, IRHT>(cw.x, cw.y, word, hb, sgn, out + e * ES);
        deq16_hif4<OUT_F32, IRHT>(cw.z, cw.w, word, hb + 1, sgn, out + (e + 16) * ES);
      } else if constexpr (B == 32) {
        const float sv = block_scale_value<FMT>(get_scale<true>(q, f, (uint64_t)e / 32));
        deq16<FMT, OUT_F32, IRHT>(cw.x, cw.y, sv, g, sgn, out + e * ES);
        deq16<FMT, OUT_F32, IRHT>(cw.z, cw.w, sv, g, sgn, out + (e + 16) * ES);
      } else {
        const float s0 = block_scale_value<FMT>(get_scale(q, f, (uint64_t)e / 16));
        const float s1 = block_scale_value<FMT>(get_scale(q, f, (uint64_t)e / 16 + 1));
        // two-level NVFP4 and MBS: the scale of the element's 128-element block
        const float gs = kOuterScaled<FMT> ? __ldg(q.tensor_scale + outer_index(q, f, e)) : g;
        deq16<FMT, OUT_F32, IRHT>(cw.x, cw.y, s0, gs, sgn, out + e * ES);
        deq16<FMT, OUT_F32, IRHT>(cw.z, cw.w, s1, gs, sgn, out + (e + 16) * ES);
      }
    } else if constexpr (FMT != 7) {   // a lone 16-block at the very end (16-element formats only)
      const uint2 cw = __ldg(reinterpret_cast<const uint2*>(q.codes + e / 2));
      const float s0 = block_scale_value<FMT>(get_scale(q, f, (uint64_t)e / B));
      const float gs = kOuterScaled<FMT> ? __ldg(q.tensor_scale + outer_index(q, f, e)) : g;
      deq16<FMT, OUT_F32, IRHT>(cw.x, cw.y, s0, gs, sgn, out + e * ES);
    }
  }
}

// ---- host side ---------------------------------------------------------------------
// Scale vectors per row in the MMA layout (one per 16 elements, padded to 4).
int64_t mma_vectors_padded(int64_t cols) { return (cols / 16 + 3) / 4 * 4; }

Flat make_flat(const void* src, int64_t rows, int64_t cols, int block) {
  Flat f{};
  f.src = static_cast<const uint8_t*>(src);
  f.n = rows * cols;
  f.nchunks = (f.n + CH - 1) / CH;
  const int64_t nkb = cols / block;
  f.nkb = make_fastdiv((uint32_t)nkb);
  f.small = (f.n / block < (int64_t(1) << 32) && nkb < (int64_t(1) << 32)) ? 1 : 0;
  return f;
}

// A launch that may begin while the previous kernel on the stream is still
// running (programmatic stream serialisation); the kernel itself waits for
// that kernel's results (griddepcontrol.wait) before it reads them.
template <typename K, typename... Args>
cudaError_t launch_dependent(K kernel, int grid, int smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(RT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename K>
int grid_for(K kernel, int smem, int64_t nchunks) {
  const int occ = cached_occupancy(reinterpret_cast<const void*>(kernel), RT, smem);
  int64_t g = (int64_t)sm_count() * (occ > 0 ? occ : 1);
  if (g > kMaxCtas) g = kMaxCtas;
  return (int)(nchunks < g ? nchunks : g);
}

template <typename K>
cudaError_t prepare(K kernel, int smem) {
  static_assert(sizeof(K) > 0, "");
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <bool F32, bool RHT>
cudaError_t launch_amax_rows(const Flat& f, uint64_t seed, Workspace* ws, cudaStream_t s) {
  auto k = amax_rows_kernel<F32, RHT>;
  constexpr int smem = Ring<F32>::kSmem;
  cudaError_t e = prepare(k, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(k, grid_for(k, smem, f.nchunks), smem, s, f, seed, ws, kRingTimeoutNs);
}

template <int FMT, bool F32, bool RHT, bool SR>
cudaError_t launch_quant_rows(const Flat& f, uint64_t seed, const CopyOut& o, Workspace* ws,
                              cudaStream_t s, int* grid_out) {
  auto k = quant_rows_kernel<FMT, F32, RHT, SR>;
  constexpr int smem = Ring<F32>::kSmem;
  cudaError_t e = prepare(k, smem);
  if (e != cudaSuccess) return e;
  const int grid = grid_for(k, smem, f.nchunks);
  if (grid_out) *grid_out = grid;
  return launch_dependent(k, grid, smem, s, f, seed, philox_key(seed), o, ws, kRingTimeoutNs);
}

template <int FMT, bool F32>
cudaError_t dispatch_quant_rows(int rht, int sr, const Flat& f, uint64_t seed, const CopyOut& o,
                                Workspace* ws, cudaStream_t s, int* grid_out) {
  if (rht) return sr ? launch_quant_rows<FMT, F32, true, true>(f, seed, o, ws, s, grid_out)
                     : launch_quant_rows<FMT, F32, true, false>(f, seed, o, ws, s, grid_out);
  return sr ? launch_quant_rows<FMT, F32, false, true>(f, seed, o, ws, s, grid_out)
            : launch_quant_rows<FMT, F32, false, false>(f, seed, o, ws, s, grid_out);
}

template <int FMT, bool F32, bool RHT, bool SR>
cudaError_t launch_cols_outer(const CUtensorMap& map, const TileGeom& g, uint64_t seed, const CopyOut& c,
                              Workspace* ws, int row_np, cudaStream_t s) {
  auto k = quant_cols_outer_kernel<FMT, F32, RHT, SR>;
  constexpr int smem = TileRing<F32, TOR>::kSmem;
  cudaError_t e = prepare(k, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(k, grid_for(k, smem, g.ntiles), smem, s, map, g, seed, philox_key(seed), c, ws,
                          kRingTimeoutNs, row_np);
}

template <int FMT, bool F32>
cudaError_t dispatch_cols_outer(int rht, int sr, const CUtensorMap& m, const TileGeom& g, uint64_t seed,
                                const CopyOut& c, Workspace* ws, int row_np, cudaStream_t s) {
  if (rht) return sr ? launch_cols_outer<FMT, F32, true, true>(m, g, seed, c, ws, row_np, s)
                     : launch_cols_outer<FMT, F32, true, false>(m, g, seed, c, ws, row_np, s);
  return sr ? launch_cols_outer<FMT, F32, false, true>(m, g, seed, c, ws, row_np, s)
            : launch_cols_outer<FMT, F32, false, false>(m, g, seed, c, ws, row_np, s);
}

template <bool F32, bool ROWS>
cudaError_t launch_amax_tiles(const CUtensorMap& map, const TileGeom& g, uint64_t seed, Workspace* ws,
                              cudaStream_t s) {
  auto k = amax_tiles_kernel<F32, ROWS>;
  constexpr int smem = TileRing<F32>::kSmem;
  cudaError_t e = prepare(k, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(k, grid_for(k, smem, g.ntiles), smem, s, map, g, seed, ws, kRingTimeoutNs);
}

template <int FMT, bool F32, bool RHT, bool SR>
cudaError_t launch_quant_tiles(const CUtensorMap& map, const TileGeom& g, uint64_t seed, bool rows,
                               const CopyOut& r, const CopyOut& c, Workspace* ws, cudaStream_t s) {
  auto k = rows ? quant_tiles_kernel<FMT, F32, RHT, SR, true> : quant_tiles_kernel<FMT, F32, RHT, SR, false>;
  constexpr int smem = TileRing<F32>::kSmem;
  cudaError_t e = prepare(k, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(k, grid_for(k, smem, g.ntiles), smem, s, map, g, seed, philox_key(seed), r, c, ws,
                          kRingTimeoutNs);
}

template <int FMT, bool F32>
cudaError_t dispatch_quant_tiles(int rht, int sr, const CUtensorMap& m, const TileGeom& g, uint64_t seed,
                                 bool rows, const CopyOut& r, const CopyOut& c, Workspace* ws, cudaStream_t s) {
  if (rht) return sr ? launch_quant_tiles<FMT, F32, true, true>(m, g, seed, rows, r, c, ws, s)
                     : launch_quant_tiles<FMT, F32, true, false>(m, g, seed, rows, r, c, ws, s);
  return sr ? launch_quant_tiles<FMT, F32, false, true>(m, g, seed, rows, r, c, ws, s)
            : launch_quant_tiles<FMT, F32, false, false>(m, g, seed, rows, r, c, ws, s);
}

// The source as a 2-D TMA map whose box is one 64-row x 128-byte box of a tile.
bool make_tile_map(CUtensorMap* map, const QuantArgs& a, int tile_rows = TTR) {
  const bool f32 = a.dtype == 1;
  return encode_tiled_2d(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.src,
                         (uint64_t)a.cols, (uint64_t)a.rows, (uint64_t)a.cols * (f32 ? 4u : 2u),
                         f32 ? (uint32_t)TileRing<true>::kBoxCols : (uint32_t)TileRing<false>::kBoxCols,
                         (uint32_t)tile_rows);
}

TileGeom make_tile_geom(const QuantArgs& a, int tile_rows = TTR) {
  TileGeom g;
  g.rows = a.rows;
  g.cols = a.cols;
  g.ntc = (a.cols + TTC - 1) / TTC;
  g.ntiles = ((a.rows + tile_rows - 1) / tile_rows) * g.ntc;
  return g;
}

CopyOut tile_copy(const QOut& q, int64_t crows, int64_t ccols, int block) {
  CopyOut o{};
  o.codes = q.codes;
  o.scales = q.scales;
  o.tensor_scale = q.tensor_scale;
  o.mma = q.scale_layout;
  o.ld = ccols / 2;
  o.nkb = ccols / block;
  o.nkb_p = mma_vectors_padded(ccols);
  o.rows = crows;
  return o;
}

}  // namespace

template <int FMT>
cudaError_t launch_dequant_rows(const Flat& f, const CopyOut& q, int irht, uint64_t seed, void* dst,
                                int f32, cudaStream_t s) {
  const int64_t nseg = (f.n + 31) / 32;
  int64_t grid = (nseg + 255) / 256;
  const int64_t gmax = (int64_t)sm_count() * 8;
  if (grid > gmax) grid = gmax;
  if (grid < 1) grid = 1;
  if (f32) return irht ? launch_dependent(dequant_rows_kernel<FMT, true, true>, (int)grid, 0, s, f, q, seed, dst)
                      : launch_dependent(dequant_rows_kernel<FMT, true, false>, (int)grid, 0, s, f, q, seed, dst);
  return irht ? launch_dependent(dequant_rows_kernel<FMT, false, true>, (int)grid, 0, s, f, q, seed, dst)
              : launch_dependent(dequant_rows_kernel<FMT, false, false>, (int)grid, 0, s, f, q, seed, dst);
}

template <int FMT, bool F32, bool RHT, bool SR>
cudaError_t launch_quant_fused(const Flat& f, uint64_t seed, const CopyOut& o, Workspace* ws,
                               cudaStream_t s) {
  auto k = quant_fused_kernel<FMT, F32, RHT, SR>;
  constexpr int smem = Ring<F32>::kSmem;
  cudaError_t e = prepare(k, smem);
  if (e != cudaSuccess) return e;
  const int grid = grid_for(k, smem, f.nchunks);    // at most the co-resident CTAs
  Flat fa = f;
  uint64_t sd = seed, to = kRingTimeoutNs;
  PhiloxKey pk = philox_key(seed);
  CopyOut oa = o;
  Workspace* wa = ws;
  void* args[] = {&fa, &sd, &pk, &oa, &wa, &to};
  // A grid barrier that ran out of time leaves its arrival count part-way; a
  // stale count would release this launch's barrier early (or never), so the
  // count starts from zero on every call.
  e = cudaMemsetAsync(&ws->gbar_count, 0, sizeof(ws->gbar_count), s);
  if (e != cudaSuccess) return e;
  e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k), dim3(grid), dim3(RT), args, smem, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int FMT, bool F32>
cudaError_t dispatch_quant_fused(int rht, int sr, const Flat& f, uint64_t seed, const CopyOut& o,
                                 Workspace* ws, cudaStream_t s) {
  if (rht) return sr ? launch_quant_fused<FMT, F32, true, true>(f, seed, o, ws, s)
                     : launch_quant_fused<FMT, F32, true, false>(f, seed, o, ws, s);
  return sr ? launch_quant_fused<FMT, F32, false, true>(f, seed, o, ws, s)
            : launch_quant_fused<FMT, F32, false, false>(f, seed, o, ws, s);
}

cudaError_t run_amax_rows(const QuantArgs& a, cudaStream_t s) {
  const Flat f = make_flat(a.src, a.rows, a.cols, a.fmt == 1 ? 32 : 16);
  Workspace* ws = static_cast<Workspace*>(a.ws);
  if (a.dtype == 1) return a.rht ? launch_amax_rows<true, true>(f, a.seed, ws, s)
                                 : launch_amax_rows<true, false>(f, a.seed, ws, s);
  return a.rht ? launch_amax_rows<false, true>(f, a.seed, ws, s)
               : launch_amax_rows<false, false>(f, a.seed, ws, s);
}

cudaError_t run_quant_rows(const QuantArgs& a, cudaStream_t s, int* grid_out) {
  const int block = a.fmt == 1 ? 32 : 16;
  const Flat f = make_flat(a.src, a.rows, a.cols, block);
  CopyOut o{};
  o.codes = a.row.codes;
  o.scales = a.row.scales;
  o.tensor_scale = a.row.tensor_scale;
  o.mma = a.row.scale_layout;
  o.ld = a.cols / 2;
  o.nkb = a.cols / block;
  o.nkb_p = mma_vectors_padded(a.cols);
  o.rows = a.rows;
  Workspace* ws = static_cast<Workspace*>(a.ws);
  const bool f32 = a.dtype == 1;
  const int sr = a.rounding == 1;
  switch (a.fmt) {
    case 0: return f32 ? dispatch_quant_rows<0, true>(a.rht, sr, f, a.seed, o, ws, s, grid_out)
                       : dispatch_quant_rows<0, false>(a.rht, sr, f, a.seed, o, ws, s, grid_out);
    case 1: return f32 ? dispatch_quant_rows<1, true>(a.rht, sr, f, a.seed, o, ws, s, grid_out)
                       : dispatch_quant_rows<1, false>(a.rht, sr, f, a.seed, o, ws, s, grid_out);
    case 2: return f32 ? dispatch_quant_rows<2, true>(a.rht, sr, f, a.seed, o, ws, s, grid_out)
                       : dispatch_quant_rows<2, false>(a.rht, sr, f, a.seed, o, ws, s, grid_out);
    case 3: return f32 ? dispatch_quant_rows<3, true>(a.rht, sr, f, a.seed, o, ws, s, grid_out)
                       : dispatch_quant_rows<3, false>(a.rht, sr, f, a.seed, o, ws, s, grid_out);
    case 4: return f32 ? dispatch_quant_rows<4, true>(a.rht, sr, f, a.seed, o, ws, s, grid_out)
                       : dispatch_quant_rows<4, false>(a.rht, sr, f, a.seed, o, ws, s, grid_out);
    case 5: return f32 ? dispatch_quant_rows<5, true>(a.rht, sr, f, a.seed, o, ws, s, grid_out)
                       : dispatch_quant_rows<5, false>(a.rht, sr, f, a.seed, o, ws, s, grid_out);
    case 6: return f32 ? dispatch_quant_rows<6, true>(a.rht, sr, f, a.seed, o, ws, s, grid_out)
                       : dispatch_quant_rows<6, false>(a.rht, sr, f, a.seed, o, ws, s, grid_out);
    case 7: return f32 ? dispatch_quant_rows<7, true>(a.rht, sr, f, a.seed, o, ws, s, grid_out)
                       : dispatch_quant_rows<7, false>(a.rht, sr, f, a.seed, o, ws, s, grid_out);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t run_dequantize(const DequantArgs& a, cudaStream_t s) {
  const int block = a.fmt == 1 ? 32 : 16;
  const Flat f = make_flat(a.q.codes, a.rows, a.cols, block);
  CopyOut q{};
  q.codes = a.q.codes;
  q.scales = a.q.scales;
  q.tensor_scale = a.q.tensor_scale;
  q.mma = a.q.scale_layout;
  q.ld = a.cols / 2;
  q.nkb = a.cols / block;
  q.nkb_p = mma_vectors_padded(a.cols);
  q.rows = a.rows;
  switch (a.fmt) {
    case 0: return launch_dequant_rows<0>(f, q, a.inverse_rht, a.seed, a.dst, a.dst_dtype, s);
    case 1: return launch_dequant_rows<1>(f, q, a.inverse_rht, a.seed, a.dst, a.dst_dtype, s);
    case 2: return launch_dequant_rows<2>(f, q, a.inverse_rht, a.seed, a.dst, a.dst_dtype, s);
    case 3: return launch_dequant_rows<3>(f, q, a.inverse_rht, a.seed, a.dst, a.dst_dtype, s);
    case 4: return launch_dequant_rows<4>(f, q, a.inverse_rht, a.seed, a.dst, a.dst_dtype, s);
    case 5: return launch_dequant_rows<5>(f, q, a.inverse_rht, a.seed, a.dst, a.dst_dtype, s);
    case 6: return launch_dequant_rows<6>(f, q, a.inverse_rht, a.seed, a.dst, a.dst_dtype, s);
    case 7: return launch_dequant_rows<7>(f, q, a.inverse_rht, a.seed, a.dst, a.dst_dtype, s);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t run_quant_fused(const QuantArgs& a, cudaStream_t s) {
  const Flat f = make_flat(a.src, a.rows, a.cols, 16);
  CopyOut o{};
  o.codes = a.row.codes;
  o.scales = a.row.scales;
  o.tensor_scale = a.row.tensor_scale;
  o.mma = a.row.scale_layout;
  o.ld = a.cols / 2;
  o.nkb = a.cols / 16;
  o.nkb_p = mma_vectors_padded(a.cols);
  o.rows = a.rows;
  Workspace* ws = static_cast<Workspace*>(a.ws);
  const bool f32 = a.dtype == 1;
  const int sr = a.rounding == 1;
  if (a.fmt == 0) return f32 ? dispatch_quant_fused<0, true>(a.rht, sr, f, a.seed, o, ws, s)
                             : dispatch_quant_fused<0, false>(a.rht, sr, f, a.seed, o, ws, s);
  return f32 ? dispatch_quant_fused<2, true>(a.rht, sr, f, a.seed, o, ws, s)
             : dispatch_quant_fused<2, false>(a.rht, sr, f, a.seed, o, ws, s);
}

cudaError_t run_amax_tiles(const QuantArgs& a, cudaStream_t s) {
  CUtensorMap map;
  if (!make_tile_map(&map, a)) return cudaErrorNotSupported;
  const TileGeom g = make_tile_geom(a);
  Workspace* ws = static_cast<Workspace*>(a.ws);
  const bool rows = (a.axis & 1) != 0;
  if (a.dtype == 1) return rows ? launch_amax_tiles<true, true>(map, g, a.seed, ws, s)
                                : launch_amax_tiles<true, false>(map, g, a.seed, ws, s);
  return rows ? launch_amax_tiles<false, true>(map, g, a.seed, ws, s)
              : launch_amax_tiles<false, false>(map, g, a.seed, ws, s);
}

cudaError_t run_quant_tiles(const QuantArgs& a, cudaStream_t s) {
  CUtensorMap map;
  if (!make_tile_map(&map, a)) return cudaErrorNotSupported;
  const int block = a.fmt == 1 ? 32 : 16;
  const TileGeom g = make_tile_geom(a);
  const CopyOut r = tile_copy(a.row, a.rows, a.cols, block);
  const CopyOut c = tile_copy(a.col, a.cols, a.rows, block);
  Workspace* ws = static_cast<Workspace*>(a.ws);
  const bool f32 = a.dtype == 1, rows = (a.axis & 1) != 0;
  const int sr = a.rounding == 1;
  switch (a.fmt) {
    case 0: return f32 ? dispatch_quant_tiles<0, true>(a.rht, sr, map, g, a.seed, rows, r, c, ws, s)
                       : dispatch_quant_tiles<0, false>(a.rht, sr, map, g, a.seed, rows, r, c, ws, s);
    case 1: return f32 ? dispatch_quant_tiles<1, true>(a.rht, sr, map, g, a.seed, rows, r, c, ws, s)
                       : dispatch_quant_tiles<1, false>(a.rht, sr, map, g, a.seed, rows, r, c, ws, s);
    case 2: return f32 ? dispatch_quant_tiles<2, true>(a.rht, sr, map, g, a.seed, rows, r, c, ws, s)
                       : dispatch_quant_tiles<2, false>(a.rht, sr, map, g, a.seed, rows, r, c, ws, s);
    case 4: return f32 ? dispatch_quant_tiles<4, true>(a.rht, sr, map, g, a.seed, rows, r, c, ws, s)
                       : dispatch_quant_tiles<4, false>(a.rht, sr, map, g, a.seed, rows, r, c, ws, s);
    case 5: return f32 ? dispatch_quant_tiles<5, true>(a.rht, sr, map, g, a.seed, rows, r, c, ws, s)
                       : dispatch_quant_tiles<5, false>(a.rht, sr, map, g, a.seed, rows, r, c, ws, s);
    default: return cudaErrorNotSupported;     // the two-level and MBS formats are row-wise only
  }
}

cudaError_t run_quant_cols_outer(const QuantArgs& a, int row_np, cudaStream_t s) {
  CUtensorMap map;
  if (!make_tile_map(&map, a, TOR)) return cudaErrorNotSupported;
  const TileGeom g = make_tile_geom(a, TOR);
  const CopyOut c = tile_copy(a.col, a.cols, a.rows, 16);
  Workspace* ws = static_cast<Workspace*>(a.ws);
  const bool f32 = a.dtype == 1;
  const int sr = a.rounding == 1;
  switch (a.fmt) {
    case 3: return f32 ? dispatch_cols_outer<3, true>(a.rht, sr, map, g, a.seed, c, ws, row_np, s)
                       : dispatch_cols_outer<3, false>(a.rht, sr, map, g, a.seed, c, ws, row_np, s);
    case 6: return f32 ? dispatch_cols_outer<6, true>(a.rht, sr, map, g, a.seed, c, ws, row_np, s)
                       : dispatch_cols_outer<6, false>(a.rht, sr, map, g, a.seed, c, ws, row_np, s);
    case 7: return f32 ? dispatch_cols_outer<7, true>(a.rht, sr, map, g, a.seed, c, ws, row_np, s)
                       : dispatch_cols_outer<7, false>(a.rht, sr, map, g, a.seed, c, ws, row_np, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fp4q
