// Block-scaled operands on a 16-bit tensor-core contraction (sm_103a).
//
// "Replanteamiento del Sesgo de Contraccion en el Preentrenamiento de LLM en
// FP4", Metodologia §2 and Resultados: UFP4 (the uniform E1M2 grid) with the
// RHT on every training GEMM. No tensor-core format holds UFP4, so this GEMM
// dequantises on the fly: its converter warps turn each operand's 4-bit codes
// and block scales into the exact 16-bit block values level * s_b in shared
// memory, and tcgen05.mma.kind::f16 multiplies them with FP32 accumulation in
// TMEM; the epilogue applies g_A * g_B. Nothing dequantised ever goes to HBM.
//
// Which 16-bit type holds level * s_b exactly:
//   UFP4 (levels 0..7) and NVFP4 (E2M1 levels) with E4M3 scales: FP16. The
//     product has at most 3 + 4 significant bits and lies in [2^-10, 3136].
//   The E8M0 formats (MXFP4 on 32- or 16-element blocks, OAS): BF16, whose
//     exponent range covers 2^e for every E8M0 code.
//   HiF4 ("Unleashing Low-Bit Inference on Ascend NPUs ...", Resumen tecnico
//     §2): BF16. A value is level * S * 2^-(d_8 + d_4), levels 0..7 and S an
//     E6M2 value: at most 3 + 3 significant bits in [2^-34, 7 * 1.75 * 2^32].
//     One scale word per row and 64-element K stage.
// The FP16 / BF16 products of two such values are exact in FP32, so the only
// rounding is the FP32 accumulation. The uniform levels (UFP4, HiF4) are made
// by one packed FMA on a magic-number word per pair of values
// (convert8_uniform: 1402 against 1623 us for HiF4 at 8192^3 with two byte
// look-ups per pair, 1072 against 1109 us for UFP4 with one); the E2M1 levels
// by byte look-ups. HiF4's micro-block scale pairs come from the shift count
// by one integer multiply-add each, not by selects (1315 against 1402 us).
//
// Structure: pairs of CTAs (two-CTA clusters, 672 threads each) compute one
// 256 x 256 tile of Y with the two-SM MMA (cta_group::2): CTA r of the pair
// converts rows [128 r, 128 r + 128) of the tile's A rows and of its B rows,
// so each SM converts 256 rows per K stage for 128 x 256 x 64 multiply-adds
// (a one-CTA 128 x 256 tile converts 384).
//   warps 0-15  converters: per K stage of 64 elements, each thread takes one
//               half row (32 elements: one 16-byte load of codes and its
//               scales, issued two stages ahead from per-tile pointers), makes
//               four 16-byte chunks of 16-bit values and stores them in the
//               128-byte-swizzled K-major layout the MMA reads; then fences
//               the stores for the async proxy and arrives on the stage's
//               "full" barrier.
//   warp 16     allocates 512 TMEM columns in both CTAs (two 256-column
//               accumulators). In CTA 0 one thread waits for both CTAs' stage
//               (CTA 1's warp 16 relays its "full" to CTA 0), issues four
//               tcgen05.mma.cta_group::2.kind::f16 (M = 256, N = 256, K = 16)
//               and commits the stage back to both CTAs' converters and, after
//               the last stage, the accumulator to both epilogues.
//   warps 17-20 epilogue, one per TMEM lane quadrant: reads the accumulator in
//               32-column chunks, multiplies by g_A * g_B, stores BF16
//               (nearest-even) or FP32, then frees the accumulator; the other
//               accumulator already takes the next tile's MMAs.
// The relay is a relaxed arrival of an event the relaying thread observed
// complete in its own CTA (every converter's stores fenced and released on
// the stage barrier). Rows of A or B past M or N are converted as zeros and
// never stored, so M and N need not be tile multiples. Every mbarrier wait is
// bounded; on expiry the kernel records FP4Q_ETIMEOUT in the workspace and
// returns.
#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fp4q_device.cuh"
#include "fp4q_ptx.cuh"
#include "fp4q_tc.cuh"
#include "fp4q_internal.h"

namespace fp4q {
namespace {

constexpr int kTile = 256;                     // a CTA pair's tile: 256 rows of A x 256 rows of B
constexpr int kBM = 128, kBN = 128;            // each CTA's rows of A and of B
constexpr int kBK = 64;                        // K elements per stage (128 bytes of 16-bit values per row)
constexpr int kStages = 6;
constexpr int kABytes = kBM * 128;             // 16 KB
constexpr int kBBytes = kBN * 128;             // 16 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kConvWarps = 16;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kMmaWarp = kConvWarps;
constexpr int kEpiWarp0 = kConvWarps + 1;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (kConvWarps + 1 + kEpiWarps);
constexpr int kTasks = (kBM + kBN) * 2 / kConvThreads;   // half rows per converter thread per stage
constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
constexpr uint64_t kTimeoutNs = 2000000000ull;
static_assert((kBM + kBN) * 2 % kConvThreads == 0, "whole tasks per thread");
static_assert(kSmem <= 227 * 1024, "shared memory budget");

// Kinds of operand: how a code and a block scale become a 16-bit value.
enum Kind { kNvfp4F16 = 0, kUfp4F16 = 1, kE8m0Bf16 = 2, kHif4Bf16 = 3 };

// High bytes of the FP16 values of the 8 E2M1 magnitudes {0, 0.5, 1, 1.5, 2,
// 3, 4, 6} (their low bytes are all zero).
constexpr uint32_t kE2m1F16Lo = 0x3E3C3800u, kE2m1F16Hi = 0x46444240u;
// BF16 values of the E2M1 magnitudes, split into high and low bytes.
constexpr uint32_t kE2m1Bf16HiLo = 0x3F3F3F00u, kE2m1Bf16HiHi = 0x40404040u;
constexpr uint32_t kE2m1Bf16LoLo = 0xC0800000u, kE2m1Bf16LoHi = 0xC0804000u;

struct DqArgs {
  const uint8_t* codes;    // rows x K/2
  const uint8_t* scales;   // linear (rows x K/block) or tiled (16-element positions)
  int rows;
  int tiled;               // scale layout
  int block32;             // linear MXFP4 scales: one per 32 elements
  int hif4;                // HiF4: one 32-bit scale word per 64 elements (linear)
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

struct Task {
  uint4 codes;
  uint32_t scales;
};

// Pairs of block scales as 16-bit pairs (first block's in sa, second's in sb).
template <int KIND>
__device__ __forceinline__ void scale_pairs(uint32_t sc, uint32_t& sa, uint32_t& sb) {
  if constexpr (KIND == kE8m0Bf16) {
    const uint32_t c0 = sc & 0xFFu, c1 = (sc >> 8) & 0xFFu;
    const uint32_t b0 = c0 ? (c0 << 7) : 0x40u;          // 2^(c - 127); code 0 is the subnormal 2^-127
    const uint32_t b1 = c1 ? (c1 << 7) : 0x40u;
    sa = b0 | (b0 << 16);
    sb = b1 | (b1 << 16);
  } else {
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(sc));
    sa = prmt(h2, h2, 0x1010u);
    sb = prmt(h2, h2, 0x3232u);
  }
}

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_bf16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// HiF4: the eight 4-element micro-blocks of half h of a 64-element block as
// BF16 scale pairs, S * 2^-(d_8 + d_4) (S = 0 stays 0). S is E6M2 (bias 31):
// exponent field E >= 1 -> BF16 exponent E + 96 and mantissa m << 5; E = 0 ->
// m * 2^-32, exact in FP32 and then in BF16. The three possible pairs (S,
// S / 2, S / 4: one BF16 exponent step each) are formed once; each micro-block
// selects one by its two bits.
__device__ __forceinline__ void hif4_scale_pairs(uint32_t wd, int h, uint32_t (&mp)[8], uint32_t (&ap)[8]) {
  const uint32_t c = wd & 0xFFu, E = c >> 2, m = c & 3u;
  const uint32_t sb = E ? (((E + 96u) << 7) | (m << 5))
                        : (__float_as_uint(__fmul_rn((float)m, 2.3283064365386963e-10f)) >> 16);
  // S / 16 (exponent - 4) and -8 S (exponent + 3, sign set) in both halves;
  // a micro-block's pair is k = d_8 + d_4 BF16 exponent steps below them
  // (all normal: S >= 2^-32), or 0 when S = 0
  const uint32_t t0 = sb * 0x00010001u;
  const uint32_t m0 = sb ? t0 - 0x02000200u : 0u;
  const uint32_t a0 = sb ? (t0 + 0x01800180u) | 0x80008000u : 0u;
  const uint32_t step = sb ? 0x00800080u : 0u;
  const uint32_t b8 = wd >> (8 + 4 * h), b4 = wd >> (16 + 8 * h);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t k = ((b8 >> (i >> 1)) & 1u) + ((b4 >> i) & 1u);
    mp[i] = m0 - k * step;
    ap[i] = a0 - k * step;
  }
}

__device__ __forceinline__ uint32_t fma2_f16(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t fma2_bf16(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Eight uniform-level codes (UFP4, HiF4; one 32-bit word: element 2j in the
// low nibble of byte j) times scale pairs -> four 16-bit pairs (one 16-byte
// chunk, element order), without table look-ups: a word whose 16-bit halves are +-(B + 16 |code|), B = 1024 (FP16,
// high byte 0x64) or 128 (BF16, high byte 0x43), is one prmt (the code's
// magnitude bits 4-6 of a byte; its sign bit replicated over the next byte)
// and one LOP3; then fma(a, s / 16, -+B s / 16) = code * s, exact since the
// product fits the 16-bit format (one rounding of an exact value). mlo / mhi
// hold s / 16 and alo / ahi -B s / 16 for codes 0-3 / 4-7.
template <bool BF16>
__device__ __forceinline__ uint4 convert8_uniform(uint32_t w, uint32_t mlo, uint32_t alo, uint32_t mhi,
                                                  uint32_t ahi) {
  const uint32_t t = w << 4;                 // byte j: code 2j in bits 4-7 (its sign in bit 7)
  constexpr uint32_t kHigh = BF16 ? 0x43004300u : 0x64006400u;
  uint32_t out[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // bytes: t.j (code 2j), sign of t.j replicated, w.j (code 2j + 1), sign of w.j replicated
    const uint32_t x = prmt(t, w, (uint32_t)j | ((8u | (uint32_t)j) << 4) | ((uint32_t)(4 + j) << 8) |
                                      ((uint32_t)(12 + j) << 12));
    const uint32_t a = (x & 0x80708070u) | kHigh;
    const uint32_t m2 = j < 2 ? mlo : mhi, a2 = j < 2 ? alo : ahi;
    const uint32_t c2 = a2 ^ (a & 0x80008000u);
    out[j] = BF16 ? fma2_bf16(a, m2, c2) : fma2_f16(a, m2, c2);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Eight E2M1 codes (NVFP4 with FP16 block values, the E8M0 formats with BF16)
// times scale pairs, the level by a byte look-up (prmt); codes 0-3 take s2lo,
// codes 4-7 s2hi.
template <int KIND>
__device__ __forceinline__ uint4 convert8(uint32_t w, uint32_t s2lo, uint32_t s2hi) {
  const uint32_t t = w << 4;                 // byte j: low code's nibble in bits 4-7
  const uint32_t e4 = t & 0x70707070u;       // byte j, bits 4-6: magnitude of code 2j
  const uint32_t o4 = w & 0x70707070u;       // byte j, bits 4-6: magnitude of code 2j + 1
  uint32_t out[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // selector nibbles (0, |code 2j|, 0, |code 2j + 1|): entry 0 of every table is 0
    const uint32_t x = prmt(e4, o4, (uint32_t)j | ((uint32_t)(4 + j) << 4));
    const uint32_t s2 = j < 2 ? s2lo : s2hi;
    uint32_t v;
    if constexpr (KIND == kNvfp4F16) {
      v = hmul2_f16(prmt(kE2m1F16Lo, kE2m1F16Hi, x), s2);
    } else {
      const uint32_t hi = prmt(kE2m1Bf16HiLo, kE2m1Bf16HiHi, x);
      const uint32_t lo = prmt(kE2m1Bf16LoLo, kE2m1Bf16LoHi, x >> 4);
      v = hmul2_bf16(hi | lo, s2);
    }
    // sign bits: code 2j's (bit 3 of byte j of w, bit 7 of byte j of t) to
    // bit 15, code 2j + 1's (bit 7 of byte j of w) to bit 31
    const uint32_t sg = prmt(t, w, ((uint32_t)j << 4) | ((uint32_t)(4 + j) << 12));
    out[j] = v ^ (sg & 0x80008000u);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Instruction descriptor, kind::f16: FP32 accumulator, A and B of one 16-bit
// type (0 FP16, 1 BF16), both K-major, N >> 3 in bits 17-22, M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n, uint32_t type) {
  return (1u << 4) | (type << 7) | (type << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tc2_mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

template <int KIND, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
gemm_dq_kernel(DqArgs A, DqArgs B, int K, const float* __restrict__ g_a, const float* __restrict__ g_b,
               void* __restrict__ y, int M, int N, Workspace* ws, uint64_t timeout_ns) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  // bars[0..S): full, [S..2S): empty, [2S..3S): pfull, 3S + b: tfull[b], 3S + 2 + b: tempty[b], 3S + 4: drain
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = (int)cluster_id_x(), npairs = (int)cluster_count_x();
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto pfull_bar = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (3 * kStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (3 * kStages + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (3 * kStages + 4);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), kConvThreads);
      mbar_init(empty_bar(s), 1);
      mbar_init(pfull_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * kEpiWarps);        // one arrival per epilogue warp of each CTA
    }
    mbar_init(drain_bar, 1);
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    // one warp of each CTA of the pair allocates, collectively, in both TMEMs
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(&s_tmem_base)), "r"(512) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // both CTAs' barriers exist before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tmem = s_tmem_base;

  const int num_n = (N + kTile - 1) / kTile;
  const int num_tiles = ((M + kTile - 1) / kTile) * num_n;
  const int nk = K / kBK;
  const int my_tiles = pair < num_tiles ? (num_tiles - 1 - pair) / npairs + 1 : 0;

  auto fail = [&]() {
    if (!s_abort) {
      s_abort = 1;
      atomicOr(&ws->status, kStatusTimeout);
    }
  };

  if (warp < kConvWarps) {
    // ---------------- converters ----------------
    const int tid = threadIdx.x;
    const int64_t total = (int64_t)my_tiles * nk;          // this CTA's stages
    // What each of this thread's tasks is, fixed for the kernel: its half row
    // (operand, row within the tile, half h) and where its 16-byte chunks go.
    int trow[kTasks];            // row within the operand's tile
    bool tis_a[kTasks];
    uint32_t tsmem[kTasks];      // byte offset of the row within a stage
    uint32_t tkey[kTasks];       // 128-byte swizzle: chunk c sits at (c ^ key) * 16
#pragma unroll
    for (int j = 0; j < kTasks; ++j) {
      const int q = tid + kConvThreads * j;
      const int lr = q >> 1;
      tis_a[j] = lr < kBM;
      trow[j] = tis_a[j] ? lr : lr - kBM;
      tsmem[j] = (tis_a[j] ? 0u : (uint32_t)kABytes) + (uint32_t)((trow[j] >> 3) * 1024 + (trow[j] & 7) * 128);
      tkey[j] = (uint32_t)(trow[j] & 7);
    }
    const int h = tid & 1;       // every task of a thread has the same half (kConvThreads is even)
    // The fetch cursor runs two stages ahead of the conversion: its tile, K
    // stage, and each task's code and scale pointers (advanced per stage).
    int f_tile_i = 0, f_ks = 0;
    const uint8_t* cptr[kTasks];
    const uint8_t* sptr[kTasks];
    int sstep[kTasks];
    bool valid[kTasks];
    auto start_tile = [&](int tile_i) {
      const int tile = pair + tile_i * npairs;
      const int m = tile / num_n, n = tile % num_n;
#pragma unroll
      for (int j = 0; j < kTasks; ++j) {
        const DqArgs& o = tis_a[j] ? A : B;
        const int r = (tis_a[j] ? m : n) * kTile + (int)rank * 128 + trow[j];
        valid[j] = r < o.rows;
        const int rr = valid[j] ? r : 0;
        cptr[j] = o.codes + (int64_t)rr * (K / 2) + h * 16;
        const int nkb = K / 16;
        if (o.tiled) {
          sptr[j] = o.scales + (int64_t)(rr >> 7) * (nkb >> 2) * 512 + (rr & 31) * 16 + ((rr >> 5) & 3) * 4 + 2 * h;
          sstep[j] = 512;
        } else if (o.hif4) {       // both halves read the block's word
          sptr[j] = o.scales + (int64_t)rr * (K / 16);
          sstep[j] = 4;
        } else if (o.block32) {
          sptr[j] = o.scales + (int64_t)rr * (K / 32) + h;
          sstep[j] = 2;
        } else {
          sptr[j] = o.scales + (int64_t)rr * nkb + 2 * h;
          sstep[j] = 4;
        }
      }
    };
    auto fetch = [&](Task (&t)[kTasks]) {
      if (f_tile_i >= my_tiles) return;
#pragma unroll
      for (int j = 0; j < kTasks; ++j) {
        if (valid[j]) {
          t[j].codes = __ldg(reinterpret_cast<const uint4*>(cptr[j]));
          if constexpr (KIND == kHif4Bf16) {
            t[j].scales = __ldg(reinterpret_cast<const uint32_t*>(sptr[j]));
          } else if (sstep[j] == 2) {
            const uint32_t b = __ldg(sptr[j]);
            t[j].scales = b | (b << 8);
          } else {
            t[j].scales = __ldg(reinterpret_cast<const uint16_t*>(sptr[j]));
          }
          cptr[j] += 32;
          sptr[j] += sstep[j];
        } else {
          t[j].codes = make_uint4(0u, 0u, 0u, 0u);
          t[j].scales = 0u;
        }
      }
      if (++f_ks == nk) {
        f_ks = 0;
        if (++f_tile_i < my_tiles) start_tile(f_tile_i);
      }
    };
    auto convert_stage = [&](int64_t g, const Task (&t)[kTasks]) -> bool {
      const int s = (int)(g % kStages);
      const uint32_t ph = (uint32_t)((g / kStages) & 1);
      if (!mbar_wait(empty_bar(s), ph ^ 1u, &s_abort, timeout_ns)) return false;
      uint8_t* st = smem + s * kStageBytes;
#pragma unroll
      for (int j = 0; j < kTasks; ++j) {
        uint8_t* rowp = st + tsmem[j];
        const uint32_t w[4] = {t[j].codes.x, t[j].codes.y, t[j].codes.z, t[j].codes.w};
        if constexpr (KIND == kHif4Bf16) {
          uint32_t mp[8], ap[8];
          hif4_scale_pairs(t[j].scales, h, mp, ap);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t c = (uint32_t)(4 * h + i);
            *reinterpret_cast<uint4*>(rowp + ((c ^ tkey[j]) << 4)) =
                convert8_uniform<true>(w[i], mp[2 * i], ap[2 * i], mp[2 * i + 1], ap[2 * i + 1]);
          }
        } else if constexpr (KIND == kUfp4F16) {
          uint32_t sa, sb;
          scale_pairs<KIND>(t[j].scales, sa, sb);
          // s / 16 and -64 s (exact: s is E4M3, >= 2^-9 when not 0)
          const uint32_t ma = hmul2_f16(sa, 0x2C002C00u), mb = hmul2_f16(sb, 0x2C002C00u);
          const uint32_t aa = hmul2_f16(sa, 0xD400D400u), ab = hmul2_f16(sb, 0xD400D400u);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t c = (uint32_t)(4 * h + i);
            *reinterpret_cast<uint4*>(rowp + ((c ^ tkey[j]) << 4)) =
                i < 2 ? convert8_uniform<false>(w[i], ma, aa, ma, aa) : convert8_uniform<false>(w[i], mb, ab, mb, ab);
          }
        } else {
          uint32_t sa, sb;
          scale_pairs<KIND>(t[j].scales, sa, sb);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t c = (uint32_t)(4 * h + i);         // 16-byte chunk of the 128-byte row
            const uint32_t s2 = i < 2 ? sa : sb;
            *reinterpret_cast<uint4*>(rowp + ((c ^ tkey[j]) << 4)) = convert8<KIND>(w[i], s2, s2);
          }
        }
      }
      // the stores become visible to the tensor cores' (async) reads
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(full_bar(s));
      return true;
    };
    Task t0[kTasks], t1[kTasks];
    if (my_tiles > 0) start_tile(0);
    fetch(t0);
    fetch(t1);
    for (int64_t g = 0; g < total; g += 2) {
      if (!convert_stage(g, t0)) { fail(); break; }
      fetch(t0);
      if (g + 1 >= total) break;
      if (!convert_stage(g + 1, t1)) { fail(); break; }
      fetch(t1);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0 && rank == 1) {
      // ---------------- rank 1: hand each converted stage to rank 0 ----------------
      const uint32_t peer_pfull0 = peer_addr(pfull_bar(0), 0);
      const int64_t total = (int64_t)my_tiles * nk;
      for (int64_t g = 0; g < total; ++g) {
        const int s = (int)(g % kStages);
        if (!mbar_wait(full_bar(s), (uint32_t)((g / kStages) & 1), &s_abort, timeout_ns)) { fail(); break; }
        mbar_arrive_remote(peer_pfull0 + 8u * s);
      }
    } else if (lane == 0) {
      // ---------------- rank 0: MMA issuer for the pair ----------------
      const uint32_t idesc = idesc_f16(2 * kBM, 2 * kBN, (KIND == kE8m0Bf16 || KIND == kHif4Bf16) ? 1u : 0u);
      const uint32_t base = smem_u32(smem);
      const uint64_t da0 = smem_desc(base, 16, 1024, 2);
      const uint64_t db0 = smem_desc(base + kABytes, 16, 1024, 2);
      const uint32_t peer_empty0 = peer_addr(empty_bar(0), 1);
      const uint32_t peer_tfull0 = peer_addr(tfull_bar(0), 1);
      bool ok = true, issued_any = false;
      int64_t g = 0;
      for (int i = 0; i < my_tiles && ok; ++i) {
        const int b = i & 1;
        if (!mbar_wait_cluster(tempty_bar(b), (uint32_t)(((i >> 1) & 1) ^ 1), &s_abort, timeout_ns)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * kTile);
        for (int ks = 0; ks < nk; ++ks, ++g) {
          const int s = (int)(g % kStages);
          const uint32_t ph = (uint32_t)((g / kStages) & 1);
          if (!mbar_wait(full_bar(s), ph, &s_abort, timeout_ns) ||
              !mbar_wait_cluster(pfull_bar(s), ph, &s_abort, timeout_ns)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t off = (uint64_t)(s * (kStageBytes >> 4));
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j)
            tc2_mma_f16(d, da0 + off + 2 * j, db0 + off + 2 * j, idesc, (ks | j) != 0 ? 1u : 0u);
          issued_any = true;
          tc2_commit(empty_bar(s));
          tc2_commit(peer_empty0 + 8u * s);
        }
        if (!ok) break;
        tc2_commit(tfull_bar(b));
        tc2_commit(peer_tfull0 + 8u * b);
      }
      if (!ok && issued_any) {
        tc2_commit(drain_bar);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < 50000000ull) {
        }
      }
    }
  } else {
    // ---------------- epilogue (one warp per TMEM lane quadrant) ----------------
    const int q = warp & 3;
    const float alpha = __fmul_rn(__ldg(g_a), __ldg(g_b));
    const uint32_t tempty0 = rank == 0 ? tempty_bar(0) : peer_addr(tempty_bar(0), 0);
    for (int i = 0; i < my_tiles; ++i) {
      const int tile = pair + i * npairs;
      const int m = tile / num_n, n = tile % num_n;
      const int b = i & 1;
      if (!mbar_wait(tfull_bar(b), (uint32_t)((i >> 1) & 1), &s_abort, timeout_ns)) { fail(); break; }
      tc_fence_after();
      const int row = m * kTile + (int)rank * 128 + q * 32 + lane;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * kTile);
#pragma unroll 1
      for (int c = 0; c < kTile / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(taddr + (uint32_t)(c * 32), r);
        const int col0 = n * kTile + c * 32;
        if (row >= M) continue;
        if constexpr (OUT_F32) {
          float* out = static_cast<float*>(y) + (int64_t)row * N + col0;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            if (col0 + 4 * v >= N) break;
            *reinterpret_cast<float4*>(out + 4 * v) =
                make_float4(__fmul_rn(__uint_as_float(r[4 * v]), alpha), __fmul_rn(__uint_as_float(r[4 * v + 1]), alpha),
                            __fmul_rn(__uint_as_float(r[4 * v + 2]), alpha), __fmul_rn(__uint_as_float(r[4 * v + 3]), alpha));
          }
        } else {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(y) + (int64_t)row * N + col0;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            if (col0 + 8 * v >= N) break;
            uint32_t hw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(r[8 * v + 2 * k]), alpha),
                                                              __fmul_rn(__uint_as_float(r[8 * v + 2 * k + 1]), alpha));
              hw[k] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(out + 8 * v) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(tempty0 + 8u * b);
        else mbar_arrive_remote(tempty0 + 8u * b);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // no cross-CTA arrival or shared-memory read is still under way
  tc_fence_after();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

template <int KIND, bool OUT_F32>
cudaError_t launch_dq(const GemmArgs& a, cudaStream_t s) {
  auto k = gemm_dq_kernel<KIND, OUT_F32>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const bool b32 = a.fmt == 1;     // MXFP4: one scale per 32 elements in the linear layout
  const int hif4 = a.fmt == 7 ? 1 : 0;
  DqArgs da{a.a.codes, a.a.scales, (int)a.m, a.a.scale_layout, b32 && !a.a.scale_layout, hif4};
  DqArgs db{a.b.codes, a.b.scales, (int)a.n, a.b.scale_layout, b32 && !a.b.scale_layout, hif4};
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int pairs = sm_count() / 2;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  int resident = 0;
  if (cudaOccupancyMaxActiveClusters(&resident, k, &cfg) == cudaSuccess && resident > 0) {
    if (resident < pairs) pairs = resident;
  } else {
    cudaGetLastError();
  }
  const int tiles = (int)(((a.m + kTile - 1) / kTile) * ((a.n + kTile - 1) / kTile));
  if (tiles < pairs) pairs = tiles;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  e = cudaLaunchKernelEx(&cfg, k, da, db, (int)a.k, (const float*)a.a.tensor_scale,
                         (const float*)a.b.tensor_scale, a.y, (int)a.m, (int)a.n,
                         static_cast<Workspace*>(a.ws), kTimeoutNs);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int KIND>
cudaError_t launch_dq_out(const GemmArgs& a, cudaStream_t s) {
  return a.out_dtype == 1 ? launch_dq<KIND, true>(a, s) : launch_dq<KIND, false>(a, s);
}

}  // namespace

cudaError_t run_gemm_dequant(const GemmArgs& a, cudaStream_t s) {
  switch (a.fmt) {
    case 0: return launch_dq_out<kNvfp4F16>(a, s);
    case 2: return launch_dq_out<kUfp4F16>(a, s);
    case 1: case 4: case 5: return launch_dq_out<kE8m0Bf16>(a, s);
    case 7: return launch_dq_out<kHif4Bf16>(a, s);
    default: return cudaErrorNotSupported;      // per-128 scales: not one 16-bit value per element
  }
}

}  // namespace fp4q
