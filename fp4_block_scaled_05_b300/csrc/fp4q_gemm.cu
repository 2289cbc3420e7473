// Block-scaled FP4 GEMM on the 5th-generation tensor cores (sm_103a).
//
// Y[M][N] = (sum_k A[m][k] * B[n][k]) * g_A * g_B, with A, B row-wise NVFP4
// copies (E2M1 codes, one E4M3 scale per 16 elements along K, one FP32 tensor
// scale each): "Le Architetture Normalizzate sono Nativamente a 4 Bit",
// Metodologia (NVFP4 consumed natively by Blackwell tensor cores); "Unveiling
// the Potential of Quantization with MXFP4 ...", Resume technique §2B (scale
// factors handled beside the dense tensor-core math). The same kernel takes
// the MXFP4 formats (E8M0 scales, g = 1): the instruction's scale type
// switches to UE8M0, and a 32-element block's scale sits in the scale layout
// once for each of its 16-element halves.
//
// Two kernels: when M and N are multiples of 256, CTA pairs share each
// 256 x 256 tile through the two-SM MMA (gemm_nvf4_pair_kernel, below);
// otherwise one CTA per 128 x BN tile (gemm_nvf4_kernel).
//
// One-CTA structure (one persistent CTA per SM, 448 threads):
//   warp 0      TMA producer: per K stage of 256 elements, one 2-D tiled TMA
//               load (128B swizzle) of the A and B code tiles and 1-D bulk
//               copies of their scale tiles into a shared-memory ring (4
//               stages for BN = 256, 6 for BN = 128; mbarrier transaction
//               counts).
//   warp 1      allocates the 512 TMEM columns; one thread issues, once the
//               stage's scales are in TMEM, four
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X
//               (M = 128, N = BN, K = 64) into an FP32 accumulator in TMEM;
//               tcgen05.commit frees the ring slot and, after the last stage,
//               hands the accumulator to the epilogue.
//   warps 2-9   epilogue: each warp reads its 32 TMEM lanes x BN/2 columns
//               into registers, 64 columns at a time, releases the
//               accumulator after the last read (the next tile's MMAs
//               start), multiplies by g_A * g_B and stores BF16
//               (nearest-even) or FP32.
//   warps 10-13 scale writers, one per TMEM lane quadrant: each stage's scale
//               tiles go from shared memory into TMEM by tcgen05.st (moving
//               them with tcgen05.cp, in the MMA thread's stream, took tensor-
//               pipe time from the MMAs: 306 against 227 us at 8064 x 8192 x
//               8192).
// Every mbarrier wait is bounded by a global-timer deadline; on expiry the
// kernel records FP4Q_ETIMEOUT in the workspace, drains what it issued and
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

constexpr int BM = 128;           // rows of A per tile (= MMA M)
constexpr int BK_BYTES = 128;     // bytes of codes per row per stage (256 FP4 values)
constexpr int BK = 256;           // K elements per stage
constexpr int kEpiWarps = 8;              // two per TMEM lane quadrant
constexpr int kScaleWarps = 4;            // one per TMEM lane quadrant
constexpr int kScaleWarp = 2 + kEpiWarps; // the first of them
constexpr int kThreads = 64 + 32 * kEpiWarps + 32 * kScaleWarps;
constexpr int kTmemCols = 512;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s

template <int BN>
struct Cfg {
  static constexpr int kStages = BN == 128 ? 6 : 4;   // as many as shared memory holds
  static constexpr int kABytes = BM * BK_BYTES;
  static constexpr int kBBytes = BN * BK_BYTES;
  static constexpr int kSfaBytes = 2048;                 // 128 rows x 16 scales
  static constexpr int kSfbBytes = (BN / 128) * 2048;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kSfaCols = 16;                    // 4 K chunks x 4 TMEM columns
  static constexpr int kSfbCols = (BN / 128) * 16;
  static constexpr int kSfStageCols = kSfaCols + kSfbCols;
  static constexpr int kSfBase = BN;                     // accumulator uses columns [0, BN)
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
  static_assert(kSfBase + kStages * kSfStageCols <= kTmemCols, "TMEM budget");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
};

// ---- the kernel -----------------------------------------------------------------
template <int BN, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                 const uint8_t* __restrict__ sfa, const uint8_t* __restrict__ sfb,
                 const float* __restrict__ g_a, const float* __restrict__ g_b, void* __restrict__ y,
                 int M, int N, int K, Workspace* ws, uint64_t timeout_ns, int skip_first_stage,
                 int ue8m0) {
  using C = Cfg<BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  // bars[0..S): full, bars[S..2S): empty, bars[2S]: tmem_full, bars[2S+1]: tmem_empty, bars[2S+2]: drain,
  // bars[2S+3+s]: sfull[s] (the scales of stage s written into TMEM)
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cid = (int)blockIdx.x, ncl = (int)gridDim.x;   // first tile, tile stride
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::kStages + s); };
  const uint32_t tmem_full = bar0 + 8u * (2 * C::kStages);
  const uint32_t tmem_empty = bar0 + 8u * (2 * C::kStages + 1);
  const uint32_t drain_bar = bar0 + 8u * (2 * C::kStages + 2);
  auto sfull_bar = [&](int s) { return bar0 + 8u * (2 * C::kStages + 3 + s); };

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sfull_bar(s), kScaleWarps);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, 32 * kEpiWarps);
    mbar_init(drain_bar, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(&s_tmem_base)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem_base;

  const int num_n = N / BN;
  const int num_tiles = (M / BM) * num_n;
  const int nk = K / BK;
  const int64_t sf_row_stride = (int64_t)(K / 64) * 512;   // bytes per 128-row scale tile row

  auto fail = [&]() {
    if (!s_abort) {
      s_abort = 1;
      atomicOr(&ws->status, kStatusTimeout);
    }
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t pending = 0;    // bit ss: stage ss has copies whose phase may not have completed
      uint32_t pend_ph = 0;    // bit ss: the parity of that phase
      bool ok = true;
      for (int gi = cid; gi < num_tiles && ok; gi += ncl) {
        const int m = gi / num_n, n = gi % num_n;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, &s_abort, timeout_ns)) { fail(); ok = false; break; }
          const bool skip = skip_first_stage && blockIdx.x == 0 && gi == cid && ks == 0;
          pending &= ~(1u << s);
          if (!skip) {
            uint8_t* st = smem + s * C::kStageBytes;
            const uint32_t fb = full_bar(s);
            mbar_arrive_expect_tx(fb, C::kStageBytes);
            tma_load_2d(smem_u32(st), &tmap_a, fb, ks * BK_BYTES, m * BM);
            bulk_load(smem_u32(st + C::kABytes + C::kBBytes),
                      sfa + (int64_t)m * sf_row_stride + (int64_t)ks * 2048, 2048, fb);
            tma_load_2d(smem_u32(st + C::kABytes), &tmap_b, fb, ks * BK_BYTES, n * BN);
#pragma unroll
            for (int j = 0; j < BN / 128; ++j) {
              const uint32_t d = smem_u32(st + C::kABytes + C::kBBytes + C::kSfaBytes + 2048 * j);
              const uint8_t* src = sfb + (int64_t)(n * (BN / 128) + j) * sf_row_stride + (int64_t)ks * 2048;
              bulk_load(d, src, 2048, fb);
            }
            pending |= 1u << s;
            pend_ph = (pend_ph & ~(1u << s)) | (ph << s);
          }
          if (++s == C::kStages) { s = 0; ph ^= 1u; }
        }
      }
      if (ok) {
        // every slot released: no commit arrival is still on its way to this
        // CTA's barriers when it exits
        for (int i = 0; i < C::kStages && ok; ++i) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, &s_abort, timeout_ns)) { fail(); ok = false; break; }
          if (++s == C::kStages) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {
        // drain: the copies of every stage issued here land before the CTA exits
        const uint64_t t0 = globaltimer();
        for (int ss = 0; ss < C::kStages; ++ss) {
          if (!(pending & (1u << ss))) continue;
          const uint32_t par = (pend_ph >> ss) & 1u;
          while (!mbar_try_wait(full_bar(ss), par) && globaltimer() - t0 < 50000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = ue8m0 ? idesc_nvf4(BM, BN, true) : idesc_nvf4(BM, BN);
      // Descriptors of stage 0; a stage's descriptors differ only in the start
      // address field (bits 0-13, address >> 4), so each is this base plus the
      // stage offset >> 4 (shared addresses stay below 2^18: no carry out).
      const uint32_t base = smem_u32(smem);
      const uint64_t da0 = smem_desc(base, 16, 1024, 2);
      const uint64_t db0 = smem_desc(base + C::kABytes, 16, 1024, 2);
      const uint32_t sf_base = tmem + C::kSfBase;
      int s = 0;
      uint32_t ph = 0, acc_ph = 0;
      bool ok = true;
      bool issued_any = false;
      for (int gi = cid; gi < num_tiles && ok; gi += ncl) {
        if (!mbar_wait(tmem_empty, acc_ph ^ 1u, &s_abort, timeout_ns)) { fail(); ok = false; break; }
        tc_fence_after();
        for (int ks = 0; ks < nk; ++ks) {
          // the stage's scales in TMEM (their writers saw the stage land)
          if (!mbar_wait(sfull_bar(s), ph, &s_abort, timeout_ns)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint64_t off = (uint64_t)(s * (C::kStageBytes >> 4));
          const uint32_t sf_col = sf_base + s * C::kSfStageCols;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tc_mma_nvf4(tmem, da0 + off + 2 * j, db0 + off + 2 * j, idesc, sf_col + 4 * j,
                        sf_col + C::kSfaCols + (BN / 128) * 4 * j, (ks | j) != 0 ? 1u : 0u);
          }
          issued_any = true;
          tc_commit(empty_bar(s));
          if (++s == C::kStages) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tmem_full);
        acc_ph ^= 1u;
      }
      if (!ok && issued_any) {
        // drain: wait (bounded) until every MMA issued so far has completed
        tc_commit(drain_bar);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < 50000000ull) {
        }
      }
    }
  } else if (warp >= kScaleWarp) {
    // ---------------- scale writers ----------------
    // Warp w reaches TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31 only; lane l of
    // each writes the 16-byte row l of every 512-byte scale tile of the stage
    // into its lane: A's four K chunks at columns 4 j + c, then B's (BN / 128
    // tiles per chunk) at kSfaCols + (BN / 128) 4 j + 4 h + c. The stage's slot
    // is free when the stage lands (its TMA followed the MMAs that last read it).
    constexpr int NB = BN / 128;
    const uint32_t quad = (uint32_t)(warp & 3);
    int s = 0;
    uint32_t ph = 0;
    for (int gi = cid; gi < num_tiles; gi += ncl) {
      bool ok = true;
      for (int ks = 0; ks < nk; ++ks) {
        // the warp leaves together (the TMEM stores below are warp-collective)
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(full_bar(s), ph, &s_abort, timeout_ns))) { fail(); ok = false; break; }
        const uint8_t* raw = smem + s * C::kStageBytes + C::kABytes + C::kBBytes;
        uint32_t va[16], vb[16 * NB];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 u = *reinterpret_cast<const uint4*>(raw + 512 * j + 16 * lane);
          va[4 * j] = u.x; va[4 * j + 1] = u.y; va[4 * j + 2] = u.z; va[4 * j + 3] = u.w;
#pragma unroll
          for (int h = 0; h < NB; ++h) {
            const uint4 w = *reinterpret_cast<const uint4*>(raw + C::kSfaBytes + 2048 * h + 512 * j + 16 * lane);
            uint32_t* d = vb + 4 * NB * j + 4 * h;
            d[0] = w.x; d[1] = w.y; d[2] = w.z; d[3] = w.w;
          }
        }
        const uint32_t taddr = tmem + ((32u * quad) << 16) + (uint32_t)(C::kSfBase + s * C::kSfStageCols);
        tmem_st16(taddr, va);
        if constexpr (NB == 2) {
          tmem_st32(taddr + C::kSfaCols, vb);
        } else {
          tmem_st16(taddr + C::kSfaCols, vb);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfull_bar(s));
        if (++s == C::kStages) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    const int q = warp & 3;                    // TMEM lane quadrant this warp may access
    const int hcol = (warp - 2) >> 2;          // which half of the tile's columns
    constexpr int kCols = BN / 2;
    constexpr int kParts = kCols / 64;         // read 64 columns at a time (64 registers live)
    const float alpha = __fmul_rn(__ldg(g_a), __ldg(g_b));
    uint32_t acc_ph = 0;
    for (int gi = cid; gi < num_tiles; gi += ncl) {
      const int m = gi / num_n, n = gi % num_n;
      if (!mbar_wait(tmem_full, acc_ph, &s_abort, timeout_ns)) { fail(); break; }
      tc_fence_after();
      const int row = m * BM + q * 32 + lane;
      const int col0 = n * BN + hcol * kCols;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(hcol * kCols);
      uint32_t r[64], hpk[32];
#pragma unroll
      for (int part = 0; part < kParts; ++part) {
        tmem_ld32_async(tbase + 64 * part, r);
        tmem_ld32_async(tbase + 64 * part + 32, r + 32);
        tmem_ld_wait();
        reg_fence32(r);
        reg_fence32(r + 32);
        if (part == kParts - 1) {
          // the accumulator is in registers: the next tile's MMAs may overwrite it
          tc_fence_before();
          mbar_arrive(tmem_empty);
        }
        if constexpr (OUT_F32) {
          float4* out = reinterpret_cast<float4*>(static_cast<float*>(y) + (int64_t)row * N + col0 + 64 * part);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            out[i] = make_float4(__fmul_rn(__uint_as_float(r[4 * i]), alpha),
                                 __fmul_rn(__uint_as_float(r[4 * i + 1]), alpha),
                                 __fmul_rn(__uint_as_float(r[4 * i + 2]), alpha),
                                 __fmul_rn(__uint_as_float(r[4 * i + 3]), alpha));
        } else {
          uint32_t h[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(r[2 * k]), alpha),
                                                            __fmul_rn(__uint_as_float(r[2 * k + 1]), alpha));
            h[k] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          if (part + 1 < kParts) {
#pragma unroll
            for (int k = 0; k < 32; ++k) hpk[k] = h[k];
          } else {
            uint4* out = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(y) + (int64_t)row * N + col0);
            if (kParts == 2) {
#pragma unroll
              for (int i = 0; i < 8; ++i) out[i] = make_uint4(hpk[4 * i], hpk[4 * i + 1], hpk[4 * i + 2], hpk[4 * i + 3]);
              out += 8;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) out[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
          }
        }
      }
      acc_ph ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---- the CTA-pair kernel (tcgen05 cta_group::2) ----------------------------------------
// Two CTAs of a cluster (ranks 0 and 1, on the two SMs of a pair) compute one
// 256 x 256 tile of Y together: rank r holds rows [128 r, 128 r + 128) of the
// tile's A rows and of its B rows (the B tile is split along N), the scales of
// its own A rows, and the scales of all 256 B rows. One thread of rank 0 issues
// every MMA for both (cta_group::2): each instruction reads the shared memory
// of both CTAs at the same offsets, and the TMEM of both (scales and
// accumulator), so each SM takes in half of B per multiply-add instead of all
// of it. Each CTA's TMEM holds its 128 rows x 256 columns of the accumulator
// and the scales of its stages.
//
// Hand-offs between the two CTAs (no multicast):
//   rank 1's stage ready (TMA landed, its scales in its TMEM) -> rank 1 warp 1
//     relays it to rank 0's pfull[s]
//   rank 0's MMA thread commits each stage to empty[s] of both CTAs (two
//     unicast commits) and each finished tile to tfull of both CTAs
//   every epilogue warp of both CTAs -> rank 0's tempty (accumulator read out)
// The relays are relaxed arrivals: each hands on an event the relaying thread
// has observed complete within its own CTA (the stage's TMA bytes counted in
// by the mbarrier and the writers' TMEM stores finished (tcgen05.wait::st,
// then tcgen05.fence::before_thread_sync and an arrival on a CTA barrier); or
// a warp's TMEM reads finished, tcgen05.wait::ld). A release at cluster scope measured ~0.8 us per arrival
// here, which the stage time cannot afford.
//
// Scale factors: the block-scaled MMA reads each operand's scales from TMEM.
// Four writer warps per CTA, one per 32-lane TMEM quadrant (a warp reaches
// only the lanes of quadrant warp % 4), put each stage's scales there with
// tcgen05.st once the stage has landed: lane l of each writes the 16-byte row
// l of every 512-byte scale tile (128 rows x 64 K elements, the layout the
// quantiser writes) into its own lane of the quadrant, so each quadrant holds
// the whole 32-row pattern. Moving the scales with tcgen05.cp instead (one
// thread, in the MMA issuer's stream) measured 292 us at 8192^3 against 212
// us this way: each copy took tensor-pipe time from the MMAs. A stage's TMEM
// slot is free when the stage lands, since its TMA was issued only after the
// MMAs that last read the slot had completed.
// Every wait is bounded, as in the one-CTA kernel.
struct PairCfg {
  static constexpr int kStages = 5;
  static constexpr int kABytes = 128 * BK_BYTES;          // this CTA's 128 rows of A
  static constexpr int kBBytes = 128 * BK_BYTES;          // this CTA's 128 rows of B
  static constexpr int kSfaBytes = 2048;                  // its A rows' scales: 4 K chunks x 512 B
  static constexpr int kSfbBytes = 4096;                  // all 256 B rows' scales
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kSfaCols = 16;
  static constexpr int kSfbCols = 32;
  static constexpr int kSfStageCols = kSfaCols + kSfbCols;
  static constexpr int kSfBase = 256;                     // accumulator: columns [0, 256)
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
  static constexpr int kScaleWarps = 4;                   // scale writers: one per TMEM lane quadrant
  static constexpr int kThreads = 64 + 32 * kEpiWarps + 32 * kScaleWarps;
  static constexpr int kScaleWarp = 2 + kEpiWarps;
  static_assert(kSfBase + kStages * kSfStageCols <= kTmemCols, "TMEM budget");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};


template <bool OUT_F32>
__global__ void __launch_bounds__(PairCfg::kThreads, 1)
gemm_nvf4_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                      const uint8_t* __restrict__ sfa, const uint8_t* __restrict__ sfb,
                      const float* __restrict__ g_a, const float* __restrict__ g_b, void* __restrict__ y,
                      int M, int N, int K, Workspace* ws, uint64_t timeout_ns, int skip_first_stage,
                      int ue8m0) {
  using C = PairCfg;
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::kStageBytes);
  // bars[0..S): full, [S..2S): pfull, [2S..3S): empty, 3S: tfull, 3S+1: tempty, 3S+2: drain,
  // 3S+3+s: rfull[s] (the scales of stage s written into this CTA's TMEM)
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = (int)cluster_id_x(), npairs = (int)cluster_count_x();
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto pfull_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto empty_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
  const uint32_t tfull = bar0 + 8u * (3 * S);
  const uint32_t tempty = bar0 + 8u * (3 * S + 1);
  const uint32_t drain_bar = bar0 + 8u * (3 * S + 2);
  auto rfull_bar = [&](int r) { return bar0 + 8u * (3 * S + 3 + r); };

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(pfull_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 2 * kEpiWarps);
    mbar_init(drain_bar, 1);
    for (int r = 0; r < S; ++r) mbar_init(rfull_bar(r), C::kScaleWarps);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    // one warp of each CTA of the pair allocates, collectively, in both TMEMs
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(&s_tmem_base)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // both CTAs' barriers exist before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tmem = s_tmem_base;

  const int num_n = N / 256;
  const int num_tiles = (M / 256) * num_n;
  const int nk = K / BK;
  const int64_t sf_row_stride = (int64_t)(K / 64) * 512;   // bytes per 128-row scale tile row

  auto fail = [&]() {
    if (!s_abort) {
      s_abort = 1;
      atomicOr(&ws->status, kStatusTimeout);
    }
  };

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t pending = 0, pend_ph = 0;
      bool ok = true;
      for (int t = pair; t < num_tiles && ok; t += npairs) {
        const int pm = t / num_n, n = t % num_n;
        const int arow = pm * 256 + (int)rank * 128;
        const int brow = n * 256 + (int)rank * 128;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, &s_abort, timeout_ns)) { fail(); ok = false; break; }
          const bool skip = skip_first_stage && rank == 0 && pair == 0 && t == pair && ks == 0;
          pending &= ~(1u << s);
          if (!skip) {
            uint8_t* st = smem + s * C::kStageBytes;
            const uint32_t fb = full_bar(s);
            mbar_arrive_expect_tx(fb, C::kStageBytes);
            tma_load_2d(smem_u32(st), &tmap_a, fb, ks * BK_BYTES, arow);
            tma_load_2d(smem_u32(st + C::kABytes), &tmap_b, fb, ks * BK_BYTES, brow);
            bulk_load(smem_u32(st + C::kABytes + C::kBBytes),
                      sfa + (int64_t)(arow / 128) * sf_row_stride + (int64_t)ks * 2048, 2048, fb);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              bulk_load(smem_u32(st + C::kABytes + C::kBBytes + C::kSfaBytes + 2048 * h),
                        sfb + (int64_t)(n * 2 + h) * sf_row_stride + (int64_t)ks * 2048, 2048, fb);
            pending |= 1u << s;
            pend_ph = (pend_ph & ~(1u << s)) | (ph << s);
          }
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
      if (ok) {
        // every slot released: no commit is still on its way to this CTA's
        // barriers when it exits
        for (int i = 0; i < S && ok; ++i) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, &s_abort, timeout_ns)) { fail(); ok = false; break; }
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {
        const uint64_t t0 = globaltimer();
        for (int ss = 0; ss < S; ++ss) {
          if (!(pending & (1u << ss))) continue;
          const uint32_t par = (pend_ph >> ss) & 1u;
          while (!mbar_try_wait(full_bar(ss), par) && globaltimer() - t0 < 50000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 1) {
      // ---------------- rank 1: hand each landed stage to rank 0 ----------------
      // (its A, B and scales: the scale writers waited for the stage's copies)
      const uint32_t peer_pfull0 = peer_addr(pfull_bar(0), 0);
      int s = 0;
      uint32_t ph = 0;
      for (int t = pair; t < num_tiles; t += npairs) {
        bool ok = true;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(rfull_bar(s), ph, &s_abort, timeout_ns)) { fail(); ok = false; break; }
          mbar_arrive_remote(peer_pfull0 + 8u * s);
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
      }
    } else if (lane == 0) {
      // ---------------- rank 0: MMA issuer for the pair ----------------
      const uint32_t idesc = ue8m0 ? idesc_nvf4(256, 256, true) : idesc_nvf4(256, 256);
      const uint32_t base = smem_u32(smem);
      const uint64_t da0 = smem_desc(base, 16, 1024, 2);
      const uint64_t db0 = smem_desc(base + C::kABytes, 16, 1024, 2);
      const uint32_t sf_base = tmem + C::kSfBase;
      const uint32_t peer_empty0 = peer_addr(empty_bar(0), 1);
      const uint32_t peer_tfull = peer_addr(tfull, 1);
      int s = 0;
      uint32_t ph = 0, acc_ph = 0;
      bool ok = true, issued_any = false;
      for (int t = pair; t < num_tiles && ok; t += npairs) {
        if (!mbar_wait_cluster(tempty, acc_ph ^ 1u, &s_abort, timeout_ns)) { fail(); ok = false; break; }
        tc_fence_after();
        for (int ks = 0; ks < nk; ++ks) {
          // this CTA's scales in TMEM (its writers saw the stage land), then rank 1's stage
          if (!mbar_wait(rfull_bar(s), ph, &s_abort, timeout_ns) ||
              !mbar_wait_cluster(pfull_bar(s), ph, &s_abort, timeout_ns)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint64_t off = (uint64_t)(s * (C::kStageBytes >> 4));
          const uint32_t sf_col = sf_base + s * C::kSfStageCols;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc2_mma_nvf4(tmem, da0 + off + 2 * j, db0 + off + 2 * j, idesc, sf_col + 4 * j,
                         sf_col + C::kSfaCols + 8 * j, (ks | j) != 0 ? 1u : 0u);
          issued_any = true;
          tc2_commit(empty_bar(s));
          tc2_commit(peer_empty0 + 8u * s);
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc2_commit(tfull);
        tc2_commit(peer_tfull);
        acc_ph ^= 1u;
      }
      if (!ok && issued_any) {
        tc2_commit(drain_bar);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < 50000000ull) {
        }
      }
    }
  } else if (warp >= C::kScaleWarp) {
    // ---------------- scale writers (both CTAs) ----------------
    // Warp w may access TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31 only; the
    // four writers cover the four quadrants. Lane l of each writes, into 48
    // columns of its lane 32 (w % 4) + l, the 16-byte row l of each 512-byte
    // scale tile: A's four K chunks (columns 4 j + c), then per K chunk both
    // 128-row halves of B's (columns 16 + 8 j + 4 h + c). The slot of stage s
    // is free when the stage lands: its TMA was issued after the MMAs that
    // read the slot before had completed.
    const uint32_t quad = (uint32_t)(warp & 3);
    int s = 0;
    uint32_t ph = 0;
    for (int t = pair; t < num_tiles; t += npairs) {
      bool ok = true;
      for (int ks = 0; ks < nk; ++ks) {
        // the warp leaves together (the TMEM stores below are warp-collective)
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(full_bar(s), ph, &s_abort, timeout_ns))) { fail(); ok = false; break; }
        const uint8_t* raw = smem + s * C::kStageBytes + C::kABytes + C::kBBytes;
        uint32_t va[16], vb[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 u = *reinterpret_cast<const uint4*>(raw + 512 * j + 16 * lane);
          va[4 * j] = u.x; va[4 * j + 1] = u.y; va[4 * j + 2] = u.z; va[4 * j + 3] = u.w;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 w = *reinterpret_cast<const uint4*>(raw + C::kSfaBytes + 2048 * h + 512 * j + 16 * lane);
            vb[8 * j + 4 * h] = w.x; vb[8 * j + 4 * h + 1] = w.y; vb[8 * j + 4 * h + 2] = w.z; vb[8 * j + 4 * h + 3] = w.w;
          }
        }
        const uint32_t taddr = tmem + ((32u * quad) << 16) + (uint32_t)(C::kSfBase + s * C::kSfStageCols);
        tmem_st16(taddr, va);
        tmem_st32(taddr + C::kSfaCols, vb);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(rfull_bar(s));
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
    }
  } else {
    // ---------------- epilogue (warps 2..9 of both CTAs) ----------------
    const int q = warp & 3;
    const int hcol = (warp - 2) >> 2;
    constexpr int kCols = 128;
    const float alpha = __fmul_rn(__ldg(g_a), __ldg(g_b));
    const uint32_t tempty0 = rank == 0 ? tempty : peer_addr(tempty, 0);
    uint32_t acc_ph = 0;
    for (int t = pair; t < num_tiles; t += npairs) {
      const int pm = t / num_n, n = t % num_n;
      if (!mbar_wait(tfull, acc_ph, &s_abort, timeout_ns)) { fail(); break; }
      tc_fence_after();
      const int row = pm * 256 + (int)rank * 128 + q * 32 + lane;
      const int col0 = n * 256 + hcol * kCols;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(hcol * kCols);
      // two halves of 64 columns (64 registers live at a time): the first is
      // packed (BF16) or stored (FP32) before the second is read; the
      // accumulator is released after the second read
      uint32_t r[64], hpk[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        tmem_ld32_async(tbase + 64 * half, r);
        tmem_ld32_async(tbase + 64 * half + 32, r + 32);
        tmem_ld_wait();
        reg_fence32(r);
        reg_fence32(r + 32);
        if (half == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (rank == 0) mbar_arrive(tempty0);
            else mbar_arrive_remote(tempty0);
          }
        }
        if constexpr (OUT_F32) {
          float4* out = reinterpret_cast<float4*>(static_cast<float*>(y) + (int64_t)row * N + col0 + 64 * half);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            out[i] = make_float4(__fmul_rn(__uint_as_float(r[4 * i]), alpha),
                                 __fmul_rn(__uint_as_float(r[4 * i + 1]), alpha),
                                 __fmul_rn(__uint_as_float(r[4 * i + 2]), alpha),
                                 __fmul_rn(__uint_as_float(r[4 * i + 3]), alpha));
        } else {
          uint32_t h[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(r[2 * k]), alpha),
                                                            __fmul_rn(__uint_as_float(r[2 * k + 1]), alpha));
            h[k] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          if (half == 0) {
#pragma unroll
            for (int k = 0; k < 32; ++k) hpk[k] = h[k];
          } else {
            uint4* out = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(y) + (int64_t)row * N + col0);
#pragma unroll
            for (int i = 0; i < 8; ++i) out[i] = make_uint4(hpk[4 * i], hpk[4 * i + 1], hpk[4 * i + 2], hpk[4 * i + 3]);
#pragma unroll
            for (int i = 0; i < 8; ++i) out[8 + i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
          }
        }
      }
      acc_ph ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // no cross-CTA arrival or shared-memory read is still under way
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---- host side ----------------------------------------------------------------------
// 2-D map over a rows x (K/2)-byte code matrix; box = `box_rows` rows x 128 bytes.
bool make_code_map(CUtensorMap* map, const void* base, int64_t rows, int64_t kbytes, int box_rows) {
  return encode_tiled_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, (uint64_t)kbytes, (uint64_t)rows,
                         (uint64_t)kbytes, BK_BYTES, (uint32_t)box_rows);
}

template <int BN, bool OUT_F32>
cudaError_t launch(const GemmArgs& a, uint64_t timeout_ns, int skip, cudaStream_t s) {
  using C = Cfg<BN>;
  CUtensorMap ma, mb;
  if (!make_code_map(&ma, a.a.codes, a.m, a.k / 2, BM) || !make_code_map(&mb, a.b.codes, a.n, a.k / 2, BN))
    return cudaErrorInvalidValue;
  auto k = gemm_nvf4_kernel<BN, OUT_F32>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  // one persistent CTA per SM
  const int tiles = (int)((a.m / BM) * (a.n / BN));
  const int grid = tiles < sm_count() ? tiles : sm_count();
  k<<<grid, kThreads, C::kSmem, s>>>(ma, mb, (const uint8_t*)a.a.scales, (const uint8_t*)a.b.scales,
                                     (const float*)a.a.tensor_scale, (const float*)a.b.tensor_scale, a.y,
                                     (int)a.m, (int)a.n, (int)a.k, static_cast<Workspace*>(a.ws), timeout_ns,
                                     skip, a.fmt == 0 ? 0 : 1);
  return cudaGetLastError();
}

// The pair kernel: clusters of two CTAs, as many pairs as can be resident.
template <bool OUT_F32>
cudaError_t launch_pair(const GemmArgs& a, uint64_t timeout_ns, int skip, cudaStream_t s) {
  using C = PairCfg;
  CUtensorMap ma, mb;
  if (!make_code_map(&ma, a.a.codes, a.m, a.k / 2, 128) || !make_code_map(&mb, a.b.codes, a.n, a.k / 2, 128))
    return cudaErrorInvalidValue;
  auto k = gemm_nvf4_pair_kernel<OUT_F32>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
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
  const int tiles = (int)((a.m / 256) * (a.n / 256));
  if (tiles < pairs) pairs = tiles;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  e = cudaLaunchKernelEx(&cfg, k, ma, mb, (const uint8_t*)a.a.scales, (const uint8_t*)a.b.scales,
                         (const float*)a.a.tensor_scale, (const float*)a.b.tensor_scale, a.y, (int)a.m,
                         (int)a.n, (int)a.k, static_cast<Workspace*>(a.ws), timeout_ns, skip,
                         a.fmt == 0 ? 0 : 1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t run_gemm_ex(const GemmArgs& a, uint64_t timeout_ns, int skip_first_stage, cudaStream_t s) {
  // NVFP4 (E4M3 scales) or the MXFP4 formats on 32- or 16-element blocks
  // (E8M0 scales; a 32-element block's scale is stored for both halves)
  if (a.fmt != 0 && a.fmt != 1 && a.fmt != 4 && a.fmt != 5) return cudaErrorNotSupported;
  const bool f32 = a.out_dtype == 1;
  if (a.m % 256 == 0 && a.n % 256 == 0)
    return f32 ? launch_pair<true>(a, timeout_ns, skip_first_stage, s)
               : launch_pair<false>(a, timeout_ns, skip_first_stage, s);
  if (a.n % 256 == 0) return f32 ? launch<256, true>(a, timeout_ns, skip_first_stage, s)
                                 : launch<256, false>(a, timeout_ns, skip_first_stage, s);
  return f32 ? launch<128, true>(a, timeout_ns, skip_first_stage, s)
             : launch<128, false>(a, timeout_ns, skip_first_stage, s);
}

cudaError_t run_gemm(const GemmArgs& a, cudaStream_t s) {
  return run_gemm_ex(a, kDefaultTimeoutNs, 0, s);
}

}  // namespace fp4q
