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
// Structure (one persistent CTA per SM, 320 threads):
//   warp 0      TMA producer: per K stage of 256 elements, one 2-D tiled TMA
//               load (128B swizzle) of the A and B code tiles and 1-D bulk
//               copies of their scale tiles into a 4-deep shared-memory ring
//               (mbarrier transaction counts).
//   warp 1      allocates the 512 TMEM columns; one thread moves each stage's
//               scale tiles into TMEM (tcgen05.cp 32x128b.warpx4) and issues
//               four tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X
//               (M = 128, N = BN, K = 64) into an FP32 accumulator in TMEM;
//               tcgen05.commit frees the ring slot and, after the last stage,
//               hands the accumulator to the epilogue.
//   warps 2-9   epilogue: each warp reads its 32 TMEM lanes x BN/2 columns
//               into registers, releases the accumulator (the next tile's
//               MMAs start), then multiplies by g_A * g_B and stores BF16
//               (nearest-even) or FP32.
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
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kTmemCols = 512;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s

template <int BN>
struct Cfg {
  static constexpr int kStages = 4;
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
  // bars[0..S): full, bars[S..2S): empty, bars[2S]: tmem_full, bars[2S+1]: tmem_empty, bars[2S+2]: drain
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

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
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
      const uint64_t dsa0 = smem_desc(base + C::kABytes + C::kBBytes, 128, 128, 0);
      const uint64_t dsb0 = smem_desc(base + C::kABytes + C::kBBytes + C::kSfaBytes, 128, 128, 0);
      const uint32_t sf_base = tmem + C::kSfBase;
      int s = 0;
      uint32_t ph = 0, acc_ph = 0;
      bool ok = true;
      bool issued_any = false;
      for (int gi = cid; gi < num_tiles && ok; gi += ncl) {
        if (!mbar_wait(tmem_empty, acc_ph ^ 1u, &s_abort, timeout_ns)) { fail(); ok = false; break; }
        tc_fence_after();
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(full_bar(s), ph, &s_abort, timeout_ns)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint64_t off = (uint64_t)(s * (C::kStageBytes >> 4));
          const uint32_t sf_col = sf_base + s * C::kSfStageCols;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tc_cp_sf(sf_col + 4 * j, dsa0 + off + 32 * j);
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tc_cp_sf(sf_col + C::kSfaCols + (BN / 128) * 4 * j + 4 * h, dsb0 + off + 128 * h + 32 * j);
          }
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
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    const int q = warp & 3;                    // TMEM lane quadrant this warp may access
    const int hcol = (warp - 2) >> 2;          // which half of the tile's columns
    constexpr int kCols = BN / 2;
    const float alpha = __fmul_rn(__ldg(g_a), __ldg(g_b));
    uint32_t acc_ph = 0;
    for (int gi = cid; gi < num_tiles; gi += ncl) {
      const int m = gi / num_n, n = gi % num_n;
      if (!mbar_wait(tmem_full, acc_ph, &s_abort, timeout_ns)) { fail(); break; }
      tc_fence_after();
      const int row = m * BM + q * 32 + lane;
      uint32_t r[kCols];
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c)
        tmem_ld32_async(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(hcol * kCols + c * 32), r + 32 * c);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c) reg_fence32(r + 32 * c);
      // the accumulator is in registers: the next tile's MMAs may overwrite it
      tc_fence_before();
      mbar_arrive(tmem_empty);
      acc_ph ^= 1u;
      const int col0 = n * BN + hcol * kCols;
      if constexpr (OUT_F32) {
        float4* out = reinterpret_cast<float4*>(static_cast<float*>(y) + (int64_t)row * N + col0);
#pragma unroll
        for (int i = 0; i < kCols / 4; ++i)
          out[i] = make_float4(__fmul_rn(__uint_as_float(r[4 * i]), alpha),
                               __fmul_rn(__uint_as_float(r[4 * i + 1]), alpha),
                               __fmul_rn(__uint_as_float(r[4 * i + 2]), alpha),
                               __fmul_rn(__uint_as_float(r[4 * i + 3]), alpha));
      } else {
        uint4* out = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(y) + (int64_t)row * N + col0);
#pragma unroll
        for (int i = 0; i < kCols / 8; ++i) {
          uint32_t h[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(r[8 * i + 2 * k]), alpha),
                                                            __fmul_rn(__uint_as_float(r[8 * i + 2 * k + 1]), alpha));
            h[k] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          out[i] = make_uint4(h[0], h[1], h[2], h[3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
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

}  // namespace

cudaError_t run_gemm_ex(const GemmArgs& a, uint64_t timeout_ns, int skip_first_stage, cudaStream_t s) {
  // NVFP4 (E4M3 scales) or the MXFP4 formats on 32- or 16-element blocks
  // (E8M0 scales; a 32-element block's scale is stored for both halves)
  if (a.fmt != 0 && a.fmt != 1 && a.fmt != 4 && a.fmt != 5) return cudaErrorNotSupported;
  const bool f32 = a.out_dtype == 1;
  if (a.n % 256 == 0) return f32 ? launch<256, true>(a, timeout_ns, skip_first_stage, s)
                                 : launch<256, false>(a, timeout_ns, skip_first_stage, s);
  return f32 ? launch<128, true>(a, timeout_ns, skip_first_stage, s)
             : launch<128, false>(a, timeout_ns, skip_first_stage, s);
}

cudaError_t run_gemm(const GemmArgs& a, cudaStream_t s) {
  return run_gemm_ex(a, kDefaultTimeoutNs, 0, s);
}

}  // namespace fp4q
