// Block-scaled FP4 GEMM for operands with an FP32 scale per 128 elements along
// K (sm_103a): two-level NVFP4 ("TetraJet-v2 ...", Riepilogo Tecnico §2A: an
// FP32 scale per 128-element outer block over 16-element E4M3 blocks) and
// MBS-static ("Unveiling the Potential of Quantization with MXFP4 ...", Resume
// technique §2B: a scale with 8 mantissa bits per 128-element macro block over
// 16-element E8M0 blocks, the scale math beside the dense tensor-core math).
//
// Y[m][n] = sum_c gA[m][c] gB[n][c] P_c[m][n], where P_c is the block-scaled
// product of K chunk c (128 elements). The per-128 scales change along K, so
// they cannot be applied once after the accumulation: each chunk's P_c is
// accumulated on its own in TMEM (two MMAs of K = 64), and the epilogue warps
// take it out of TMEM, scale it by gA gB and add it to FP32 accumulators held
// in registers, while the tensor cores work on the next chunks in the others
// of three TMEM buffers.
//
// Structure (one persistent CTA per SM, 576 threads):
//   warp 0      TMA producer: per K stage of 256 elements, the A and B code
//               tiles (2-D TMA, 128B swizzle), their block-scale tiles and the
//               per-128 scales of the tile's rows for the stage's two chunks
//               (1-D bulk copies) into a 4-deep shared-memory ring. A slot is
//               refilled once the MMAs (a commit) and the epilogue (which
//               reads the per-128 scales there) have both released it.
//   warp 1      allocates 512 TMEM columns; one thread copies each stage's
//               scale tiles into TMEM (tcgen05.cp 32x128b.warpx4) and, per
//               128-element chunk, issues two block-scaled MMAs (M = N = 128,
//               K = 64) into accumulator buffer (chunk % 3), then commits the
//               buffer to the epilogue.
//   warps 2-17  epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 and
//               columns 32 ((w - 2) / 4) .. +31 of the buffer (16x256b
//               shape: a thread holds 4 rows x 8 columns), releases it, and
//               accumulates P gA gB in registers (packed FP32x2); after a
//               tile's last chunk each thread stores its 32 values (BF16 or
//               FP32).
// The per-128 scales are read in the tiled layout: column-major, (K/128) x
// rows, so one chunk's scales of consecutive rows are contiguous. Bound
// (measured on B300 at 8192^3): the mainloop with 128 x 128 tiles and a commit
// per chunk takes 643 us even with no epilogue arithmetic; the epilogue adds
// about 100 us. Register accumulators cap the tile at 128 x 128 (a 128 x 256
// tile would need the whole register file), and wider TMEM accumulators leave
// no room for two buffers. Every wait
// is bounded by a global-timer deadline; on expiry the kernel records
// FP4Q_ETIMEOUT in the workspace, drains what it issued and returns.
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

constexpr int BM = 128;                 // rows of A per tile (= MMA M)
constexpr int BN = 128;                 // rows of B per tile (= MMA N)
constexpr int BK = 256;                 // K elements per stage
constexpr int BK_BYTES = 128;           // code bytes per row per stage
constexpr int CHUNK = 128;              // K elements per outer scale
constexpr int kStages = 4;
constexpr int kEpiWarps = 16;           // four per TMEM lane quadrant
constexpr int kEpiCols = BN * 4 / kEpiWarps;   // accumulator columns per epilogue warp (32)
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kTmemCols = 512;
constexpr int kABytes = BM * BK_BYTES;
constexpr int kBBytes = BN * BK_BYTES;
constexpr int kSfBytes = 2048;          // 128 rows x 16 scales (one stage)
constexpr int kGBytes = 2 * 128 * 4;    // the per-128 scales of the stage's two chunks, 128 rows
constexpr int kGaOff = kABytes + kBBytes + 2 * kSfBytes;
constexpr int kGbOff = kGaOff + kGBytes;
constexpr int kStageBytes = kGbOff + kGBytes;
constexpr int kSfStageCols = 32;        // A: 4 x 4 TMEM columns, then B: 4 x 4
constexpr int kAccBufs = 3;             // chunk accumulators: the MMAs run up to two chunks ahead
constexpr int kSfBase = kAccBufs * BN;  // accumulator buffers in columns [0, 384)
constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
constexpr uint64_t kTimeoutNs = 2000000000ull;   // 2 s
static_assert(kSfBase + kStages * kSfStageCols <= kTmemCols, "TMEM budget");
static_assert(kStageBytes % 1024 == 0, "stage alignment");
static_assert(kEpiCols % 32 == 0 && kEpiWarps % 4 == 0, "epilogue split");

template <bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
gemm_outer_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                  const uint8_t* __restrict__ sfa, const uint8_t* __restrict__ sfb,
                  const float* __restrict__ ga, const float* __restrict__ gb, void* __restrict__ y,
                  int M, int N, int K, Workspace* ws, uint32_t idesc, uint64_t timeout_ns) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  // bars[0..S): full, [S..2S): empty, 2S + b: acc_full[b], 2S + 3 + b: acc_empty[b], 2S + 6: drain
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto acc_full = [&](uint32_t b) { return bar0 + 8u * (2 * kStages + b); };
  auto acc_empty = [&](uint32_t b) { return bar0 + 8u * (2 * kStages + kAccBufs + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 2 * kAccBufs);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1 + kEpiThreads);     // the MMAs' commit and every epilogue thread
    }
    for (uint32_t b = 0; b < (uint32_t)kAccBufs; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), kEpiThreads);
    }
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
  const int tiles = (M / BM) * num_n;
  const int nk = K / BK;
  const int nch = K / CHUNK;
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
      uint32_t ph = 0, pending = 0, pend_ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int m = t / num_n, n = t % num_n;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, &s_abort, timeout_ns)) { fail(); ok = false; break; }
          uint8_t* st = smem + s * kStageBytes;
          const uint32_t fb = full_bar(s);
          pending &= ~(1u << s);
          mbar_arrive_expect_tx(fb, kStageBytes);
          tma_load_2d(smem_u32(st), &tmap_a, fb, ks * BK_BYTES, m * BM);
          tma_load_2d(smem_u32(st + kABytes), &tmap_b, fb, ks * BK_BYTES, n * BN);
          bulk_load(smem_u32(st + kABytes + kBBytes), sfa + (int64_t)m * sf_row_stride + (int64_t)ks * 2048,
                    kSfBytes, fb);
          bulk_load(smem_u32(st + kABytes + kBBytes + kSfBytes),
                    sfb + (int64_t)n * sf_row_stride + (int64_t)ks * 2048, kSfBytes, fb);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int64_t c = 2 * (int64_t)ks + h;
            bulk_load(smem_u32(st + kGaOff + 512 * h), ga + c * M + (int64_t)m * BM, 512, fb);
            bulk_load(smem_u32(st + kGbOff + 512 * h), gb + c * N + (int64_t)n * BN, 512, fb);
          }
          pending |= 1u << s;
          pend_ph = (pend_ph & ~(1u << s)) | (ph << s);
          if (++s == kStages) { s = 0; ph ^= 1u; }
        }
      }
      if (ok) {
        // every slot released: no commit arrival is still on its way when the CTA exits
        for (int i = 0; i < kStages && ok; ++i) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, &s_abort, timeout_ns)) { fail(); ok = false; break; }
          if (++s == kStages) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {
        // drain: the copies issued here land before the CTA exits
        const uint64_t t0 = globaltimer();
        for (int ss = 0; ss < kStages; ++ss) {
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
      const uint32_t base = smem_u32(smem);
      const uint64_t da0 = smem_desc(base, 16, 1024, 2);
      const uint64_t db0 = smem_desc(base + kABytes, 16, 1024, 2);
      const uint64_t dsa0 = smem_desc(base + kABytes + kBBytes, 128, 128, 0);
      const uint64_t dsb0 = smem_desc(base + kABytes + kBBytes + kSfBytes, 128, 128, 0);
      int s = 0;
      uint32_t ph = 0, gc = 0;
      bool ok = true, issued_any = false;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        for (int ks = 0; ks < nk && ok; ++ks) {
          if (!mbar_wait(full_bar(s), ph, &s_abort, timeout_ns)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint64_t off = (uint64_t)(s * (kStageBytes >> 4));
          const uint32_t sf_col = tmem + kSfBase + s * kSfStageCols;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tc_cp_sf(sf_col + 4 * j, dsa0 + off + 32 * j);
            tc_cp_sf(sf_col + 16 + 4 * j, dsb0 + off + 32 * j);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t b = gc % kAccBufs;
            if (!mbar_wait(acc_empty(b), ((gc / kAccBufs) & 1u) ^ 1u, &s_abort, timeout_ns)) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const int j = 2 * h + jj;
              tc_mma_nvf4(tmem + (uint32_t)(BN * b), da0 + off + 2 * j, db0 + off + 2 * j, idesc, sf_col + 4 * j,
                          sf_col + 16 + 4 * j, (uint32_t)jj);
            }
            issued_any = true;
            tc_commit(acc_full(b));
            ++gc;
          }
          if (!ok) break;
          tc_commit(empty_bar(s));
          if (++s == kStages) { s = 0; ph ^= 1u; }
        }
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
    // ---------------- epilogue (warps 2..17) ----------------
    // Each warp covers the 32 rows of its TMEM lane quadrant and 32 columns of
    // the tile, read as two 16-lane halves with the 16x256b shape: thread t
    // holds rows (t / 4, t / 4 + 8) of each half and columns 8j + 2 (t % 4) +
    // {0, 1}, so it needs 8 column scales per chunk rather than 32.
    const int q = warp & 3;                       // TMEM lane quadrant this warp may access
    const int hc = (warp - 2) >> 2;               // column group of the tile
    const int tr = lane >> 2, tc = 2 * (lane & 3);
    uint32_t gc = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
      const int m = t / num_n, n = t % num_n;
      const int row0 = q * 32 + tr;               // rows row0 + {0, 8, 16, 24} of the tile
      const int c0 = hc * kEpiCols + tc;          // columns c0 + 8j + {0, 1} of the tile
      f2 acc[16];                                 // [half][j][row offset 0 / 8]
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = f2_make(0.f, 0.f);
      bool ok = true;
      for (int c = 0; c < nch; ++c) {
        const uint32_t b = gc % kAccBufs;
        if (!mbar_wait(acc_full(b), (gc / kAccBufs) & 1u, &s_abort, timeout_ns)) { fail(); ok = false; break; }
        tc_fence_after();
        uint32_t r[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          tmem_ld16x256_x4_async(tmem + ((uint32_t)(q * 32 + 16 * hh) << 16) + (uint32_t)(BN * b + hc * kEpiCols),
                                 r + 16 * hh);
        tmem_ld_wait();
        reg_fence16(r);
        reg_fence16(r + 16);
        tc_fence_before();
        mbar_arrive(acc_empty(b));
        // this chunk's per-128 scales, staged with its codes: stage sequence
        // number gc / 2, half gc % 2. That stage's load has completed (the MMAs
        // read it); waiting on its phase makes the copy's writes visible here,
        // and the slot cannot be refilled before this thread releases it below.
        const uint32_t sq = gc >> 1, half = gc & 1u;
        const int stg = (int)(sq % kStages);
        ++gc;
        if (!mbar_wait(full_bar(stg), (sq / kStages) & 1u, &s_abort, timeout_ns)) { fail(); ok = false; break; }
        const uint8_t* st = smem + stg * kStageBytes;
        const float* ga_s = reinterpret_cast<const float*>(st + kGaOff + 512 * (int)half);
        const float* gb_s = reinterpret_cast<const float*>(st + kGbOff + 512 * (int)half);
        float a[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) a[k] = ga_s[row0 + 8 * k];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const float2 w = *reinterpret_cast<const float2*>(gb_s + c0 + 8 * jj);
          const f2 W = f2_make(w.x, w.y);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const float ak = a[2 * hh + k];
              const uint32_t* rr = r + 16 * hh + 4 * jj + 2 * k;
              f2& A = acc[8 * hh + 2 * jj + k];
              A = f2_fma(f2_make(__uint_as_float(rr[0]), __uint_as_float(rr[1])), f2_mul(f2_make(ak, ak), W), A);
            }
          }
        }
        // the stage's second chunk: its per-128 scales are no longer needed
        if (half == 1u) mbar_arrive(empty_bar(stg));
      }
      if (!ok) break;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int64_t row = (int64_t)m * BM + row0 + 16 * hh + 8 * k;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            float v0, v1;
            f2_split(acc[8 * hh + 2 * jj + k], v0, v1);
            const int64_t col = (int64_t)n * BN + c0 + 8 * jj;
            if constexpr (OUT_F32) {
              *reinterpret_cast<float2*>(static_cast<float*>(y) + row * N + col) = make_float2(v0, v1);
            } else {
              *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(y) + row * N + col) =
                  __floats2bfloat162_rn(v0, v1);
            }
          }
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

template <bool OUT_F32>
cudaError_t launch_outer(const GemmArgs& a, uint32_t idesc, cudaStream_t s) {
  CUtensorMap ma, mb;
  if (!encode_tiled_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.a.codes, (uint64_t)(a.k / 2), (uint64_t)a.m,
                       (uint64_t)(a.k / 2), BK_BYTES, BM) ||
      !encode_tiled_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.b.codes, (uint64_t)(a.k / 2), (uint64_t)a.n,
                       (uint64_t)(a.k / 2), BK_BYTES, BN))
    return cudaErrorInvalidValue;
  auto k = gemm_outer_kernel<OUT_F32>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int tiles = (int)((a.m / BM) * (a.n / BN));
  const int grid = tiles < sm_count() ? tiles : sm_count();
  k<<<grid, kThreads, kSmem, s>>>(ma, mb, static_cast<const uint8_t*>(a.a.scales),
                                  static_cast<const uint8_t*>(a.b.scales), static_cast<const float*>(a.a.tensor_scale),
                                  static_cast<const float*>(a.b.tensor_scale), a.y, (int)a.m, (int)a.n, (int)a.k,
                                  static_cast<Workspace*>(a.ws), idesc, kTimeoutNs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t run_gemm_outer(const GemmArgs& a, cudaStream_t s) {
  // two-level NVFP4 (E4M3 inner scales) or MBS (E8M0 inner scales)
  if (a.fmt != 3 && a.fmt != 6) return cudaErrorNotSupported;
  const uint32_t idesc = idesc_nvf4(BM, BN, a.fmt == 6);
  return a.out_dtype == 1 ? launch_outer<true>(a, idesc, s) : launch_outer<false>(a, idesc, s);
}

}  // namespace fp4q
