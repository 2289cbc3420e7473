/*
 * fp4q.h -- block-scaled 4-bit quantisation of GEMM operands and the
 * block-scaled FP4 GEMM, as a C ABI over hand-written sm_103a CUDA kernels.
 *
 * Method sources (page title, section):
 *   [UFP4]  "Replanteamiento del Sesgo de Contraccion en el Preentrenamiento de
 *           LLM en FP4": Metodologia §1 (E2M1 grid, RTNE, shrinkage bias
 *           (l_i - r_i)/2, RHT), §2 (uniform E1M2 grid, stochastic rounding,
 *           RHT on FPROP/DGRAD/WGRAD), Eficiencia (RHT fused into quantisation).
 *   [TJ2]   "TetraJet-v2: Accurate NVFP4 Training for Large Language Models with
 *           Oscillation Suppression and Outlier Control": Riepilogo Tecnico §2A
 *           (NVFP4 16-element groups with an 8-bit scale, stochastic rounding
 *           E[round(x)] = x, the transposed operand copy), §2C (RHT on dX, dW).
 *   [MXFP4] "Unveiling the Potential of Quantization with MXFP4: Strategies for
 *           Quantization Error Reduction": Resume technique §2 points 1-2
 *           (MXFP4 32-element blocks with E8M0 scales, NVFP4 16-element blocks
 *           with E4M3 scales), §2B (scale math beside dense tensor-core math).
 *   [NGPT]  "Le Architetture Normalizzate sono Nativamente a 4 Bit": Metodologia
 *           (NVFP4 consumed natively by Blackwell tensor cores; SNR of Y = WX).
 *   [HIF]   "Unleashing Low-Bit Inference on Ascend NPUs: A Comprehensive
 *           Evaluation of HiFloat Formats": Resumen tecnico §2 Metodologia (HiF4:
 *           E6M2 scale per 64 elements, E1M0 factors per 8 and per 4 elements,
 *           E1M2 elements).
 *
 * Conventions shared by every entry point
 *   - Every pointer named "device" is a CUDA device pointer owned by the caller.
 *     The library allocates and frees nothing and keeps no state between calls
 *     other than what the caller's workspace holds.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Work is enqueued asynchronously on it; only fp4q_stats and
 *     fp4q_status synchronise that stream.
 *   - Return value: FP4Q_OK (0) or an FP4Q_E* code. Argument errors are
 *     detected on the host before anything is launched. Device-side conditions
 *     (non-finite input, a bounded wait that ran out) are recorded in the
 *     workspace status word and returned by fp4q_status. Nothing traps or
 *     aborts on the GPU.
 *   - Element order: rows x cols, row-major. Packed codes hold two 4-bit codes
 *     per byte, element 2j in bits 0-3 and element 2j+1 in bits 4-7; bit 3 of a
 *     code is the sign (a value that rounds to zero keeps its sign).
 */
#ifndef FP4Q_H
#define FP4Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- enums and error codes ------------------------------------------------ */

typedef enum {
  FP4Q_NVFP4 = 0, /* E2M1 elements, 16-element blocks, E4M3 block scale, FP32 tensor scale [TJ2 §2A, MXFP4 §2] */
  FP4Q_MXFP4 = 1, /* E2M1 elements, 32-element blocks, E8M0 (power-of-two) block scale [MXFP4 §2]          */
  FP4Q_UFP4  = 2, /* uniform E1M2 levels 0..7, 16-element blocks, E4M3 block scale, FP32 tensor scale [UFP4 §2] */
  FP4Q_NVFP4_2L = 3, /* NVFP4 with the double-block scale [TJ2 §2A]: E2M1 elements, 16-element inner blocks with
                       an E4M3 scale, and an FP32 scale g_o = A_o / (6 * 448) per 128-element outer block along
                       the row (A_o = max |v| over it) in place of the tensor scale: one pass, no tensor amax */
  FP4Q_MXFP4_B16 = 4, /* MXFP4 on 16-element blocks [MXFP4 §2, point 1]: E2M1 elements, E8M0 scale
                       2^e, e = floor(log2 a_b) - 2 (a_b = max |v| over the block), no tensor scale */
  FP4Q_MXFP4_OAS = 5, /* overflow-aware scaling [MXFP4 §2A] on 16-element blocks: E8M0 scale with
                       e = ceil(log2(a_b / 7)), which puts a_b / 2^e in (3.5, 7] instead of [4, 8) */
  FP4Q_MXFP4_MBS = 6, /* static macro-block scaling [MXFP4 §2B]: an FP32 scale S with 8 mantissa bits per
                       128-element macro block along the row, S = A_M / 6 rounded to nearest (ties to even) on
                       the 8-fraction-bit grid (A_M = max |v| over the macro block), and 16-element E8M0 blocks
                       under it: e = floor(log2(a_b * (1/S))) - 2, y = (v * (1/S)) * 2^-e */
  FP4Q_HIF4 = 7       /* HiF4 three-level scale [HIF §2], block 64: per 64-element block along the block axis an
                       unsigned E6M2 scale S (bias 31, subnormals, all codes finite) = the value nearest
                       a_64 / 7 (ties to the even code, saturating at 1.75 * 2^32); per 8-element sub-block a
                       bit d_8 and per 4-element micro-block a bit d_4 that halve the step, set when no value of
                       the group would then exceed 7: d_8 = [RN(a_8 / S) <= 3.5], d_4 = [RN(a_4 / S) * 2^(d_8+1)
                       <= 7], with a_g = max |v| over the group and a / S formed as a * RN(1/S); elements on the
                       uniform levels 0..7 (E1M2 in units of 1/4), y = RN(v * RN(1/S)) * 2^(d_8 + d_4). The
                       page gives the structure only: this reading of it is the library's */
} fp4q_format;

typedef enum { FP4Q_RTNE = 0, FP4Q_SR = 1 } fp4q_rounding;
typedef enum { FP4Q_BF16 = 0, FP4Q_F32 = 1 } fp4q_dtype;

enum { FP4Q_ROWWISE = 1, FP4Q_COLWISE = 2 };            /* axis bit mask            */
/* Flag OR-ed into fp4q_quantize's `axis`: the tensor amax was already recorded
 * in the workspace by fp4q_amax (same src, shape, fmt, rht, seed and axis
 * bits), so the call runs the quantisation pass alone. */
enum { FP4Q_AMAX_READY = 4 };
enum { FP4Q_SCALES_LINEAR = 0, FP4Q_SCALES_MMA = 1 };   /* block-scale byte layout  */

enum {
  FP4Q_OK = 0,
  FP4Q_EINVAL = 1,     /* bad enum, shape, alignment, null pointer or small workspace   */
  FP4Q_ENOTSUP = 2,    /* valid request this library does not implement                */
  FP4Q_ECUDA = 3,      /* a CUDA runtime/driver call or a kernel launch failed          */
  FP4Q_ENONFINITE = 4, /* (status) a NaN or an infinity was read by a quantise kernel   */
  FP4Q_ETIMEOUT = 5    /* (status) a bounded wait inside a GEMM kernel ran out          */
};

/* One quantised copy. All pointers are device pointers owned by the caller.
 *   codes        rows x cols/2 bytes (packed nibbles, row-major).
 *   scales       FP4Q_SCALES_LINEAR: rows x cols/block bytes, row-major.
 *                FP4Q_SCALES_MMA: the tiled layout read by the block-scaled
 *                tensor-core MMA, one scale per 16 elements along the row
 *                (vector kv = c / 16): tiles of 128 rows x 4 vectors stored as
 *                512 contiguous bytes, tiles ordered vector-index fastest;
 *                inside a tile the scale of (row r, vector kv) sits at byte
 *                (r % 32) * 16 + ((r % 128) / 32) * 4 + kv % 4. Rows are padded
 *                to a multiple of 128 and vectors per row to a multiple of 4;
 *                padding bytes are written as 0. A 32-element block (FP4Q_MXFP4)
 *                has its scale at both of its vectors. Size: fp4q_scales_bytes().
 *                NVFP4/UFP4/NVFP4_2L scales are E4M3 codes; the MXFP4 formats'
 *                scales are E8M0 codes (exponent + 127).
 *                FP4Q_HIF4 (linear only): one little-endian uint32 word per
 *                64-element block, rows x cols/64 words (4-byte aligned): the
 *                E6M2 code in bits 0-7, d_8 of sub-block j (elements 8j .. 8j+7
 *                of the block) in bit 8 + j, d_4 of micro-block i (elements
 *                4i .. 4i+3) in bit 16 + i. Element value: level(code) * S *
 *                2^-(d_8 + d_4).
 *   tensor_scale one FP32 (device): g = amax / (Qmax * 448) for NVFP4 (Qmax 6)
 *                and UFP4 (Qmax 7, levels in integer units), 1.0 for
 *                FP4Q_MXFP4, FP4Q_MXFP4_B16, FP4Q_MXFP4_OAS and FP4Q_HIF4.
 *                FP4Q_NVFP4_2L: rows x cols/128 FP32 values (row-major), the
 *                outer-block scales g_o; element (r, c) uses g_o(r, c / 128).
 *                FP4Q_MXFP4_MBS: rows x cols/128 FP32 macro scales S, used the
 *                same way. With FP4Q_SCALES_MMA these per-128 scales are stored
 *                column-major instead: cols/128 x rows, (r, c) at c * rows + r
 *                (one K chunk's scales of consecutive rows contiguous, as the
 *                GEMM reads them).
 *   scale_layout FP4Q_SCALES_LINEAR or FP4Q_SCALES_MMA.
 * The value of element (r, c) is level(code) * scale(r, c / block) * g. */
typedef struct {
  uint8_t* codes;
  uint8_t* scales;
  float* tensor_scale;
  int scale_layout;
} fp4q_qtensor;

/* Statistics of one quantised copy ([UFP4] Metodologia §1 and Resultados).
 *   shrink_bias  mean over all n elements of (|q| - |y|) / Qmax, where y is the
 *                element after normalisation by its block (and tensor) scale and
 *                q its grid level: the mean signed rounding error in normalised
 *                magnitude.
 *   snr_db       10 log10(sum v^2 / sum (v - v_hat)^2), v the (transformed)
 *                value and v_hat its dequantised value; +inf when no error.
 *   sum_sig2, sum_err2, sum_bias  the underlying sums (sum_bias in grid units).
 *   n            element count. */
typedef struct {
  double shrink_bias;
  double snr_db;
  double sum_sig2;
  double sum_err2;
  double sum_bias;
  int64_t n;
} fp4q_stats_t;

/* ---- workspace -------------------------------------------------------------- */

/* Bytes of device workspace every call below needs (a fixed size, a few
 * hundred KB). The workspace holds the tensor amaxes, the statistics, the
 * cross-block counters and the status word. It must be zero-filled once
 * before its first use (fp4q_workspace_init); every call leaves its counters
 * back at zero. Calls that share one workspace must not overlap on the GPU. */
size_t fp4q_workspace_size(void);

/* Zero-fill a workspace of fp4q_workspace_size() bytes on `stream`. */
int fp4q_workspace_init(void* workspace, void* stream);

/* Bytes of the scale array of one copy with `rows` rows of `cols` elements in
 * blocks of `block`, for the given layout (FP4Q_SCALES_MMA counts one scale
 * per 16 elements whatever the block). Block 64 (FP4Q_HIF4): 4 bytes per
 * block in the linear layout, 0 for FP4Q_SCALES_MMA (not supported). */
size_t fp4q_scales_bytes(int64_t rows, int64_t cols, int block, int scale_layout);

/* ---- quantisation ------------------------------------------------------------ */

/* The first of fp4q_quantize's two passes on its own: the tensor amax A of
 * each requested copy (max |v| over the copy, v after the RHT when `rht`),
 * which sets the FP32 tensor scale g = A / (Qmax * 448) of NVFP4 and UFP4
 * ([TJ2] Riepilogo Tecnico §2A: NVFP4 block scales under a per-tensor scale).
 * The amaxes are recorded in `workspace`; a following fp4q_quantize call on
 * the same workspace with FP4Q_AMAX_READY in its `axis` then skips this pass.
 * Splitting the call lets a caller time or schedule the two passes apart.
 * The MXFP4 formats, FP4Q_NVFP4_2L and FP4Q_HIF4 have no tensor scale: the
 * call validates its arguments and launches nothing. Arguments and errors as for fp4q_quantize (no outputs). */
int fp4q_amax(const void* src, int dtype, int64_t rows, int64_t cols, int fmt, int block,
              int rht, uint64_t seed, int axis, void* workspace, size_t ws_bytes, void* stream);

/* Quantise a rows x cols tensor into block-scaled 4-bit copies.
 *
 * Operation (per copy; [UFP4] Metodologia §1-2, Eficiencia; [TJ2] §2A, §2C;
 * [MXFP4] §2): widen to FP32; if `rht`, apply v = (1/4) H16 diag(sigma) x to
 * every 16 consecutive elements along the block axis (H16 Sylvester, sigma a
 * seeded +-1 vector: bit j of word 0 of Philox4x32-10(key = seed, counter =
 * (0, 0, 0, 0xFFFFFFFF)), one vector for the whole call), as the FP32
 * butterfly with stages 1, 2, 4, 8 then * 0.25. NVFP4/UFP4: A = max |v| over
 * the copy, g = A / (Qmax * 448), per block t = a_b / (Qmax * g) rounded to
 * E4M3 (nearest-even, saturating at 448), r_b = 1 / (s_b * g), y = v * r_b.
 * MXFP4: e_b = floor(log2 a_b) - 2 clamped to [-127, 127], y = v * 2^-e_b
 * (FP4Q_MXFP4_OAS: e_b = ceil(log2(a_b / 7)); FP4Q_MXFP4_MBS, FP4Q_HIF4: see
 * the enum).
 * y is rounded onto the grid: FP4Q_RTNE nearest level ties to the even code,
 * values beyond the top level saturate; FP4Q_SR rounds |y| up from its lower
 * neighbouring level iff u < f, f the fractional position between the two
 * levels and u = (w >> 8) * 2^-24, w word (i mod 4) of Philox4x32-10(key =
 * seed, counter = (i/4 low, i/4 high, axis, 0)), i the element's row-major
 * index inside the copy, axis 0 for the row-wise copy and 1 for the
 * column-wise copy. Statistics per copy are fused (fp4q_stats).
 *
 * Arguments
 *   src          device, rows x cols elements of `dtype` (FP4Q_BF16 or
 *                FP4Q_F32), row-major, 16-byte aligned.
 *   fmt, block   FP4Q_MXFP4 with block 32, FP4Q_HIF4 with block 64, every
 *                other format with block 16 (else FP4Q_ENOTSUP).
 *                FP4Q_NVFP4_2L and FP4Q_MXFP4_MBS: cols % 128 == 0 for the
 *                row-wise copy, rows % 128 == 0 for the column-wise copy.
 *                FP4Q_HIF4: linear scales only (FP4Q_SCALES_MMA ->
 *                FP4Q_ENOTSUP), scale words 4-byte aligned.
 *   rht          0 or 1. rounding: FP4Q_RTNE or FP4Q_SR. seed: RHT signs and SR.
 *   axis         FP4Q_ROWWISE: blocks along rows, copy row_out (rows x cols).
 *                FP4Q_COLWISE: blocks along columns, emitted transposed into
 *                col_out (cols x rows: codes cols x rows/2, scales per column).
 *                Both bits: both copies from one read of src. May also carry
 *                FP4Q_AMAX_READY (see fp4q_amax).
 *   row_out, col_out  host pointers to fp4q_qtensor descriptors of device
 *                buffers; the one whose axis bit is clear may be NULL. codes
 *                must be 16-byte aligned; MMA-layout scales 16-byte aligned.
 *   workspace    device, ws_bytes >= fp4q_workspace_size(), zero-filled once.
 * Shapes: cols % 16 == 0 always (rows of src start on 32-byte boundaries),
 * cols % block == 0 for the row-wise copy, rows % block == 0 for the
 * column-wise copy; rows or cols 0 is valid (writes g = 0 for NVFP4/UFP4 and
 * empty statistics). Errors: FP4Q_EINVAL, FP4Q_ENOTSUP, FP4Q_ECUDA. */
int fp4q_quantize(const void* src, int dtype, int64_t rows, int64_t cols,
                  int fmt, int block, int rht, int rounding, uint64_t seed, int axis,
                  const fp4q_qtensor* row_out, const fp4q_qtensor* col_out,
                  void* workspace, size_t ws_bytes, void* stream);

/* fp4q_quantize without a workspace argument, for callers that cannot
 * allocate device memory: runtimes and plugins that must live inside a memory
 * pool fixed at start-up, or latency-critical code that cannot afford
 * cudaMalloc/cudaFree, which may synchronise the whole device. The method
 * pages have no counterpart: this is a calling convention, not a step of the
 * method.
 *
 * The scratch the two quantisation passes need lives in a 128 KiB array
 * (`static __device__`) inside the library, which every GPU that loads the
 * library holds until the process exits. The call itself allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine); the caller still
 * allocates src and the output buffers. The first call on each device looks
 * up the array's device address (cudaGetSymbolAddress) with that device
 * current, so make that first call before any stream capture. Every call
 * clears the status word and the counters of the array, then runs exactly
 * what fp4q_quantize runs; the device status it records (non-finite input,
 * a bounded wait that ran out) is read by fp4q_status_noalloc, while its
 * statistics stay in the array and are not readable (use fp4q_quantize with
 * a workspace for them).
 * All calls on a device share the one array: calls that overlap on the GPU
 * (other streams, other threads) race and must be serialised by the caller.
 * Arguments, outputs and errors as for fp4q_quantize, except that
 * FP4Q_AMAX_READY is rejected (FP4Q_EINVAL: there is no workspace to carry
 * an earlier fp4q_amax result), and FP4Q_EINVAL if the library's scratch
 * requirement (fp4q_workspace_size()) exceeds the 128 KiB array. */
int fp4q_quantize_noalloc(const void* src, int dtype, int64_t rows, int64_t cols,
                          int fmt, int block, int rht, int rounding, uint64_t seed, int axis,
                          const fp4q_qtensor* row_out, const fp4q_qtensor* col_out,
                          void* stream);

/* fp4q_status for fp4q_quantize_noalloc's library-owned scratch (no paper
 * counterpart: a calling convention). Synchronises `stream`, returns the
 * device status the no-allocation calls on the current device recorded since
 * the previous call of this function or since their last start (each
 * fp4q_quantize_noalloc call clears it), FP4Q_OK, FP4Q_ENONFINITE or
 * FP4Q_ETIMEOUT, and clears it. Allocates nothing. FP4Q_ECUDA if the lookup
 * of the scratch or the synchronisation failed. */
int fp4q_status_noalloc(void* stream);

/* Dequantise one copy ([UFP4] §2: UFP4 has no tensor-core format and is
 * consumed through this call): v_hat = (level * s_b) * g in FP32, two
 * round-to-nearest products in that order (MXFP4 formats: level * 2^e_b,
 * FP4Q_MXFP4_MBS: (level * 2^e_b) * S); if
 * `inverse_rht`, apply R^T = (1/4) diag(sigma) H16 per 16-block along the row
 * (the same FP32 butterfly, then * 0.25, then the sign flip). Writes rows x
 * cols elements of `dst_dtype` (BF16 rounded to nearest-even, or FP32) to the
 * device buffer `dst` (16-byte aligned). q is a host pointer to a descriptor of
 * device buffers laid out as fp4q_quantize wrote them for a copy of rows x
 * cols. FP4Q_NVFP4_2L: g is the outer-block scale of the element, cols %
 * 128 == 0; FP4Q_MXFP4_MBS likewise with the macro scale. FP4Q_HIF4:
 * v_hat = level * (S * 2^-(d_8 + d_4)), exact in FP32. Errors: FP4Q_EINVAL, FP4Q_ENOTSUP, FP4Q_ECUDA. */
int fp4q_dequantize(const fp4q_qtensor* q, int64_t rows, int64_t cols, int fmt, int block,
                    int inverse_rht, uint64_t seed, void* dst, int dst_dtype, void* stream);

/* Statistics of the last fp4q_quantize call that used `workspace`
 * ([UFP4] Metodologia §1 shrinkage bias, Resultados SQNR). Synchronises
 * `stream`, then fills the host structs row_stats / col_stats (either may be
 * NULL; a copy that was not produced reads n = 0). Errors: FP4Q_EINVAL,
 * FP4Q_ECUDA. */
int fp4q_stats(const void* workspace, fp4q_stats_t* row_stats, fp4q_stats_t* col_stats,
               void* stream);

/* Synchronise `stream`, return the device status recorded in `workspace` since
 * the previous fp4q_status call (FP4Q_OK, FP4Q_ENONFINITE or FP4Q_ETIMEOUT;
 * timeout wins) and clear it. FP4Q_ECUDA if the synchronisation failed. */
int fp4q_status(void* workspace, void* stream);

/* ---- code utilisation ----------------------------------------------------------- */

/* Histogram of the 4-bit codes of one copy ([UFP4] Resultados: the RHT raises
 * the effective bucket ratio of both grids). q->codes: device, rows x cols/2
 * packed bytes as fp4q_quantize wrote them (16-byte aligned; q's scales and
 * tensor scale are not read). counts: device array of 16 unsigned 64-bit
 * integers, 8-byte aligned, overwritten with the number of elements carrying
 * each code 0..15 (bit 3 the sign, bits 0-2 the level). Asynchronous on
 * `stream`. Errors: FP4Q_EINVAL (null or misaligned pointers, negative sizes,
 * odd cols), FP4Q_ECUDA. */
int fp4q_code_histogram(const fp4q_qtensor* q, int64_t rows, int64_t cols, unsigned long long* counts,
                        void* stream);

/* Effective bucket ratio of a code histogram (host array of 16 counts):
 * exp(H) / 8, H = -sum p_l ln p_l over the 8 levels (a code and its negative
 * count together): 1 when the 8 levels are used equally, 1/8 when one level
 * holds every element, 0 for an empty histogram. */
double fp4q_effective_bucket_ratio(const unsigned long long* counts);

/* ---- block-scaled GEMM --------------------------------------------------------- */

/* Y = dequant(A) * dequant(B)^T on the tensor cores ([NGPT] Metodologia: NVFP4
 * consumed natively by Blackwell tensor cores; [MXFP4] §2B: scale factors
 * applied beside the dense MMA; [UFP4] Resultados: single-GEMM output of the
 * quantised operands). A is M x K and B is N x K, both row-wise copies of
 * format `fmt` (blocks along K) with FP4Q_SCALES_MMA scales; the K-block
 * products are accumulated in FP32 by tcgen05 block-scaled MMAs (E4M3 or E8M0
 * scale per 16 elements) and the result is multiplied by g_A * g_B. When both operands were quantised with the RHT
 * along K under the same seed, the transforms cancel (R R^T = I).
 *   A, B       host pointers to descriptors of device buffers.
 *   fmt        FP4Q_NVFP4, FP4Q_MXFP4, FP4Q_MXFP4_B16 or FP4Q_MXFP4_OAS
 *              ([MXFP4] §2: the MX formats' E8M0 scales on the same MMA);
 *              FP4Q_NVFP4_2L and FP4Q_MXFP4_MBS ([TJ2] §2A, [MXFP4] §2B):
 *              their FP32 per-128 scales change along K, so each 128-element
 *              K chunk's product is formed apart in TMEM and scaled by
 *              g_A(m, c) g_B(n, c) into FP32 accumulators (tensor_scale:
 *              the column-major per-128 scales, 16-byte aligned).
 *              FP4Q_UFP4 (no tensor-core format holds its levels): runs as
 *              fp4q_gemm_dequant, with that call's shape rules; so does
 *              FP4Q_HIF4 ([HIF] §2: no tensor-core format takes its scales).
 *   Y          device, M x N row-major, `out_dtype` FP4Q_BF16 (nearest-even)
 *              or FP4Q_F32, 16-byte aligned.
 *   workspace  as for fp4q_quantize (the status word records a bounded wait
 *              that ran out: FP4Q_ETIMEOUT via fp4q_status).
 * Shapes: M % 128 == 0, N % 128 == 0, K % 256 == 0, all > 0 (else FP4Q_EINVAL).
 * M and N multiples of 256 run on pairs of SMs (the two-SM MMA), others on
 * single SMs; the results are the same.
 * Errors: FP4Q_EINVAL, FP4Q_ENOTSUP, FP4Q_ECUDA. */
int fp4q_gemm(const fp4q_qtensor* A, const fp4q_qtensor* B, int64_t M, int64_t N, int64_t K,
              int fmt, void* Y, int out_dtype, void* workspace, size_t ws_bytes, void* stream);

/* Y = dequant(A) * dequant(B)^T on the tensor cores for block-scaled formats
 * whose values the block-scaled MMA cannot take: UFP4 ([UFP4] Metodologia §2
 * and Resultados: the uniform grid with the RHT on every training GEMM) and
 * HiF4 ([HIF] §2; values level * S * 2^-(d_8 + d_4), exact in BF16); NVFP4
 * and the E8M0 formats (FP4Q_MXFP4, FP4Q_MXFP4_B16, FP4Q_MXFP4_OAS) are
 * accepted too, to compare with fp4q_gemm. The kernel's converter warps turn
 * each operand's codes and block scales into the 16-bit block values
 * level * s_b in shared memory -- FP16 for UFP4 and NVFP4 (E4M3 scales; exact:
 * at most 7 significant bits in [2^-10, 3136]), BF16 for the E8M0 formats
 * and HiF4 (exact) -- and tcgen05.mma.kind::f16 accumulates their products, exact in
 * FP32, in FP32; the result is multiplied by g_A * g_B (their FP32 product;
 * 1 for the E8M0 formats). No dequantised operand is written to memory. When
 * both operands were quantised with the RHT along K under the same seed, the
 * transforms cancel.
 *   A, B       host pointers to descriptors of row-wise copies (M x K, N x K)
 *              of format `fmt`, linear or tiled scales (2-byte aligned; HiF4:
 *              linear scale words, 4-byte aligned, else FP4Q_ENOTSUP /
 *              FP4Q_EINVAL).
 *   Y          device, M x N row-major, FP4Q_BF16 (nearest-even) or FP4Q_F32,
 *              16-byte aligned.
 *   workspace  as for fp4q_gemm (FP4Q_ETIMEOUT via fp4q_status).
 * Shapes: M, N > 0 (any; rows past a 128 x 256 tile are zeros), N % 8 == 0,
 * K > 0, K % 64 == 0 (else FP4Q_EINVAL).
 * Errors: FP4Q_EINVAL, FP4Q_ENOTSUP (FP4Q_NVFP4_2L, FP4Q_MXFP4_MBS: their
 * per-128 scales are not one 16-bit value per element), FP4Q_ECUDA. */
int fp4q_gemm_dequant(const fp4q_qtensor* A, const fp4q_qtensor* B, int64_t M, int64_t N, int64_t K,
                      int fmt, void* Y, int out_dtype, void* workspace, size_t ws_bytes, void* stream);

/* Test hook for the device-side failure path (not a step of the method): runs
 * fp4q_gemm with the producer of the first CTA withholding the first stage of
 * its first tile and every wait bounded by `timeout_ns`, so the waits that
 * depend on that stage run out. The kernel records FP4Q_ETIMEOUT in the
 * workspace status word, lets the copies it issued land, frees its Tensor
 * Memory and returns; nothing traps, and the CUDA context stays usable (the
 * output Y is then incomplete). Arguments as fp4q_gemm; 1 ms <= timeout_ns
 * <= 10 s (else FP4Q_EINVAL). */
int fp4q_gemm_selftest_timeout(const fp4q_qtensor* A, const fp4q_qtensor* B, int64_t M, int64_t N,
                               int64_t K, int fmt, void* Y, int out_dtype, void* workspace,
                               size_t ws_bytes, uint64_t timeout_ns, void* stream);

/* ---- misc ----------------------------------------------------------------------- */

/* Static text for an FP4Q_* code. */
const char* fp4q_strerror(int code);

/* Library version as major * 10000 + minor * 100 + patch. */
int fp4q_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP4Q_H */
