"""Plain CPU oracle for block-scaled 4-bit quantisation and the block-scaled GEMM.

TEST INFRASTRUCTURE ONLY. This module is the independent reference the CUDA
library is checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the library itself never does, and
this module imports nothing from the library.

Everything here is written for a reader to check by eye against the method:
numpy arrays, FP32 where the method computes in FP32 (every such step is a
single IEEE round-to-nearest numpy operation, in the order stated), FP64 for the
statistics and the GEMM. No blocking, fusion or reordering beyond what each
definition states.

Sources (page title, section):
  [UFP4]  "Replanteamiento del Sesgo de Contracción en el Preentrenamiento de LLM
          en FP4" -- Metodología §1 (shrinkage bias, (l_i - r_i)/2), §2 (uniform
          E1M2/INT4 grid, RHT on all GEMMs, stochastic rounding), Eficiencia
          (fused RHT + FP4 quantisation).
  [NGPT]  "Le Architetture Normalizzate sono Nativamente a 4 Bit" -- Metodologia
          (NVFP4 on Blackwell; SNR of Y = WX).
  [TJ2]   "TetraJet-v2: Accurate NVFP4 Training for Large Language Models ..." --
          Riepilogo Tecnico §2A (NVFP4: 16-element groups, 8-bit scale,
          stochastic rounding with E[round(x)] = x, transposed weight copy), §2C
          (RHT on the backward GEMMs).
  [MXFP4] "Unveiling the Potential of Quantization with MXFP4: Strategies for
          Quantization Error Reduction" -- Résumé technique §2 points 1-2
          (MXFP4: 32-element blocks, E8M0 power-of-two scale; NVFP4: 16-element
          blocks, E4M3 scale), §2A (alpha_max mapped to a power-of-two window).
  [HIF]   "Unleashing Low-Bit Inference on Ascend NPUs: A Comprehensive
          Evaluation of HiFloat Formats" -- Resumen técnico §2 Metodología
          (HiF4: one E6M2 scale per 64 elements, E1M0 factors per 8 and per 4
          elements, E1M2 elements).
  [OCP-MX] OCP Microscaling Formats (MX) v1.0: shared scale exponent
          floor(log2 amax) - emax_elem, emax_elem = 2 for E2M1.
  [PHILOX] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1,
          2, 3", SC'11: the Philox4x32-10 counter-based generator (pinned
          against cuRAND's host generator: see philox4x32_10).

Readings where the pages are silent (each is listed with its reason in the
design notes of the repository):
  R1 RHT = (1/4) * H16 * diag(sigma), H16 Sylvester (natural order), one sign
     vector for the whole tensor and both copies, sigma_j = bit j of one Philox
     word (key = seed, counter = (0, 0, 0, 0xFFFFFFFF)).
  R2 UFP4 levels in integer units 0..7 (E1M2 value k/4 scaled by 4), Qmax = 7,
     tensor scale amax / (7 * 448); codes and block scales are identical to the
     E1M2-unit reading.
  R3 NVFP4/UFP4 normalisation: r_b = 1 / (s_b * g) once per block, y = v * r_b.
  R4 zero keeps its sign in the code (sign bit = sign bit of y).
  R5 stochastic rounding: round up iff u < f, u = (w >> 8) * 2^-24, w one
     Philox word keyed on (seed) with counter (i / 4, axis, 0) picking word
     i mod 4; i = index of the element inside the copy being produced.
  R6 shrinkage bias = mean over elements of (|q| - |y|) / Qmax.
  R14 code utilisation ("effective bucket ratio", [UFP4] Resultados): the
     histogram of the 16 codes of a copy; the effective bucket ratio is
     exp(H) / 8, H the Shannon entropy (natural log) of the distribution of
     the 8 magnitude levels, i.e. the effective number of levels in use over
     the number available.
  R15 the E8M0 variants of [MXFP4] §2A-§2B sit on 16-element blocks (the page
     applies both techniques at block size 16): ``mxfp4_b16`` keeps the OCP
     exponent rule; ``mxfp4_oas`` (overflow-aware scaling) takes the smallest
     power of two 2^e with alpha_max / 2^e <= 7, i.e. e = ceil(log2(alpha_max
     / 7)), which puts alpha_max / 2^e in (3.5, 7] instead of [4, 8).
  R16 MBS-static ([MXFP4] §2B): every macro block of 128 consecutive values
     along the block axis has a scale S with 8 mantissa bits, S = alpha_M / 6
     rounded to nearest (ties to even) on FP32's grid with 8 fraction bits
     (alpha_M = max |v| over the macro block), so the macro block's maximum
     lands on the top level; inside it, each 16-element block gets an E8M0
     exponent by the OCP rule applied to a_b * (1/S), and y = (v * (1/S)) *
     2^-e_b; 1/S is one FP32 reciprocal (0 when S = 0, FLT_MAX if it
     overflows), as r_b is under R3.
  R17 HiF4 ([HIF] §2 gives the structure, not the arithmetic; parity
     unpinned for the reading itself): elements on the uniform E1M2 grid in
     integer units 0..7 (as R2); E6M2 = an unsigned float with 6 exponent and
     2 mantissa bits, bias 31, subnormals, every code finite; per 64-block
     S = E6M2_rne_sat(a_64 / 7), r = 1/S (FP32; 0 if S = 0); an E1M0 factor
     is one bit d that halves the step of its group: d_8 = 1 iff
     RN(a_8 * r) * 2 <= 7, then d_4 = 1 iff RN(a_4 * r) * 2^(d_8 + 1) <= 7
     (a group halves its step whenever none of its values would then clamp);
     y = RN(v * r) * 2^(d_8 + d_4), rounded onto the grid. One 32-bit word per
     64-block: E6M2 code in bits 0-7, d_8 of sub-block j in bit 8 + j, d_4 of
     micro-block i in bit 16 + i.
  R13 two-level NVFP4 (the double-block scale of [TJ2] §2A): every outer block
     of 128 consecutive values along the block axis has its own FP32 scale
     g_o = A_o / (6 * 448), A_o = max |v| over the outer block, in place of the
     tensor scale; the 16-element inner blocks inside it are scaled and rounded
     exactly as NVFP4 is under a tensor scale, with g replaced by g_o.
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------- #
# Element grids                                                               #
# --------------------------------------------------------------------------- #

#: E2M1 magnitudes indexed by the three low code bits (1 sign, 2 exponent,
#: 1 mantissa bit) -- [UFP4] Declaración del Problema / Metodología §1.
E2M1_LEVELS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)

#: UFP4 (uniform E1M2 / INT4-like) magnitudes in integer units, reading R2 --
#: [UFP4] Metodología §2 "Rejilla Uniforme": equal left/right bin widths.
UFP4_LEVELS = np.arange(8, dtype=np.float64)

FORMATS = ("nvfp4", "mxfp4", "ufp4", "mxfp4_b16", "mxfp4_oas")
QMAX = {"nvfp4": 6.0, "mxfp4": 6.0, "ufp4": 7.0, "mxfp4_b16": 6.0, "mxfp4_oas": 6.0}
BLOCK = {"nvfp4": 16, "mxfp4": 32, "ufp4": 16, "mxfp4_b16": 16, "mxfp4_oas": 16}
#: formats whose block scale is an E8M0 power of two (no tensor scale)
E8M0_FORMATS = ("mxfp4", "mxfp4_b16", "mxfp4_oas")
E4M3_MAX = 448.0

F32 = np.float32


def grid_levels(fmt: str) -> np.ndarray:
    return UFP4_LEVELS if fmt == "ufp4" else E2M1_LEVELS


# --------------------------------------------------------------------------- #
# BF16 -> FP32 widening (exact)                                               #
# --------------------------------------------------------------------------- #

def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """BF16 is the top half of an FP32 word: shift the 16 bits up by 16."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """Round FP32 to BF16 (nearest, ties to even); NaN stays a quiet NaN."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    return np.where(nan, np.uint16(0x7FC0), r)


# --------------------------------------------------------------------------- #
# Scale formats                                                               #
# --------------------------------------------------------------------------- #

def e4m3_decode(code) -> np.ndarray:
    """Value of an FP8 E4M3 (bias 7, no infinities) code 0..126, as FP64.

    Exponent field 0 is subnormal (m * 2^-9); otherwise (1 + m/8) * 2^(e-7).
    Largest finite value: e = 15, m = 6 -> 448 ([MXFP4] Résumé technique §2, point 2).
    """
    c = np.asarray(code, dtype=np.int64) & 0x7F
    e = c >> 3
    m = c & 7
    sub = m * 2.0 ** -9
    nrm = (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64))
    return np.where(e == 0, sub, nrm)


#: all 127 finite non-negative E4M3 values, ascending with the code.
E4M3_VALUES = e4m3_decode(np.arange(127))


def _nearest_even(a: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Index into an ascending ``table`` nearest to ``a`` (inside the table's
    range), ties to the even index. ``a`` and ``table`` are FP64 and every
    difference taken here is exact."""
    lo = np.searchsorted(table, a, side="right") - 1
    lo = np.clip(lo, 0, len(table) - 1)
    hi = np.minimum(lo + 1, len(table) - 1)
    d_lo = a - table[lo]
    d_hi = table[hi] - a
    take_hi = (hi != lo) & ((d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0)))
    return np.where(take_hi, hi, lo)


def e4m3_encode_rne_sat(t) -> np.ndarray:
    """FP32 t >= 0 -> E4M3 code: nearest value, ties to even code, values above
    the largest finite value saturate to 448 (no NaN is produced)."""
    a = np.minimum(np.asarray(t, dtype=np.float64), E4M3_MAX)
    return _nearest_even(a, E4M3_VALUES).astype(np.uint8)


def e8m0_exponent(amax) -> np.ndarray:
    """MXFP4 shared exponent of a block: floor(log2 amax) - 2 ([OCP-MX];
    [MXFP4] §2 point 2: power-of-two scale), clamped to the E8M0 range
    [-127, 127]; amax = 0 gives -127. frexp gives amax = m * 2^ex with m in
    [0.5, 1), so floor(log2 amax) = ex - 1 (subnormals included)."""
    a = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(a)
    e = ex.astype(np.int64) - 1 - 2
    e = np.where(a == 0.0, -127, e)
    return np.clip(e, -127, 127)


def e8m0_exponent_oas(amax) -> np.ndarray:
    """Overflow-aware shared exponent ([MXFP4] §2A, reading R15): the smallest
    e with amax / 2^e <= 7, so that amax / 2^e lies in (3.5, 7]. With amax =
    m * 2^ex (frexp, m in [0.5, 1)): amax / 2^(ex-3) = 8m <= 7 iff m <= 7/8,
    giving e = ex - 3, else e = ex - 2. Clamped to [-127, 127]; amax = 0 gives
    -127."""
    a = np.asarray(amax, dtype=np.float64)
    m, ex = np.frexp(a)
    e = np.where(m <= 0.875, ex.astype(np.int64) - 3, ex.astype(np.int64) - 2)
    e = np.where(a == 0.0, -127, e)
    return np.clip(e, -127, 127)


def block_exponent(amax, fmt: str) -> np.ndarray:
    """E8M0 exponent of a block under the format's rule."""
    return e8m0_exponent_oas(amax) if fmt == "mxfp4_oas" else e8m0_exponent(amax)


def mbs_macro_scale(alpha) -> np.ndarray:
    """MBS-static macro-block scale ([MXFP4] §2B, reading R16): alpha / 6
    rounded to nearest, ties to even, on the FP32 grid with 8 fraction bits
    (quantum 2^(E - 8) for alpha / 6 in [2^E, 2^(E+1)), E >= -126; 2^-134 below
    2^-126). alpha / 6 is formed in FP64: for an FP32 alpha it is either exact
    or has a non-terminating binary expansion (alternating bits from the 24th
    significant bit on), so it is never a tie of the 8-bit grid unless exactly
    one, and the FP64 rounding cannot cross one. Returns FP32."""
    t = np.asarray(alpha, dtype=np.float32).astype(np.float64) / 6.0
    _, ex = np.frexp(t)
    quantum = np.exp2((np.maximum(ex.astype(np.int64) - 1, -126) - 8).astype(np.float64))
    return (np.rint(t / quantum) * quantum).astype(np.float32)


# --------------------------------------------------------------------------- #
# Philox4x32-10 [PHILOX]                                                      #
# --------------------------------------------------------------------------- #

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Ten Philox rounds on a 4x32-bit counter under a 2x32-bit key.

    One round: (hi0, lo0) = M0 * c0 and (hi1, lo1) = M1 * c2 as 64-bit
    products; the new counter is (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0).
    Between rounds the key is bumped by the Weyl constants (W0, W1) mod 2^32.
    Inputs broadcast; returns four uint64 arrays holding 32-bit words.
    Pinned word for word against cuRAND's host-side Philox4x32-10 generator
    (an implementation this oracle shares no code with), over several keys
    including all-zero and all-ones and counters whose first three words vary
    (tests/test_oracle_rht_sr.py); the construction's properties (distinct
    outputs, avalanche, uniformity) are checked as well.
    """
    c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(
        *[np.asarray(v, dtype=np.uint64) & _MASK32 for v in (c0, c1, c2, c3, k0, k1)])
    c0, c1, c2, c3, k0, k1 = (v.copy() for v in (c0, c1, c2, c3, k0, k1))
    m0, m1 = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK32
            k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK32
        p0 = m0 * c0
        p1 = m1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def _seed_words(seed: int):
    s = int(seed) & 0xFFFFFFFFFFFFFFFF
    return s & 0xFFFFFFFF, s >> 32


def rht_signs(seed: int) -> np.ndarray:
    """Reading R1: sigma_j = -1 iff bit j of word 0 of
    Philox(key = seed, counter = (0, 0, 0, 0xFFFFFFFF)) is set, j = 0..15."""
    k0, k1 = _seed_words(seed)
    w0 = int(philox4x32_10(0, 0, 0, 0xFFFFFFFF, k0, k1)[0])
    bits = (w0 >> np.arange(16)) & 1
    return np.where(bits == 1, -1.0, 1.0)


def sr_uniforms(index, seed: int, axis: int) -> np.ndarray:
    """Reading R5: the uniform u in [0, 1) used to round element ``index`` of
    copy ``axis`` (0 row-wise, 1 column-wise): u = (w >> 8) * 2^-24 with w word
    (index mod 4) of Philox(key = seed, counter = (index/4 low 32 bits,
    index/4 high 32 bits, axis, 0))."""
    idx = np.asarray(index, dtype=np.int64)
    q = (idx // 4).astype(np.uint64)
    k0, k1 = _seed_words(seed)
    words = philox4x32_10(q & _MASK32, q >> np.uint64(32), axis, 0, k0, k1)
    lane = idx % 4
    w = np.choose(lane, words)
    return (w >> np.uint64(8)).astype(np.float64) * 2.0 ** -24


# --------------------------------------------------------------------------- #
# Random Hadamard Transform (16-point)                                        #
# --------------------------------------------------------------------------- #

def hadamard16() -> np.ndarray:
    """Sylvester Hadamard matrix, natural order: H[i, j] = (-1)^popcount(i & j)."""
    i = np.arange(16)[:, None]
    j = np.arange(16)[None, :]
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    return np.where(pc % 2 == 0, 1.0, -1.0)


_H16 = hadamard16()


def rht_definition(blocks: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """v = (1/4) * H16 * diag(sigma) * x for every 16-vector on the last axis,
    as a dense FP64 product rounded once to FP32 ([UFP4] Metodología §1 and
    Eficiencia; [TJ2] §2C). Input FP32 [..., 16]."""
    x = np.asarray(blocks, dtype=np.float64) * signs
    v = 0.25 * np.einsum("ij,...j->...i", _H16, x)
    return v.astype(np.float32)


def rht_butterfly(blocks: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """The same transform as the fast Walsh-Hadamard butterfly in FP32:
    w = sigma * x (exact), then stages h = 1, 2, 4, 8 replace (w_i, w_{i+h})
    for every i with bit h clear by (w_i + w_{i+h}, w_i - w_{i+h}), each a
    single FP32 rounding, and finally v = 0.25 * w (FP32)."""
    w = (np.asarray(blocks, dtype=np.float32) * signs.astype(np.float32)).astype(np.float32)
    w = w.copy()
    for h in (1, 2, 4, 8):
        idx = np.array([i for i in range(16) if i & h == 0])
        a = w[..., idx].copy()
        b = w[..., idx + h].copy()
        w[..., idx] = a + b
        w[..., idx + h] = a - b
    return (w * F32(0.25)).astype(np.float32)


def rht_inverse_butterfly(blocks: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """Transpose of the RHT, R^T = (1/4) diag(sigma) H16: the same FP32
    butterfly on v, then 0.25 *, then the sign flip."""
    w = np.asarray(blocks, dtype=np.float32).copy()
    for h in (1, 2, 4, 8):
        idx = np.array([i for i in range(16) if i & h == 0])
        a = w[..., idx].copy()
        b = w[..., idx + h].copy()
        w[..., idx] = a + b
        w[..., idx + h] = a - b
    return ((w * F32(0.25)) * signs.astype(np.float32)).astype(np.float32)


def rht_inverse_definition(blocks: np.ndarray, signs: np.ndarray) -> np.ndarray:
    x = np.einsum("ij,...j->...i", _H16, np.asarray(blocks, dtype=np.float64))
    return (0.25 * x * signs).astype(np.float32)


# --------------------------------------------------------------------------- #
# Rounding onto the element grid                                              #
# --------------------------------------------------------------------------- #

def round_rtne(y: np.ndarray, fmt: str) -> np.ndarray:
    """RTNE onto the grid ([UFP4] Metodología §1): |y| is clamped to the
    largest level, then rounded to the nearest level, ties to the level whose
    code is even. Returns 4-bit codes: sign bit (bit 3) from y's sign bit
    (reading R4), level index in bits 0-2."""
    levels = grid_levels(fmt)
    a = np.minimum(np.abs(np.asarray(y, dtype=np.float64)), levels[-1])
    k = _nearest_even(a, levels)
    sign = np.signbit(y).astype(np.uint8)
    return (sign << 3) | k.astype(np.uint8)


def round_sr(y: np.ndarray, fmt: str, u: np.ndarray) -> np.ndarray:
    """Stochastic rounding ([UFP4] §2; [TJ2] §2A, E[round(x)] = x): with
    lo <= |y| < hi adjacent levels and f = (|y| - lo) / (hi - lo), round up iff
    u < f; |y| at or above the top level gives the top level. Sign kept."""
    levels = grid_levels(fmt)
    top = levels[-1]
    a = np.abs(np.asarray(y, dtype=np.float64))
    at_top = a >= top
    lo = np.searchsorted(levels, np.minimum(a, top), side="right") - 1
    hi = np.minimum(lo + 1, 7)
    gap = np.where(hi > lo, levels[hi] - levels[lo], 1.0)
    f = np.where(at_top, 0.0, (a - levels[lo]) / gap)
    up = (~at_top) & (np.asarray(u, dtype=np.float64) < f)
    k = np.where(at_top, 7, lo + up.astype(np.int64))
    sign = np.signbit(y).astype(np.uint8)
    return (sign << 3) | k.astype(np.uint8)


def code_value(codes: np.ndarray, fmt: str) -> np.ndarray:
    """Grid value (FP64) of 4-bit codes."""
    c = np.asarray(codes, dtype=np.int64)
    mag = grid_levels(fmt)[c & 7]
    return np.where(c & 8, -mag, mag)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Two codes per byte along the last axis: element 2j in bits 0-3,
    element 2j+1 in bits 4-7."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# --------------------------------------------------------------------------- #
# Quantisation of one copy                                                    #
# --------------------------------------------------------------------------- #

def _as_f32_matrix(x) -> np.ndarray:
    a = np.asarray(x)
    if a.dtype == np.uint16:
        return bf16_bits_to_f32(a)
    return np.ascontiguousarray(a, dtype=np.float32)


def transform_copy(m32: np.ndarray, fmt: str, rht: bool, seed: int,
                   rht_mode: str = "butterfly") -> np.ndarray:
    """Values v of a copy (rows x cols, blocks along cols), after the optional
    16-point RHT. MXFP4 applies two 16-point transforms per 32-block."""
    if not rht:
        return m32
    n, k = m32.shape
    signs = rht_signs(seed)
    fn = rht_butterfly if rht_mode == "butterfly" else rht_definition
    return fn(m32.reshape(n, k // 16, 16), signs).reshape(n, k)


def tensor_amax(v: np.ndarray) -> np.float32:
    """A = max |v| over the whole copy (FP32)."""
    if v.size == 0:
        return F32(0.0)
    return F32(np.max(np.abs(v)))


def tensor_scale(amax: np.float32, fmt: str) -> np.float32:
    """NVFP4 per-tensor FP32 scale g = A / (Qmax * 448), one FP32 division
    by the exact constant 2688 (NVFP4) or 3136 (UFP4, reading R2); the E8M0
    formats have no tensor scale (1.0)."""
    if fmt in E8M0_FORMATS:
        return F32(1.0)
    return F32(F32(amax) / F32(QMAX[fmt] * E4M3_MAX))


def copy_amax(m32: np.ndarray, fmt: str, rht: bool = False, seed: int = 0,
              rht_mode: str = "butterfly", chunk_rows: int = 256) -> np.float32:
    """Pass 1 of a copy: A = max |v| over every (transformed) value of the
    rows x cols matrix m32, blocks along its columns."""
    amax = F32(0.0)
    for r0 in range(0, m32.shape[0], chunk_rows):
        v = transform_copy(m32[r0:r0 + chunk_rows], fmt, rht, seed, rht_mode)
        if v.size:
            amax = max(amax, tensor_amax(v))
    return amax


def quantize_copy(m32: np.ndarray, fmt: str, rht: bool = False, rounding: str = "rtne",
                  seed: int = 0, axis: int = 0, rht_mode: str = "butterfly",
                  chunk_rows: int = 256, keep_y: bool = False, rows_subset=None,
                  amax=None) -> dict:
    """Quantise one copy: a rows x cols FP32 matrix whose blocks run along the
    columns. For the row-wise copy this is X itself; for the column-wise copy it
    is X^T ([TJ2] §2A: the transposed operand of the weight-gradient GEMM).

    Steps, per block b of ``block`` consecutive values:
      v   = RHT(x) or x
      A   = max |v| over the copy;  g = A / (Qmax * 448)           (FP32)
      a_b = max |v| over the block
      NVFP4/UFP4: d = Qmax * g (FP32, once); t = a_b / d (FP32);
                  s_b = E4M3_rne_sat(t); p = s_b * g (FP32);
                  r_b = 1 / p (FP32; 0 if p = 0, FLT_MAX if it overflows);
                  y = v * r_b (FP32)                                  (reading R3)
                  if g = 0 every scale and code is 0.
      MXFP4:      e_b = floor(log2 a_b) - 2 in [-127, 127]; scale code e_b + 127;
                  y = v * 2^-e_b (FP32); mxfp4_b16 the same on 16-element
                  blocks, mxfp4_oas with e_b = ceil(log2(a_b / 7)) (R15)
      q   = RTNE(y) or SR(y, u_i)
    ``rows_subset`` (row indices of the copy) restricts the codes, scales and
    statistics to those rows; the tensor amax still covers the whole copy.
    ``amax``: the copy's tensor amax when pass 1 already ran (copy_amax over
    the whole copy); m32 may then hold only some of the copy's rows.
    Statistics (FP64): bias = sum(|q| - |y|) / (Qmax * N)   (reading R6)
                       snr_db = 10 log10(sum v^2 / sum (v - v_hat)^2), v_hat =
                       q * s_b * g (or q * 2^e_b) exactly in FP64.
    """
    if fmt not in FORMATS:
        raise ValueError(fmt)
    b = BLOCK[fmt]
    n, k = m32.shape
    if k % b:
        raise ValueError("cols must be a multiple of the block size")
    qmax = QMAX[fmt]
    levels_top = grid_levels(fmt)[-1]
    assert levels_top == qmax

    # Pass 1: the tensor amax over every transformed value of the copy.
    if amax is None:
        amax = copy_amax(m32, fmt, rht, seed, rht_mode, chunk_rows)
    amax = F32(amax)
    g = tensor_scale(amax, fmt)
    d = F32(F32(qmax) * g)

    sel = np.arange(n) if rows_subset is None else np.asarray(rows_subset, dtype=np.int64)
    ns = sel.size
    codes = np.zeros((ns, k), dtype=np.uint8)
    scales = np.zeros((ns, k // b), dtype=np.uint8)
    ys = np.zeros((ns, k), dtype=np.float32) if keep_y else None
    sum_bias = 0.0
    sum_abs_bias = 0.0
    sum_sig2 = 0.0
    sum_err2 = 0.0
    for r0 in range(0, ns, chunk_rows):
        ridx = sel[r0:r0 + chunk_rows]
        v = transform_copy(m32[ridx], fmt, rht, seed, rht_mode)
        rows = v.shape[0]
        vb = v.reshape(rows, k // b, b)
        a_b = np.max(np.abs(vb), axis=2).astype(np.float32)
        if fmt in E8M0_FORMATS:
            e_b = block_exponent(a_b, fmt)
            scales[r0:r0 + rows] = (e_b + 127).astype(np.uint8)
            mult = np.exp2(-e_b.astype(np.float64)).astype(np.float32)
            y = (vb * mult[..., None]).astype(np.float32)
            step64 = np.exp2(e_b.astype(np.float64))
        else:
            if g == 0.0:
                s_code = np.zeros_like(a_b, dtype=np.uint8)
            else:
                t = (a_b / d).astype(np.float32)
                s_code = e4m3_encode_rne_sat(t)
            scales[r0:r0 + rows] = s_code
            s_val = e4m3_decode(s_code).astype(np.float32)
            p = (s_val * g).astype(np.float32)
            with np.errstate(divide="ignore", over="ignore"):
                r_b = np.where(p == 0.0, F32(0.0), (F32(1.0) / p)).astype(np.float32)
            r_b = np.where(np.isinf(r_b), np.finfo(np.float32).max, r_b).astype(np.float32)
            y = (vb * r_b[..., None]).astype(np.float32)
            step64 = s_val.astype(np.float64) * np.float64(g)
        y = y.reshape(rows, k)
        if rounding == "rtne":
            c = round_rtne(y, fmt)
        elif rounding == "sr":
            idx = ridx[:, None] * k + np.arange(k, dtype=np.int64)[None, :]
            c = round_sr(y, fmt, sr_uniforms(idx, seed, axis))
        else:
            raise ValueError(rounding)
        codes[r0:r0 + rows] = c
        if keep_y:
            ys[r0:r0 + rows] = y
        qv = code_value(c, fmt)
        term = np.abs(qv) - np.abs(y.astype(np.float64))
        sum_bias += float(np.sum(term))
        sum_abs_bias += float(np.sum(np.abs(term)))
        vhat = (qv.reshape(rows, k // b, b) * step64[..., None]).reshape(rows, k)
        v64 = v.astype(np.float64)
        sum_sig2 += float(np.sum(v64 * v64))
        sum_err2 += float(np.sum((v64 - vhat) ** 2))

    nel = ns * k
    out = {
        "fmt": fmt, "block": b, "rows": ns, "cols": k, "rows_subset": rows_subset,
        "codes": pack_nibbles(codes),
        "scales": scales,
        "tensor_scale": F32(g),
        "amax": F32(amax),
        "stats": stats_from_sums(sum_bias, sum_abs_bias, sum_sig2, sum_err2, nel, qmax),
    }
    if keep_y:
        out["y"] = ys
    return out


#: outer block of the two-level NVFP4 scale ([TJ2] Riepilogo Tecnico §2A).
OUTER_BLOCK = 128


def quantize_copy_two_level(m32: np.ndarray, rht: bool = False, rounding: str = "rtne",
                            seed: int = 0, axis: int = 0, rht_mode: str = "butterfly",
                            rows_subset=None) -> dict:
    """NVFP4 with the double-block scale ([TJ2] Riepilogo Tecnico §2A, reading
    R13): "an outer block of 128 elements is scaled globally, the inner blocks
    of 16 locally", which avoids the whole-tensor amax. Per copy row (blocks
    along the columns), per outer block o of 128 values and inner block b of 16:
      v   = RHT(x) or x
      A_o = max |v| over the outer block;  g_o = A_o / (6 * 448)       (FP32)
      d_o = 6 * g_o (FP32); t = a_b / d_o (FP32); s_b = E4M3_rne_sat(t);
      p = s_b * g_o (FP32); r_b = 1 / p (FP32; 0 if p = 0, FLT_MAX if it
      overflows); y = v * r_b (FP32); if g_o = 0 the outer block's scales and
      codes are all 0
      q   = RTNE(y) or SR(y, u_i) on the E2M1 grid
    Returns codes and inner scales as NVFP4 does, and ``outer_scales`` (FP32,
    rows x cols/128) in place of the tensor scale. Statistics as for NVFP4
    with v_hat = q * s_b * g_o (FP64)."""
    n, k = m32.shape
    if k % OUTER_BLOCK:
        raise ValueError("cols must be a multiple of the outer block (128)")
    sel = np.arange(n) if rows_subset is None else np.asarray(rows_subset, dtype=np.int64)
    v = transform_copy(np.ascontiguousarray(m32[sel]), "nvfp4", rht, seed, rht_mode)
    rows = v.shape[0]
    no, nb = k // OUTER_BLOCK, OUTER_BLOCK // 16
    vb = v.reshape(rows, no, nb, 16)
    a_o = np.max(np.abs(vb), axis=(2, 3)).astype(np.float32) if rows else np.zeros((0, no), np.float32)
    g_o = (a_o / F32(6.0 * E4M3_MAX)).astype(np.float32)
    d_o = (F32(6.0) * g_o).astype(np.float32)
    a_b = np.max(np.abs(vb), axis=3).astype(np.float32) if rows else np.zeros((0, no, nb), np.float32)
    zero = (g_o == 0.0)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (a_b / d_o[..., None]).astype(np.float32)
    s_code = np.where(zero, 0, e4m3_encode_rne_sat(np.where(zero, F32(0.0), t))).astype(np.uint8)
    s_val = e4m3_decode(s_code).astype(np.float32)
    p = (s_val * g_o[..., None]).astype(np.float32)
    with np.errstate(divide="ignore", over="ignore"):
        r_b = np.where(p == 0.0, F32(0.0), (F32(1.0) / p)).astype(np.float32)
    r_b = np.where(np.isinf(r_b), np.finfo(np.float32).max, r_b).astype(np.float32)
    y = (vb * r_b[..., None]).astype(np.float32).reshape(rows, k)
    if rounding == "rtne":
        c = round_rtne(y, "nvfp4")
    elif rounding == "sr":
        idx = sel[:, None] * k + np.arange(k, dtype=np.int64)[None, :]
        c = round_sr(y, "nvfp4", sr_uniforms(idx, seed, axis))
    else:
        raise ValueError(rounding)
    qv = code_value(c, "nvfp4")
    term = np.abs(qv) - np.abs(y.astype(np.float64))
    step64 = s_val.astype(np.float64) * g_o.astype(np.float64)[..., None]
    vhat = (qv.reshape(rows, no, nb, 16) * step64[..., None]).reshape(rows, k)
    v64 = v.astype(np.float64)
    stats = stats_from_sums(float(np.sum(term)), float(np.sum(np.abs(term))), float(np.sum(v64 * v64)),
                            float(np.sum((v64 - vhat) ** 2)), rows * k, QMAX["nvfp4"])
    return {"fmt": "nvfp4_2l", "block": 16, "rows": rows, "cols": k, "rows_subset": rows_subset,
            "codes": pack_nibbles(c), "scales": s_code.reshape(rows, k // 16),
            "outer_scales": g_o, "stats": stats}


def dequantize_two_level(codes_packed: np.ndarray, scales: np.ndarray, outer_scales: np.ndarray,
                         inverse_rht: bool = False, seed: int = 0) -> np.ndarray:
    """v_hat = (q * s_b) * g_o in FP32, two round-to-nearest products in that
    order, g_o the scale of the element's outer block of 128; optionally
    followed by R^T (FP32 butterfly)."""
    c = unpack_nibbles(codes_packed)
    n, k = c.shape
    q = code_value(c, "nvfp4").astype(np.float32).reshape(n, k // 16, 16)
    s_val = e4m3_decode(scales).astype(np.float32)
    g = np.repeat(np.asarray(outer_scales, dtype=np.float32), OUTER_BLOCK // 16, axis=1)
    v = ((q * s_val[..., None]).astype(np.float32) * g[..., None]).astype(np.float32).reshape(n, k)
    if inverse_rht:
        v = rht_inverse_butterfly(v.reshape(n, k // 16, 16), rht_signs(seed)).reshape(n, k)
    return v


#: macro block of MBS-static ([MXFP4] Résumé technique §2B)
MACRO_BLOCK = 128


def quantize_copy_mbs(m32: np.ndarray, rht: bool = False, rounding: str = "rtne",
                      seed: int = 0, axis: int = 0, rht_mode: str = "butterfly",
                      rows_subset=None) -> dict:
    """MXFP4 with the static macro-block scale ([MXFP4] Résumé technique §2B,
    reading R16): a scale with 8 mantissa bits per macro block of 128 values,
    E8M0 scales per 16-element block under it. Per copy row, macro block M and
    16-element block b inside it:
      v   = RHT(x) or x
      alpha_M = max |v| over M;  S = RN8(alpha_M / 6)                  (FP32)
      rS  = 1 / S (FP32; 0 if S = 0, FLT_MAX if it overflows)
      a_b = max |v| over b;  a1 = a_b * rS (FP32);  e_b = floor(log2 a1) - 2
            in [-127, 127] (a1 = 0 gives -127); scale code e_b + 127
      w   = v * rS (FP32);  y = w * 2^-e_b (exact)
      q   = RTNE(y) or SR(y, u_i) on the E2M1 grid
    Returns codes and E8M0 scale codes, and ``macro_scales`` (FP32, rows x
    cols/128). Statistics as for MXFP4 with v_hat = q * 2^e_b * S (FP64)."""
    n, k = m32.shape
    if k % MACRO_BLOCK:
        raise ValueError("cols must be a multiple of the macro block (128)")
    sel = np.arange(n) if rows_subset is None else np.asarray(rows_subset, dtype=np.int64)
    v = transform_copy(np.ascontiguousarray(m32[sel]), "mxfp4", rht, seed, rht_mode)
    rows = v.shape[0]
    nm, nb = k // MACRO_BLOCK, MACRO_BLOCK // 16
    vb = v.reshape(rows, nm, nb, 16)
    if rows:
        alpha = np.max(np.abs(vb), axis=(2, 3)).astype(np.float32)
        a_b = np.max(np.abs(vb), axis=3).astype(np.float32)
    else:
        alpha = np.zeros((0, nm), np.float32)
        a_b = np.zeros((0, nm, nb), np.float32)
    S = mbs_macro_scale(alpha)
    with np.errstate(divide="ignore", over="ignore"):
        rS = np.where(S == 0.0, F32(0.0), F32(1.0) / S).astype(np.float32)
    rS = np.where(np.isinf(rS), np.finfo(np.float32).max, rS).astype(np.float32)
    a1 = (a_b * rS[..., None]).astype(np.float32)
    e_b = e8m0_exponent(a1)
    w = (vb * rS[..., None, None]).astype(np.float32)
    y = (w.astype(np.float64) * np.exp2(-e_b.astype(np.float64))[..., None]).astype(np.float32)
    y = y.reshape(rows, k)
    if rounding == "rtne":
        c = round_rtne(y, "mxfp4")
    elif rounding == "sr":
        idx = sel[:, None] * k + np.arange(k, dtype=np.int64)[None, :]
        c = round_sr(y, "mxfp4", sr_uniforms(idx, seed, axis))
    else:
        raise ValueError(rounding)
    qv = code_value(c, "mxfp4")
    term = np.abs(qv) - np.abs(y.astype(np.float64))
    step64 = np.exp2(e_b.astype(np.float64)) * S.astype(np.float64)[..., None]
    vhat = (qv.reshape(rows, nm, nb, 16) * step64[..., None]).reshape(rows, k)
    v64 = v.astype(np.float64)
    stats = stats_from_sums(float(np.sum(term)), float(np.sum(np.abs(term))), float(np.sum(v64 * v64)),
                            float(np.sum((v64 - vhat) ** 2)), rows * k, 6.0)
    return {"fmt": "mxfp4_mbs", "block": 16, "rows": rows, "cols": k, "rows_subset": rows_subset,
            "codes": pack_nibbles(c), "scales": (e_b + 127).astype(np.uint8).reshape(rows, k // 16),
            "macro_scales": S, "stats": stats}


def dequantize_mbs(codes_packed: np.ndarray, scales: np.ndarray, macro_scales: np.ndarray,
                   inverse_rht: bool = False, seed: int = 0) -> np.ndarray:
    """v_hat = (q * 2^e_b) * S in FP32, two round-to-nearest products in that
    order (the first is exact), S the scale of the element's macro block;
    optionally followed by R^T (FP32 butterfly)."""
    c = unpack_nibbles(codes_packed)
    n, k = c.shape
    q = code_value(c, "mxfp4").astype(np.float32).reshape(n, k // 16, 16)
    mult = np.exp2((np.asarray(scales, dtype=np.int64) - 127).astype(np.float64)).astype(np.float32)
    S = np.repeat(np.asarray(macro_scales, dtype=np.float32), MACRO_BLOCK // 16, axis=1)
    v = ((q * mult[..., None]).astype(np.float32) * S[..., None]).astype(np.float32).reshape(n, k)
    if inverse_rht:
        v = rht_inverse_butterfly(v.reshape(n, k // 16, 16), rht_signs(seed)).reshape(n, k)
    return v


# --------------------------------------------------------------------------- #
# HiF4: three-level hierarchical scale [HIF] §2 Metodología, reading R17      #
# --------------------------------------------------------------------------- #

#: block, sub-block and micro-block of HiF4 ([HIF] Resumen técnico §2)
HIF4_BLOCK, HIF4_SUB, HIF4_MICRO = 64, 8, 4
HIF4_QMAX = 7.0
E6M2_BIAS = 31


def e6m2_decode(code) -> np.ndarray:
    """Value of an unsigned E6M2 code 0..255 (reading R17), as FP64: exponent
    field E = code >> 2, mantissa m = code & 3; E = 0 is subnormal,
    m/4 * 2^(1 - 31); otherwise (1 + m/4) * 2^(E - 31). Largest value
    1.75 * 2^32 (code 255), smallest positive 2^-32 (code 1)."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    e = c >> 2
    m = c & 3
    sub = (m / 4.0) * 2.0 ** (1 - E6M2_BIAS)
    nrm = (1.0 + m / 4.0) * np.exp2((e - E6M2_BIAS).astype(np.float64))
    return np.where(e == 0, sub, nrm)


#: all 256 E6M2 values, ascending with the code.
E6M2_VALUES = e6m2_decode(np.arange(256))


def e6m2_encode_rne_sat(t) -> np.ndarray:
    """FP32 t >= 0 -> E6M2 code: nearest value, ties to the even code; values
    above the largest (1.75 * 2^32) saturate to it."""
    a = np.minimum(np.asarray(t, dtype=np.float64), E6M2_VALUES[-1])
    return _nearest_even(a, E6M2_VALUES).astype(np.uint8)


def quantize_copy_hif4(m32: np.ndarray, rht: bool = False, rounding: str = "rtne",
                       seed: int = 0, axis: int = 0, rht_mode: str = "butterfly",
                       rows_subset=None) -> dict:
    """HiF4 ([HIF] Resumen técnico §2 Metodología, reading R17): per copy row,
    64-element block B, 8-element sub-block J inside it and 4-element
    micro-block I inside J:
      v    = RHT(x) or x (16-point transforms, four per block)
      a_64 = max |v| over B;  t = a_64 / 7 (FP32);  S = E6M2_rne_sat(t)
      r    = 1 / S (FP32; 0 if S = 0)
      d_J  = 1 iff RN(a_J * r) * 2 <= 7             (a_J = max |v| over J)
      d_I  = 1 iff RN(a_I * r) * 2^(d_J + 1) <= 7   (a_I = max |v| over I)
      y    = RN(v * r) * 2^(d_J + d_I)  (the power of two is exact)
      q    = RTNE(y) or SR(y, u_i) on the integer grid 0..7 (E1M2 in units of
             1/4), sign kept
    The element's value is q * S * 2^-(d_J + d_I). Returns the packed codes,
    ``scales`` = one uint32 word per block (E6M2 code in bits 0-7, d_J of
    sub-block j in bit 8 + j, d_I of micro-block i in bit 16 + i) and the
    statistics (Qmax 7; v_hat = q * S * 2^-(d_J + d_I), FP64)."""
    n, k = m32.shape
    if k % HIF4_BLOCK:
        raise ValueError("cols must be a multiple of the HiF4 block (64)")
    sel = np.arange(n) if rows_subset is None else np.asarray(rows_subset, dtype=np.int64)
    v = transform_copy(np.ascontiguousarray(m32[sel]), "ufp4", rht, seed, rht_mode)
    rows = v.shape[0]
    nb = k // HIF4_BLOCK
    # block, sub-block (8 per block), micro-block (2 per sub-block), element (4)
    vb = v.reshape(rows, nb, 8, 2, 4)
    av = np.abs(vb)
    a64 = av.max(axis=(2, 3, 4)).astype(np.float32)
    a8 = av.max(axis=(3, 4)).astype(np.float32)
    a4 = av.max(axis=4).astype(np.float32)
    with np.errstate(invalid="ignore"):
        t = (a64 / F32(HIF4_QMAX)).astype(np.float32)
        s_code = e6m2_encode_rne_sat(t)
    S = e6m2_decode(s_code).astype(np.float32)
    with np.errstate(divide="ignore"):
        r = np.where(S == 0.0, F32(0.0), F32(1.0) / S).astype(np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        w8 = (a8 * r[..., None]).astype(np.float32)
        d8 = (w8.astype(np.float64) * 2.0) <= HIF4_QMAX
        w4 = (a4 * r[..., None, None]).astype(np.float32)
        d4 = (w4.astype(np.float64) * np.exp2(d8[..., None].astype(np.float64) + 1.0)) <= HIF4_QMAX
        shift = d8[..., None].astype(np.int64) + d4.astype(np.int64)          # rows, nb, 8, 2
        w = (vb * r[..., None, None, None]).astype(np.float32)
        y = (w.astype(np.float64) * np.exp2(shift.astype(np.float64))[..., None]).astype(np.float32)
    y = y.reshape(rows, k)
    if rounding == "rtne":
        c = round_rtne(y, "ufp4")
    elif rounding == "sr":
        idx = sel[:, None] * k + np.arange(k, dtype=np.int64)[None, :]
        c = round_sr(y, "ufp4", sr_uniforms(idx, seed, axis))
    else:
        raise ValueError(rounding)
    d8_bits = np.sum(d8.astype(np.uint32) << np.arange(8, dtype=np.uint32), axis=-1, dtype=np.uint32)
    d4_bits = np.sum(d4.reshape(rows, nb, 16).astype(np.uint32) << np.arange(16, dtype=np.uint32),
                     axis=-1, dtype=np.uint32)
    words = (s_code.astype(np.uint32) | (d8_bits << np.uint32(8)) | (d4_bits << np.uint32(16))).astype(np.uint32)
    qv = code_value(c, "ufp4")
    term = np.abs(qv) - np.abs(y.astype(np.float64))
    step = S.astype(np.float64)[..., None, None] * np.exp2(-shift.astype(np.float64))
    vhat = (qv.reshape(rows, nb, 8, 2, 4) * step[..., None]).reshape(rows, k)
    v64 = v.astype(np.float64)
    stats = stats_from_sums(float(np.sum(term)), float(np.sum(np.abs(term))), float(np.sum(v64 * v64)),
                            float(np.sum((v64 - vhat) ** 2)), rows * k, HIF4_QMAX)
    return {"fmt": "hif4", "block": HIF4_BLOCK, "rows": rows, "cols": k, "rows_subset": rows_subset,
            "codes": pack_nibbles(c), "scales": words.reshape(rows, nb), "shift": shift.reshape(rows, nb * 16),
            "y": y, "stats": stats}


def hif4_fields(words: np.ndarray):
    """Split HiF4 scale words into (E6M2 code, d_8 bits [..., 8], d_4 bits [..., 16])."""
    w = np.asarray(words, dtype=np.uint32)
    code = (w & np.uint32(0xFF)).astype(np.uint8)
    d8 = ((w[..., None] >> (np.uint32(8) + np.arange(8, dtype=np.uint32))) & np.uint32(1)).astype(np.int64)
    d4 = ((w[..., None] >> (np.uint32(16) + np.arange(16, dtype=np.uint32))) & np.uint32(1)).astype(np.int64)
    return code, d8, d4


def dequantize_hif4_f64(codes_packed: np.ndarray, words: np.ndarray) -> np.ndarray:
    """Exact value of every element of a HiF4 copy, q * S * 2^-(d_8 + d_4)."""
    c = unpack_nibbles(codes_packed)
    n, k = c.shape
    code, d8, d4 = hif4_fields(words)
    shift = np.repeat(d8, 2, axis=-1) + d4                                # n, nb, 16
    step = e6m2_decode(code)[..., None] * np.exp2(-shift.astype(np.float64))
    q = code_value(c, "ufp4").reshape(n, k // HIF4_BLOCK, 16, HIF4_MICRO)
    return (q * step[..., None]).reshape(n, k)


def dequantize_hif4(codes_packed: np.ndarray, words: np.ndarray, inverse_rht: bool = False,
                    seed: int = 0) -> np.ndarray:
    """HiF4 values in FP32 (each is exact there: q * S has at most 6
    significant bits and the power of two 2^-(d_8 + d_4) stays in range),
    optionally followed by R^T (FP32 butterfly)."""
    v = dequantize_hif4_f64(codes_packed, words).astype(np.float32)
    if inverse_rht:
        n, k = v.shape
        v = rht_inverse_butterfly(v.reshape(n, k // 16, 16), rht_signs(seed)).reshape(n, k)
    return v


def code_histogram(codes_packed: np.ndarray) -> np.ndarray:
    """Number of elements carrying each 4-bit code 0..15 in a packed copy
    (reading R14)."""
    c = unpack_nibbles(codes_packed).ravel()
    return np.bincount(c, minlength=16).astype(np.int64)


def effective_bucket_ratio(hist16: np.ndarray) -> float:
    """exp(H) / 8, H = -sum p_l ln p_l over the 8 magnitude levels (codes c and
    c + 8 fold together): 1 when all levels are used equally, 1/8 when one
    level holds everything ([UFP4] Resultados, reading R14)."""
    h = np.asarray(hist16, dtype=np.float64)
    m = h[:8] + h[8:]
    tot = m.sum()
    if tot == 0:
        return 0.0
    p = m[m > 0] / tot
    return float(np.exp(-np.sum(p * np.log(p))) / 8.0)


def stats_from_sums(sum_bias, sum_abs_bias, sum_sig2, sum_err2, nel, qmax) -> dict:
    """Shrinkage bias (mean signed error in magnitude, normalised by Qmax;
    [UFP4] Metodología §1) and quantisation SNR in dB ([UFP4] Resultados;
    [NGPT] Risultati §1). SNR is +inf when the error energy is 0."""
    bias = sum_bias / (qmax * nel) if nel else 0.0
    if sum_err2 == 0.0:
        snr = float("inf")
    elif sum_sig2 == 0.0:
        snr = float("-inf")
    else:
        snr = 10.0 * np.log10(sum_sig2 / sum_err2)
    return {"shrink_bias": bias, "snr_db": float(snr), "sum_sig2": sum_sig2,
            "sum_err2": sum_err2, "sum_abs_bias": sum_abs_bias, "n": nel,
            "mean_abs_bias": (sum_abs_bias / (qmax * nel)) if nel else 0.0}


def quantize(x, fmt: str, rht: bool = False, rounding: str = "rtne", seed: int = 0,
             axis: str = "row", rht_mode: str = "butterfly", keep_y: bool = False,
             rows_subset=None, cols_subset=None) -> dict:
    """Quantise a rows x cols tensor (BF16 bits as uint16, or FP32).

    axis: "row" (blocks along each row), "col" (blocks along each column,
    emitted as the transposed copy [cols][rows/2]) or "both".
    rows_subset / cols_subset restrict the row-wise copy to those rows of x and
    the column-wise copy to those columns of x (rows of the transposed copy).
    Returns {"row": copy, "col": copy} with the requested copies, plus
    "nonfinite": True when the input held a NaN or an infinity.
    """
    m = _as_f32_matrix(x)
    out = {"nonfinite": bool(not np.all(np.isfinite(m)))}
    outer = {"nvfp4_2l": quantize_copy_two_level, "mxfp4_mbs": quantize_copy_mbs,
             "hif4": quantize_copy_hif4}.get(fmt)
    if outer is not None:
        if axis in ("row", "both"):
            out["row"] = outer(m, rht, rounding, seed, 0, rht_mode, rows_subset)
        if axis in ("col", "both"):
            out["col"] = outer(np.ascontiguousarray(m.T), rht, rounding, seed, 1, rht_mode, cols_subset)
        return out
    if axis in ("row", "both"):
        out["row"] = quantize_copy(m, fmt, rht, rounding, seed, 0, rht_mode, keep_y=keep_y,
                                   rows_subset=rows_subset)
    if axis in ("col", "both"):
        out["col"] = quantize_copy(np.ascontiguousarray(m.T), fmt, rht, rounding, seed, 1,
                                   rht_mode, keep_y=keep_y, rows_subset=cols_subset)
    return out


# --------------------------------------------------------------------------- #
# Dequantisation                                                              #
# --------------------------------------------------------------------------- #

def dequantize(codes_packed: np.ndarray, scales: np.ndarray, g, fmt: str,
               inverse_rht: bool = False, seed: int = 0) -> np.ndarray:
    """v_hat = (q * s_b) * g in FP32, two round-to-nearest products in that
    order (E8M0 formats: q * 2^e_b); optionally followed by R^T (FP32
    butterfly)."""
    b = BLOCK[fmt]
    c = unpack_nibbles(codes_packed)
    n, k = c.shape
    q = code_value(c, fmt).astype(np.float32).reshape(n, k // b, b)
    if fmt in E8M0_FORMATS:
        e_b = np.asarray(scales, dtype=np.int64) - 127
        mult = np.exp2(e_b.astype(np.float64)).astype(np.float32)
        v = (q * mult[..., None]).astype(np.float32)
    else:
        s_val = e4m3_decode(scales).astype(np.float32)
        v = ((q * s_val[..., None]).astype(np.float32) * F32(g)).astype(np.float32)
    v = v.reshape(n, k)
    if inverse_rht:
        v = rht_inverse_butterfly(v.reshape(n, k // 16, 16), rht_signs(seed)).reshape(n, k)
    return v


def dequantize_f64(codes_packed: np.ndarray, scales: np.ndarray, g, fmt: str,
                   rows=None) -> np.ndarray:
    """Exact FP64 value of each element: q * s_b * g (E8M0 formats:
    q * 2^e_b)."""
    b = BLOCK[fmt]
    cp = codes_packed if rows is None else codes_packed[rows]
    sc = scales if rows is None else scales[rows]
    c = unpack_nibbles(cp)
    n, k = c.shape
    q = code_value(c, fmt).reshape(n, k // b, b)
    if fmt in E8M0_FORMATS:
        step = np.exp2((np.asarray(sc, dtype=np.int64) - 127).astype(np.float64))
    else:
        step = e4m3_decode(sc) * np.float64(g)
    return (q * step[..., None]).reshape(n, k)


# --------------------------------------------------------------------------- #
# Block-scaled GEMM                                                           #
# --------------------------------------------------------------------------- #

def dequantize_outer_f64(copy: dict, rows=None) -> np.ndarray:
    """Exact FP64 value of each element of a two-level NVFP4 copy (q * s_b *
    g_o) or an MBS copy (q * 2^e_b * S), S / g_o the element's per-128 scale."""
    sel = slice(None) if rows is None else rows
    c = unpack_nibbles(copy["codes"][sel])
    n, k = c.shape
    q = code_value(c, "nvfp4").reshape(n, k // 16, 16)
    if copy["fmt"] == "nvfp4_2l":
        step = e4m3_decode(copy["scales"][sel])
        outer = copy["outer_scales"][sel]
    else:
        step = np.exp2((np.asarray(copy["scales"][sel], dtype=np.int64) - 127).astype(np.float64))
        outer = copy["macro_scales"][sel]
    step = step * np.repeat(np.asarray(outer, dtype=np.float64), OUTER_BLOCK // 16, axis=1)
    return (q * step[..., None]).reshape(n, k)


def gemm(a_copy: dict, b_copy: dict, rows=None, cols=None) -> np.ndarray:
    """Y = dequant(A) @ dequant(B)^T in FP64 ([UFP4] Resultados, single-GEMM
    output; [NGPT] Metodologia, Y = WX), optionally for a subset of output
    rows (of A) and columns (rows of B)."""
    def deq(cp, sel):
        if cp["fmt"] in ("nvfp4_2l", "mxfp4_mbs"):
            return dequantize_outer_f64(cp, sel)
        if cp["fmt"] == "hif4":
            s_ = slice(None) if sel is None else sel
            return dequantize_hif4_f64(cp["codes"][s_], cp["scales"][s_])
        return dequantize_f64(cp["codes"], cp["scales"], cp["tensor_scale"], cp["fmt"], sel)
    return deq(a_copy, rows) @ deq(b_copy, cols).T


def snr_db(ref: np.ndarray, approx: np.ndarray) -> float:
    ref = np.asarray(ref, dtype=np.float64)
    err = ref - np.asarray(approx, dtype=np.float64)
    e2 = float(np.sum(err * err))
    return float("inf") if e2 == 0.0 else 10.0 * np.log10(float(np.sum(ref * ref)) / e2)


# --------------------------------------------------------------------------- #
# Tensor-core scale-factor layout                                             #
# --------------------------------------------------------------------------- #

def mma_scale_offset(r, kb, nkb: int) -> np.ndarray:
    """Byte offset of scale (row r, block kb) in the 128x4 tiled layout the
    block-scaled tensor-core MMA reads: tiles of 128 rows x 4 blocks are 512
    contiguous bytes, tiles ordered with the block index fastest; inside a
    tile, byte (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4. ``nkb`` is the
    number of blocks per row, padded to a multiple of 4."""
    r = np.asarray(r, dtype=np.int64)
    kb = np.asarray(kb, dtype=np.int64)
    tile = (r // 128) * (nkb // 4) + kb // 4
    return tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4


def scales_to_mma_layout(scales: np.ndarray, block: int = 16) -> np.ndarray:
    """Linear [rows][nkb] scales -> the tiled layout (rows padded to 128,
    blocks to 4, padding bytes 0), as a flat uint8 array. The tensor cores read
    one scale per 16 elements along K: a 32-element block's scale is written
    for both of its 16-element halves."""
    s = np.asarray(scales, dtype=np.uint8)
    if block == 32:
        s = np.repeat(s, 2, axis=1)
    n, nkb = s.shape
    n_p = -(-n // 128) * 128
    nkb_p = -(-nkb // 4) * 4
    out = np.zeros(n_p * nkb_p, dtype=np.uint8)
    r, kb = np.meshgrid(np.arange(n), np.arange(nkb), indexing="ij")
    out[mma_scale_offset(r, kb, nkb_p)] = s
    return out


def mma_layout_bytes(rows: int, nkb: int) -> int:
    return (-(-rows // 128) * 128) * (-(-nkb // 4) * 4)
