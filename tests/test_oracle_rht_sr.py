"""Pins of the oracle's RHT, Philox and stochastic rounding (no GPU)."""

import os

import numpy as np
import pytest

from oracle import fp4q_oracle as o



# ---- RHT -------------------------------------------------------------------

def test_hadamard_orthogonal():
    H = o.hadamard16()
    assert np.array_equal(H @ H.T, 16.0 * np.eye(16))
    assert np.array_equal(H, H.T)
    # Sylvester recursion H_{2n} = [[H_n, H_n], [H_n, -H_n]] from H_1 = [1]
    S = np.array([[1.0]])
    for _ in range(4):
        S = np.block([[S, S], [S, -S]])
    assert np.array_equal(S, H)


def test_rht_unit_vectors_and_norm():
    s = o.rht_signs(1234)
    H = o.hadamard16()
    eye = np.eye(16, dtype=np.float32)
    v = o.rht_definition(eye, s)           # row j = R e_j
    assert np.array_equal(v.T.astype(np.float64), 0.25 * H * s[None, :])
    rng = np.random.default_rng(0)
    x = rng.standard_normal((4096, 16)).astype(np.float32)
    vx = o.rht_definition(x, s).astype(np.float64)
    nx = np.linalg.norm(x.astype(np.float64), axis=1)
    assert np.allclose(np.linalg.norm(vx, axis=1), nx, rtol=1e-6)
    back = o.rht_inverse_definition(vx.astype(np.float32), s)
    assert np.allclose(back, x, rtol=0, atol=4e-6 * np.max(np.abs(x)))


def test_rht_butterfly_vs_definition():
    s = o.rht_signs(99)
    rng = np.random.default_rng(1)
    # narrow exponent range (BF16 inputs, spread <= 12 binades): butterfly is exact
    x = o.bf16_bits_to_f32(o.f32_to_bf16_bits_rne(rng.uniform(0.5, 2.0, (20000, 16)).astype(np.float32)))
    x = x * np.where(rng.random((20000, 16)) < 0.5, -1, 1).astype(np.float32)
    assert np.array_equal(o.rht_butterfly(x, s), o.rht_definition(x, s))
    # heavy tails: within 2 FP32 ulp of the definition (a rounded dense product)
    y = (rng.standard_t(3, (20000, 16)) * np.exp(rng.standard_normal((1, 16)) * 3)).astype(np.float32)
    y = o.bf16_bits_to_f32(o.f32_to_bf16_bits_rne(y))
    b = o.rht_butterfly(y, s).astype(np.float64)
    d = o.rht_definition(y, s).astype(np.float64)
    ulp = np.spacing(np.abs(d).astype(np.float32)).astype(np.float64)
    # 2 ulp of the block's largest output bounds the absolute error of each output
    blockulp = np.max(ulp, axis=1, keepdims=True)
    assert np.all(np.abs(b - d) <= 2 * blockulp)
    inv = o.rht_inverse_butterfly(o.rht_butterfly(x, s), s)
    assert np.allclose(inv, x, rtol=0, atol=1e-6 * 4)


def test_rht_signs_are_seeded():
    a, b = o.rht_signs(1234), o.rht_signs(1235)
    assert set(np.unique(a)) <= {-1.0, 1.0}
    assert not np.array_equal(a, b)
    assert np.array_equal(a, o.rht_signs(1234))


def test_rht_cancels_in_a_dot_product():
    s = o.rht_signs(7)
    rng = np.random.default_rng(2)
    a = rng.standard_normal((64, 16))
    b = rng.standard_normal((64, 16))
    H = o.hadamard16()
    R = 0.25 * H * s[None, :]
    assert np.allclose((a @ R.T) @ (b @ R.T).T, a @ b.T, atol=1e-12)


# ---- Philox ----------------------------------------------------------------

def _curand_host_philox(seed: int, nwords: int, offset: int):
    """Words of cuRAND's host-side Philox4x32-10 generator (libcurand, NVIDIA's
    implementation, run on the CPU: no device needed), default ordering."""
    import ctypes
    import ctypes.util
    names = ["libcurand.so", "libcurand.so.10", ctypes.util.find_library("curand")]
    for d in ("/usr/local/cuda/lib64", "/usr/local/cuda/targets/x86_64-linux/lib"):
        names.append(os.path.join(d, "libcurand.so"))
    lib = None
    for n in names:
        if not n:
            continue
        try:
            lib = ctypes.CDLL(n)
            break
        except OSError:
            continue
    assert lib is not None, "libcurand not found: the Philox pin needs cuRAND's host generator"
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0   # CURAND_RNG_PSEUDO_PHILOX4_32_10
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(nwords, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(nwords)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out


# cuRAND's host Philox generator runs 65536 subsequences side by side: output
# quadruple q comes from subsequence t = q mod 65536 at step s = q div 65536,
# i.e. from the counter (s lo, s hi, t, 0) under the key (seed lo, seed hi) --
# the counter/key assignment its device API documents for curand_init(seed,
# subsequence t, offset 4 s). A generator offset of 4 q starts at quadruple q.
_CURAND_THREADS = 65536


@pytest.mark.parametrize("seed", [0, 0xFFFFFFFFFFFFFFFF, 1234, 0x0123456789ABCDEF])
def test_philox_matches_curand_host_generator(seed):
    """Pins the oracle's Philox4x32-10 word for word against an implementation
    it does not share code with (cuRAND). Covered: the round function (both
    multipliers, the output word order), the key schedule (bump before each
    round after the first), both key words, and the counter words c0, c1
    (steps past 2^32) and c2 (the subsequence). c3 enters the first round
    through the same round function that rounds 2-10 exercise with non-zero
    values in that slot."""
    k0, k1 = seed & 0xFFFFFFFF, seed >> 32
    # the first 64 quadruples: subsequences 0..63 at step 0
    got = _curand_host_philox(seed, 256, 0).reshape(-1, 4)
    t = np.arange(64, dtype=np.uint64)
    want = np.stack(o.philox4x32_10(0, 0, t, 0, k0, k1), axis=1).astype(np.uint32)
    assert np.array_equal(got, want)
    # step 1 and steps beyond 2^32 (the counter's second word), several subsequences
    for s, t0 in ((1, 0), (3, 65530), (1 << 32, 0), ((1 << 32) + 5, 7), ((1 << 33) + 3, 65535)):
        q = s * _CURAND_THREADS + t0
        got = _curand_host_philox(seed, 4, 4 * q)
        want = np.array([int(w) for w in o.philox4x32_10(s & 0xFFFFFFFF, s >> 32, t0, 0, k0, k1)],
                        dtype=np.uint32)
        assert np.array_equal(got, want), (hex(seed), s, t0)


def test_philox_properties():
    """Philox4x32-10 has no known-answer vectors here (parity unpinned for
    the exact bits): check what the construction guarantees instead. Each round
    is invertible for a fixed key, so distinct counters give distinct outputs;
    one flipped counter or key bit flips about half of the 128 output bits; the
    output words are uniform."""
    k0, k1 = 0x1234ABCD, 0x0F0F0F0F
    c = np.arange(1 << 14, dtype=np.uint64)
    w = np.stack([np.asarray(v, dtype=np.uint64) for v in o.philox4x32_10(c, 0, 0, 0, k0, k1)], axis=1)
    assert np.unique(w, axis=0).shape[0] == 1 << 14
    rng = np.random.default_rng(3)
    n = 400
    ctr = rng.integers(0, 1 << 32, (4, n), dtype=np.uint64)
    base = np.stack(o.philox4x32_10(*ctr, k0, k1))
    word, bit = rng.integers(0, 4, n), rng.integers(0, 32, n).astype(np.uint64)
    ctr2 = ctr.copy()
    ctr2[word, np.arange(n)] ^= np.uint64(1) << bit
    flipped = np.stack(o.philox4x32_10(*ctr2, k0, k1))
    kb = rng.integers(0, 64, n).astype(np.uint64)
    k0v = np.where(kb < 32, np.uint64(k0) ^ (np.uint64(1) << (kb % np.uint64(32))), np.uint64(k0))
    k1v = np.where(kb >= 32, np.uint64(k1) ^ (np.uint64(1) << (kb % np.uint64(32))), np.uint64(k1))
    keyed = np.stack(o.philox4x32_10(*ctr, k0v, k1v))
    def popcount(x):
        return np.array([bin(int(v)).count("1") for v in x.ravel()]).reshape(x.shape)
    flips = np.concatenate([popcount(base ^ flipped).sum(axis=0), popcount(base ^ keyed).sum(axis=0)])
    assert abs(flips.mean() - 64.0) < 2.0    # 800 samples of Binomial(128, 1/2): sd of the mean 0.2
    h, _ = np.histogram((w[:, 1] >> np.uint64(26)).astype(np.int64), bins=64, range=(0, 64))
    e = w.shape[0] / 64
    assert np.sum((h - e) ** 2 / e) < 120


def test_sr_uniforms_layout():
    u = o.sr_uniforms(np.arange(8), 1234, 0)
    k0, k1 = 1234, 0
    w = o.philox4x32_10(0, 0, 0, 0, k0, k1)
    w1 = o.philox4x32_10(1, 0, 0, 0, k0, k1)
    exp = [(int(v) >> 8) * 2.0 ** -24 for v in list(w) + list(w1)]
    assert np.array_equal(u, np.array(exp))
    assert np.all((u >= 0) & (u < 1))
    # axis word changes the stream
    assert not np.array_equal(u, o.sr_uniforms(np.arange(8), 1234, 1))
    # uniformity: chi-square over 64 bins for 2^18 draws
    uu = o.sr_uniforms(np.arange(1 << 18), 42, 0)
    h, _ = np.histogram(uu, bins=64, range=(0, 1))
    e = (1 << 18) / 64
    chi2 = np.sum((h - e) ** 2 / e)
    assert chi2 < 120  # 63 dof, p ~ 1e-5


# ---- stochastic rounding --------------------------------------------------

@pytest.mark.parametrize("fmt,y", [("nvfp4", 0.3), ("nvfp4", 1.2),
                                   ("nvfp4", 2.7), ("nvfp4", 5.1), ("ufp4", 3.37),
                                   ("nvfp4", 1e-6), ("ufp4", 6.999)])
def test_sr_exact_probability(fmt, y):
    """Enumerate every one of the 2^24 values u takes: the number that round up
    is ceil(f * 2^24), f = (|y| - lo) / (hi - lo)."""
    y32 = np.float32(y)
    levels = o.grid_levels(fmt)
    lo = levels[levels <= float(y32)].max()
    hi = levels[levels > float(y32)].min()
    f = (float(y32) - lo) / (hi - lo)
    u = np.arange(1 << 24, dtype=np.float64) * 2.0 ** -24
    c = o.round_sr(np.full(u.shape, y32), fmt, u)
    ups = int(np.sum(o.code_value(c, fmt) == hi))
    downs = int(np.sum(o.code_value(c, fmt) == lo))
    assert ups + downs == (1 << 24)
    assert ups == int(np.ceil(f * 2 ** 24))


def test_sr_on_grid_and_saturation():
    for fmt in ("nvfp4", "ufp4"):
        lv = o.grid_levels(fmt).astype(np.float32)
        u = np.zeros(lv.size)
        assert np.array_equal(o.code_value(o.round_sr(lv, fmt, u), fmt), lv)
        u = np.full(lv.size, 1 - 2.0 ** -24)
        assert np.array_equal(o.code_value(o.round_sr(lv, fmt, u), fmt), lv)
        big = np.array([lv[-1] * 1.5, -lv[-1] * 3], dtype=np.float32)
        assert np.array_equal(o.code_value(o.round_sr(big, fmt, np.zeros(2)), fmt),
                              [lv[-1], -lv[-1]])


@pytest.mark.parametrize("fmt", ["nvfp4", "ufp4"])
def test_sr_unbiased(fmt):
    """E[round(y)] = y: the mean over 2^20 independently keyed elements lies
    within 4 sigma of y."""
    n = 1 << 20
    for y in (0.37, 1.61, 2.2, 4.9):
        if y >= o.QMAX[fmt]:
            continue
        u = o.sr_uniforms(np.arange(n), 77, 0)
        q = o.code_value(o.round_sr(np.full(n, np.float32(y), dtype=np.float32), fmt, u), fmt)
        levels = o.grid_levels(fmt)
        lo = levels[levels <= y].max()
        hi = levels[levels > y].min()
        p = (np.float32(y) - lo) / (hi - lo)
        sigma = (hi - lo) * np.sqrt(p * (1 - p) / n)
        assert abs(q.mean() - np.float32(y)) < 4 * sigma + 1e-12
