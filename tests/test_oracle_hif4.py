"""Pins of the oracle's HiF4 three-level format ("Unleashing Low-Bit Inference
on Ascend NPUs: A Comprehensive Evaluation of HiFloat Formats", Resumen técnico
§2 Metodología: an E6M2 scale per 64 elements, E1M0 factors per 8 and per 4
elements, E1M2 elements).

The page gives the structure only, so the reading itself (scale rule, what an
E1M0 factor does, rounding) is parity unpinned. What is pinned here is that the
oracle computes that reading: hand-derived worked examples, the E6M2 value set
built a second way, the encoder against a brute-force nearest search, the
per-group factors against an exhaustive search of every combination, the
shift-free case against numpy's rint, and the error bound of each element."""
import os

import numpy as np
import pytest

from oracle import fp4q_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hif4_worked.txt")


def _examples():
    ex, cur = {}, None
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            if key == "name":
                cur = ex.setdefault(rest[0], {})
            else:
                cur[key] = rest
    return ex


@pytest.mark.parametrize("name", sorted(_examples()))
def test_worked_examples(name):
    e = _examples()[name]
    vals = [float(t) for t in e["v"]]
    v = np.zeros((1, 64), np.float32)
    v[0, :len(vals)] = vals
    r = o.quantize(v, "hif4")["row"]
    assert int(r["scales"][0, 0]) == int(e["word"][0], 16)
    want = np.zeros(64, np.uint8)
    cw = [int(t) for t in e["codes"]]
    want[:len(cw)] = cw
    assert np.array_equal(o.unpack_nibbles(r["codes"])[0], want)


def test_e6m2_value_set_built_from_integers():
    """The 256 E6M2 values are 0, the subnormals k * 2^-32 (k = 1..3) and, per
    binade e = -30..32, the four values (4 + m) * 2^(e - 2): every positive
    number with at most three significant bits in [2^-32, 2^33)."""
    vals = [k * 2.0 ** -32 for k in range(4)]
    for e in range(-30, 33):
        vals += [(4 + m) * 2.0 ** (e - 2) for m in range(4)]
    assert np.array_equal(o.E6M2_VALUES, np.array(vals))
    assert np.all(np.diff(o.E6M2_VALUES) > 0)
    assert o.e6m2_decode(124) == 1.0
    assert o.e6m2_decode(255) == 1.75 * 2.0 ** 32
    assert o.e6m2_decode(1) == 2.0 ** -32


def test_e6m2_encoder_brute_force():
    rng = np.random.default_rng(7)
    t = np.exp2(rng.uniform(-36, 36, 4000))
    mids = (o.E6M2_VALUES[1:] + o.E6M2_VALUES[:-1]) / 2           # every tie
    t = np.concatenate([t, mids, o.E6M2_VALUES, [0.0, 2.0 ** 40, 1.8 * 2.0 ** 32]])
    t = t[t == t.astype(np.float32)].astype(np.float32)          # FP32 inputs only
    got = o.e6m2_encode_rne_sat(t)
    for ti, gi in zip(t.astype(np.float64), got):
        d = np.abs(o.E6M2_VALUES - min(ti, o.E6M2_VALUES[-1]))
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert gi == want, (ti, gi, want)


def _heavy_rows(rows, cols, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-3, 3, (rows, cols // 8, 1))).repeat(8, 2).reshape(
        rows, cols)
    x[rng.random((rows, cols)) < 0.02] *= 30.0
    return x.astype(np.float32)


def test_factors_are_the_largest_that_never_clamp():
    """For each 8-element sub-block, every one of the 8 combinations of
    (d_8, d_4 of its two micro-blocks) is tried on the FP32 values y: a
    combination is allowed when no micro-block it gives a finer step than the
    block's own has a |y| above 7 (at the block's own step the largest value
    may sit just above 7: the E6M2 scale is rounded to nearest). The oracle's
    choice must be allowed, and no allowed combination may give a micro-block a
    finer step."""
    x = _heavy_rows(24, 256, 3)
    r = o.quantize_copy_hif4(x)
    code, d8, d4 = o.hif4_fields(r["scales"])
    S = o.e6m2_decode(code).astype(np.float32)
    rcp = np.where(S == 0, np.float32(0), np.float32(1) / S).astype(np.float32)
    w = (x.reshape(24, 4, 8, 2, 4) * rcp[:, :, None, None, None]).astype(np.float32).astype(np.float64)
    for i in range(24):
        for b in range(4):
            for j in range(8):
                chosen = (d8[i, b, j], d4[i, b, 2 * j], d4[i, b, 2 * j + 1])
                best = [0, 0]
                ok_chosen = False
                for c8 in (0, 1):
                    for c0 in (0, 1):
                        for c1 in (0, 1):
                            sh = (c8 + c0, c8 + c1)
                            fits = all(sh[h] == 0 or np.max(np.abs(w[i, b, j, h])) * 2.0 ** sh[h] <= 7.0
                                       for h in (0, 1))
                            if fits:
                                best = [max(best[0], sh[0]), max(best[1], sh[1])]
                                ok_chosen |= (c8, c0, c1) == chosen
                assert ok_chosen, (i, b, j)
                assert [chosen[0] + chosen[1], chosen[0] + chosen[2]] == best, (i, b, j)


def test_shift_free_blocks_are_plain_uniform_rounding():
    """When every micro-block of a block holds the block's maximum, no factor
    can halve a step: the codes are then rint(v / S) clamped to +-7, for
    values away from the rounding midpoints."""
    rng = np.random.default_rng(11)
    x = rng.uniform(-1, 1, (16, 128)).astype(np.float32)
    amax = rng.uniform(0.5, 40, (16, 2)).astype(np.float32)
    xb = x.reshape(16, 2, 16, 4)
    xb[..., 0] = amax[:, :, None] * np.where(rng.random((16, 2, 16)) < 0.5, -1, 1)
    xb[..., 1:] *= amax[:, :, None, None]
    x = xb.reshape(16, 128)
    r = o.quantize_copy_hif4(x)
    code, d8, d4 = o.hif4_fields(r["scales"])
    assert not d8.any() and not d4.any()
    S = np.repeat(o.e6m2_decode(code), 64, axis=1)
    u = x.astype(np.float64) / S
    far = np.abs(u - np.floor(u) - 0.5) > 1e-4
    want = np.clip(np.rint(u), -7, 7)
    got = o.code_value(o.unpack_nibbles(r["codes"]), "ufp4")
    assert np.array_equal(got[far], want[far])


def test_error_bound_per_element():
    """|v - v_hat| <= step / 2 (1 + 2^-20) for every element that does not
    clamp, step = S 2^-(d_8 + d_4); dequantisation returns exactly q * step."""
    x = _heavy_rows(32, 512, 5)
    r = o.quantize_copy_hif4(x)
    vhat = o.dequantize_hif4_f64(r["codes"], r["scales"])
    code, d8, d4 = o.hif4_fields(r["scales"])
    shift = (np.repeat(d8, 2, axis=-1) + d4).reshape(32, -1)
    assert np.array_equal(shift, r["shift"])
    step = np.repeat(np.repeat(o.e6m2_decode(code), 16, axis=1) * np.exp2(-shift.astype(np.float64)), 4, axis=1)
    unclamped = np.abs(x) <= 7 * step
    err = np.abs(x.astype(np.float64) - vhat)
    assert np.all(err[unclamped] <= step[unclamped] / 2 * (1 + 2.0 ** -20))
    assert np.array_equal(o.dequantize_hif4(r["codes"], r["scales"]).astype(np.float64), vhat)


def test_statistics_match_dequantised_values():
    x = _heavy_rows(8, 256, 9)
    r = o.quantize_copy_hif4(x)
    vhat = o.dequantize_hif4_f64(r["codes"], r["scales"])
    assert r["stats"]["snr_db"] == pytest.approx(o.snr_db(x, vhat), abs=1e-9)
    q = np.abs(o.code_value(o.unpack_nibbles(r["codes"]), "ufp4"))
    assert r["stats"]["shrink_bias"] == pytest.approx(np.mean(q - np.abs(r["y"])) / 7, abs=1e-12)


def test_finer_steps_never_lose_to_one_flat_scale():
    """Each factor halves a group's step only where nothing clamps, so on the
    same E6M2 scale the three-level copy is never worse, over a tensor, than
    the flat one (all factors 0): SNR on heavy-tailed rows."""
    x = _heavy_rows(64, 512, 13)
    r = o.quantize_copy_hif4(x)
    code, _, _ = o.hif4_fields(r["scales"])
    S = np.repeat(o.e6m2_decode(code), 64, axis=1)
    flat = np.clip(np.rint(x / S), -7, 7) * S
    assert r["stats"]["snr_db"] > o.snr_db(x, flat) + 1.0


def test_stochastic_rounding_unbiased_over_seeds():
    """SR on the HiF4 grid draws the element's Philox uniform (same stream as
    every format): averaged over seeds the value approaches y."""
    x = _heavy_rows(2, 64, 17)
    ys, qs = [], []
    for seed in range(200):
        r = o.quantize_copy_hif4(x, rounding="sr", seed=seed)
        ys.append(r["y"])
        qs.append(o.code_value(o.unpack_nibbles(r["codes"]), "ufp4"))
    y = ys[0]
    assert all(np.array_equal(y, yy) for yy in ys)       # y does not depend on the seed
    mean = np.mean(qs, axis=0)
    inside = np.abs(y) < 7
    assert np.max(np.abs(mean - y)[inside]) < 0.15


def test_rows_subset_and_rht_compose():
    x = _heavy_rows(16, 128, 19)
    full = o.quantize(x, "hif4", rht=True, seed=5)["row"]
    sub = o.quantize(x, "hif4", rht=True, seed=5, rows_subset=np.array([3, 11]))["row"]
    assert np.array_equal(sub["codes"], full["codes"][[3, 11]])
    assert np.array_equal(sub["scales"], full["scales"][[3, 11]])
    # the inverse transform of the dequantised copy approximates x
    back = o.dequantize_hif4(full["codes"], full["scales"], inverse_rht=True, seed=5)
    assert o.snr_db(x, back) > 15


def test_rejects_partial_blocks():
    with pytest.raises(ValueError):
        o.quantize_copy_hif4(np.zeros((2, 96), np.float32))
