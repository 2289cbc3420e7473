"""Pins of the oracle's code histogram and effective bucket ratio ([UFP4]
Resultados: the RHT raises the effective bucket ratio): counts of a packed
array built with known counts, the nibble order inside a byte, and the ratio's
closed forms (uniform use of the 8 levels -> 1, one level -> 1/8, two levels
equally -> 2/8, signs folded together)."""
import numpy as np

from oracle import fp4q_oracle as o


def _pack(codes):
    c = np.asarray(codes, dtype=np.uint8).reshape(1, -1)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def test_counts_of_known_codes():
    want = np.array([5, 0, 3, 7, 1, 0, 0, 2, 4, 0, 6, 0, 0, 1, 0, 3])
    codes = np.repeat(np.arange(16), want)
    rng = np.random.default_rng(0)
    rng.shuffle(codes)
    if codes.size % 2:
        codes = np.append(codes, 0)
        want[0] += 1
    assert np.array_equal(o.code_histogram(_pack(codes)), want)


def test_nibble_order():
    # byte 0x21: element 0 has code 1 (low nibble), element 1 code 2
    h = o.code_histogram(np.array([[0x21]], dtype=np.uint8))
    assert h[1] == 1 and h[2] == 1 and h.sum() == 2


def test_effective_bucket_ratio_closed_forms():
    assert abs(o.effective_bucket_ratio(np.r_[np.ones(8) * 10, np.zeros(8)]) - 1.0) < 1e-15
    one = np.zeros(16)
    one[3] = 100
    assert abs(o.effective_bucket_ratio(one) - 1 / 8) < 1e-15
    two = np.zeros(16)
    two[1] = 50
    two[9] = 0
    two[6] = 25
    two[14] = 25          # level 6 split over both signs: same as 50 on one
    assert abs(o.effective_bucket_ratio(two) - 2 / 8) < 1e-15
    assert o.effective_bucket_ratio(np.zeros(16)) == 0.0
