"""The two-piece E4M3 split of a BF16 activation row that the FP8 block applies to x and h
(header beam_moe.h, beam_moe_forward_fp8: one power-of-two row scale s, v = s p1 + (s/16) p2
with p1, p2 E4M3 values). Written here from the E4M3 and BF16 definitions, in numpy, to check
the claim made there: the split is exact for every value within 2^-10 of the row's largest
magnitude, and leaves an absolute error of at most 2^-14 s otherwise (half the smallest step
of the second piece), which is below 2.8e-7 of the row's largest magnitude. The row scale is the
least power of two s with max|v| <= 448 s (the first piece in range); p1 is v / s rounded to
the nearest E4M3 value and p2 the remainder times 16 / s rounded the same way. No GPU."""
import numpy as np

# every finite E4M3 value (both signs), ascending
_POS = np.array([k * 2.0 ** -9 for k in range(8)] +
                [(1 + m / 8) * 2.0 ** (e - 7) for e in range(1, 16) for m in range(8)][:119])
E4M3 = np.unique(np.concatenate([-_POS, _POS]))


def e4m3_rn(y):
    """Nearest E4M3 value (ties to the even code), saturated at +-448."""
    y = np.clip(y, -448.0, 448.0)
    i = np.searchsorted(E4M3, y)
    lo = E4M3[np.maximum(i - 1, 0)]
    hi = E4M3[np.minimum(i, len(E4M3) - 1)]
    pick_hi = (hi - y) < (y - lo)
    tie = (hi - y) == (y - lo)
    # ties: the value whose code is even; for this table that is the one with an even index
    # among the positive codes (mantissa bit 0 clear), mirrored for negatives
    even_hi = (np.abs(np.searchsorted(_POS, np.abs(hi))) % 2) == 0
    pick_hi = np.where(tie, even_hi, pick_hi)
    return np.where(pick_hi, hi, lo)


def bf16_round(v):
    """Round float64 values to BF16 (nearest even) and back."""
    f = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    f = (f + 0x7FFF + ((f >> 16) & 1)) & 0xFFFF0000
    return f.astype(np.uint32).view(np.float32).astype(np.float64)


def split(row):
    amax = float(np.max(np.abs(row)))
    s = 2.0 ** int(np.ceil(np.log2(amax / 448.0))) if amax > 0 else 1.0
    if amax > 0 and amax > 448 * s:
        s *= 2
    p1 = e4m3_rn(row / s)
    p2 = e4m3_rn((row - s * p1) * 16 / s)
    return s, p1, p2


def test_split_is_exact_near_the_row_maximum_and_tiny_elsewhere():
    rng = np.random.default_rng(0)
    for scale in (1e-3, 1.0, 37.0, 3000.0):
        for _ in range(200):
            row = bf16_round(rng.standard_normal(512) * scale * np.exp(rng.uniform(-6, 0, 512)))
            s, p1, p2 = split(row)
            amax = float(np.max(np.abs(row)))
            assert amax <= 448 * s < 2 * amax or amax == 0
            err = np.abs(s * p1 + s / 16 * p2 - row)
            near = np.abs(row) >= 2.0 ** -10 * amax
            assert np.all(err[near] == 0)
            assert np.all(err <= 2.0 ** -14 * s)
            assert np.all(err < 2.8e-7 * amax)


def test_extreme_rows():
    row = np.zeros(64)
    row[3] = bf16_round(np.array([-2.0 ** -40]))[0]        # a row of tiny magnitude
    s, p1, p2 = split(row)
    assert np.array_equal(s * p1 + s / 16 * p2, row)
    row = bf16_round(np.linspace(-3e4, 3e4, 256))            # the largest magnitudes
    s, p1, p2 = split(row)
    assert np.max(np.abs(s * p1 + s / 16 * p2 - row)) <= 2.0 ** -14 * s
