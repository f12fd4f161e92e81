"""The four-piece NVFP4 split of an activation block that the NVFP4 block applies to x and h
(header beam_moe.h, beam_moe_forward_nvfp4: per block of 16 elements, with r_0 = v, piece p
has the E4M3 scale u_p = the least E4M3 value >= 4^p max|r_p| / 6 and the E2M1 codes
nearest to r_p / (4^(-p) u_p); r_(p+1) = r_p - 4^(-p) u_p e2m1(code)). Written here from
the definitions of the two formats, in numpy, to check the claims the header makes: every
step is exact in FP32, and what four pieces leave is at most (1.125 / 6)^4 of the block's
largest magnitude (above the absolute floor of the smallest scales) for every block the first
piece can carry (up to 6 * 448); larger blocks are out of range. Also why the factor between
pieces is 4 and not 8: with 8 the later scales can reach the E4M3 maximum. No GPU."""
import numpy as np

# positive E4M3 values by code 0 .. 126 (code 127 is NaN): subnormals k 2^-9, then
# (1 + m/8) 2^(e-7) for exponent fields e = 1 .. 15
E4M3 = np.array([k * 2.0 ** -9 for k in range(8)] +
                [(1 + m / 8) * 2.0 ** (e - 7) for e in range(1, 16) for m in range(8)][:119], dtype=np.float64)
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
BOUND = (1.125 / 6) ** 4
FLOOR = 2.0 ** -9 * 4.0 ** -3  # the step of the last piece at the smallest scale


def e4m3_ceil(x):
    """The least E4M3 value >= x (clamped to 448) and whether x was above 448."""
    i = np.searchsorted(E4M3, x, side="left")
    over = i >= len(E4M3)
    return E4M3[np.minimum(i, len(E4M3) - 1)], over


def e2m1_nearest(y):
    """The nearest E2M1 value to y, saturated at +-6 (ties to the smaller magnitude here;
    the bound does not depend on the tie rule)."""
    a = np.minimum(np.abs(y), 6.0)
    j = np.argmin(np.abs(E2M1[None, :] - a[:, None]), axis=1)
    return np.sign(y) * E2M1[j]


def split(block, step=4):
    """The four pieces of one block (FP32 values): scales u_p, E2M1 values q_p, remainder, and
    whether the first piece was out of range. Piece p is weighted step^-p."""
    r = block.astype(np.float32)
    us, qs, over = [], [], False
    for p in range(4):
        amax = float(np.max(np.abs(r)))
        u, o = e4m3_ceil(amax * float(step) ** p / 6)
        over |= bool(o) and p == 0
        s = np.float32(u * float(step) ** (-p))
        q = e2m1_nearest(r.astype(np.float64) / float(s)).astype(np.float32) if s > 0 else np.zeros(16, np.float32)
        prod = (s * q).astype(np.float32)
        assert np.array_equal(prod.astype(np.float64), float(s) * q.astype(np.float64))  # s * q exact
        new_r = (r - prod).astype(np.float32)
        assert np.array_equal(new_r.astype(np.float64), r.astype(np.float64) - prod.astype(np.float64))  # exact
        r = new_r
        us.append(u)
        qs.append(q)
    return np.array(us), np.array(qs), r, over


def test_e4m3_table_is_the_format():
    assert len(E4M3) == 127 and E4M3[0] == 0 and E4M3[1] == 2.0 ** -9 and E4M3[8] == 2.0 ** -6
    assert E4M3[-1] == 448.0 and np.all(np.diff(E4M3) > 0)


def test_pieces_rebuild_the_block_and_leave_at_most_the_bound():
    rng = np.random.default_rng(0)
    worst = 0.0
    for kind in range(4):
        for _ in range(1500):
            if kind == 0:
                v = rng.standard_normal(16)
            elif kind == 1:
                v = rng.standard_normal(16) * np.exp(rng.uniform(-8, 6, 16))   # magnitudes over decades
            elif kind == 2:
                v = np.where(rng.random(16) < 0.8, 0.0, rng.standard_normal(16) * 50)
            else:
                v = rng.uniform(-2688, 2688, 16)
            v = v.astype(np.float32)
            us, qs, r, over = split(v)
            assert not over
            g = 4.0 ** (-np.arange(4))
            rebuilt = (g[:, None] * us[:, None] * qs.astype(np.float64)).sum(axis=0) + r
            assert np.array_equal(rebuilt, v.astype(np.float64))
            amax = float(np.max(np.abs(v)))
            assert np.max(np.abs(r)) <= BOUND * amax + FLOOR
            if amax > 1e-2:
                worst = max(worst, float(np.max(np.abs(r))) / amax)
    assert worst <= BOUND
    assert worst < 1e-3  # far inside the bound in practice


def test_the_bound_holds_up_to_the_first_pieces_range_with_step_4_not_8():
    """Blocks near 6 * 448: with piece weights 4^-p the bound holds; with 8^-p the later
    pieces' scales reach the E4M3 maximum and leave far more."""
    rng = np.random.default_rng(1)
    worst4 = worst8 = 0.0
    for _ in range(2000):
        v = rng.uniform(-1, 1, 16)
        v = (v / np.max(np.abs(v)) * rng.uniform(1200, 2688)).astype(np.float32)
        amax = float(np.max(np.abs(v)))
        worst4 = max(worst4, float(np.max(np.abs(split(v)[2]))) / amax)
        worst8 = max(worst8, float(np.max(np.abs(split(v, step=8)[2]))) / amax)
    assert worst4 <= BOUND
    assert worst8 > 4 * BOUND


def test_a_single_value_is_carried_exactly():
    for x in (1.0, -3.0, 0.3, 1234.5, 2688.0, 1e-5):
        v = np.zeros(16, np.float32)
        v[5] = x
        _, _, r, over = split(v)
        assert not over
        assert abs(float(r[5])) <= BOUND * abs(x) + FLOOR


def test_zero_block_gives_zero_scales_and_codes():
    us, qs, r, over = split(np.zeros(16, np.float32))
    assert not over and np.all(us == 0) and np.all(qs == 0) and np.all(r == 0)


def test_blocks_above_the_first_piece_are_out_of_range():
    v = np.zeros(16, np.float32)
    v[0] = 2688.0
    assert not split(v)[3]
    v[0] = 2700.0
    assert split(v)[3]
