"""The decode kernels' hi/lo fp16 split of a weight, checked on the host.

A weight w (q_d s_gd for the keys, p_t s_tg for the values, fp32) enters the
fp16 tensor-core products as two halves: hi = fp16(w with its 13 low
mantissa bits cleared), exact in fp16 when w is a normal fp16 value, and
lo = fp16_rn(w - hi) (csrc/decode_mma.cuh, split_hi_lo).  The pair carries
about 22 significant bits: |w - (hi + lo)| <= 2^-22 |w| + 2^-24.  The last
term covers weights below the fp16 normal range (2^-14), where hi and lo
are each rounded to the subnormal spacing 2^-24 (half of it each).  The
kernels scale each tile's weights by a power of two f before the split, so
that the bound on the tile's weights (max|q| times the largest key scale; the
largest value scale, the softmax weights being at most 1) lands in
[2^13, 2^14): no weight overflows fp16, and the absolute term 2^-24 / f stays
far below the tile's weights however small the statistics are.
"""
import numpy as np
import pytest


def split_hi_lo(w):
    w = np.asarray(w, np.float32)
    hi32 = (w.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    hi = hi32.astype(np.float16)
    lo = (w - hi32).astype(np.float32).astype(np.float16)
    return hi, lo


@pytest.mark.parametrize("lo_exp,hi_exp", [(-30, -14), (-14, 0), (0, 15)])
def test_split_carries_22_bits(lo_exp, hi_exp):
    rng = np.random.default_rng(lo_exp + 100)
    mant = rng.uniform(1.0, 2.0, 200000)
    w = (mant * 2.0 ** rng.integers(lo_exp, hi_exp, mant.size)).astype(np.float32)
    w = np.where(rng.random(w.size) < 0.5, -w, w).astype(np.float32)
    w = w[np.abs(w) < 65504]
    hi, lo = split_hi_lo(w)
    back = hi.astype(np.float64) + lo.astype(np.float64)
    err = np.abs(w.astype(np.float64) - back)
    assert (err <= 2.0 ** -22 * np.abs(w) + 2.0 ** -24).all(), err.max()
    normal = np.abs(w) >= 2.0 ** -14
    # hi is the weight's 11 leading bits, exactly (no rounding in the fp16 cast)
    assert np.array_equal(hi[normal].astype(np.float32),
                          (w[normal].view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32))


def test_single_fp16_rounding_is_not_enough():
    """Sensitivity: fp16(w) alone has errors up to 2^-12 |w|, far above the
    split's bound, so a dropped lo term would fail the bound above."""
    rng = np.random.default_rng(3)
    w = rng.uniform(0.5, 1.0, 10000).astype(np.float32)
    err = np.abs(w.astype(np.float64) - w.astype(np.float16).astype(np.float64))
    assert (err > 2.0 ** -22 * w + 2.0 ** -24).mean() > 0.9


def weight_scale_pow2(mx):
    """The power of two f with mx f in [2^13, 2^14) that the decode kernels
    apply to a tile's weights before the split (1 when mx is 0); the biased
    exponent of mx is clamped to [87, 254] as in the kernels."""
    mx = np.float32(mx)
    if not mx > 0:
        return np.float32(1.0)
    E = int(np.array(mx, np.float32).view(np.uint32) >> 23)
    E = min(max(E, 127 - 40), 254)
    return np.float32(2.0 ** (140 - E))


@pytest.mark.parametrize("stat_exp", [-30, -24, -12, 0, 8])
def test_scaled_split_is_relative_over_the_kernels_range(stat_exp):
    """Key weights q_d s_d of a tile, with statistics around 2^stat_exp
    (inputs scaled by 2^-12 put them near 2^-12 and below): scaled by the
    tile's power of two f, split, and scaled back, every weight is within
    2^-22 |w| + 2^-24 / f of itself (the split's bound carried through the
    exact scaling; 2^-24 / f is at most 2^-37 max|q| max s, the bound on
    the tile's weights that f is chosen from),
    and the tile's weights as a whole (what a dot product sees) are within
    2^-21 of their magnitude.  Without the scaling the tiles of small
    statistics lose that bound.  (f is at most 2^53: below max|q| max s =
    2^-40 only the absolute floor 2^-77 remains.)"""
    rng = np.random.default_rng(stat_exp + 1000)
    tiles = 400
    q = (rng.standard_normal((tiles, 128)) * 2.0).astype(np.float16).astype(np.float32)
    s = (rng.uniform(0.25, 1.0, (tiles, 128)) *
         2.0 ** (stat_exp + rng.integers(-6, 1, (tiles, 1)))).astype(np.float32)
    w = (q * s).astype(np.float32)
    worst_tile = worst_el = unscaled_tile = 0.0
    for t in range(tiles):
        qmax = float(np.abs(q[t]).max())
        f = weight_scale_pow2(np.float32(qmax) * np.float32(s[t].max()))
        ws = (w[t] * f).astype(np.float32)          # exact: f is a power of two
        assert np.abs(ws).max() < 2.0 ** 14
        hi, lo = split_hi_lo(ws)
        back = (hi.astype(np.float64) + lo.astype(np.float64)) / float(f)
        err = np.abs(w[t].astype(np.float64) - back)
        mag = np.abs(w[t].astype(np.float64))
        worst_tile = max(worst_tile, err.sum() / mag.sum())
        floor = 2.0 ** -24 / float(f)
        assert floor <= 2.0 ** -37 * qmax * float(s[t].max())
        worst_el = max(worst_el, (err / (2.0 ** -22 * mag + floor)).max())
        hu, lu = split_hi_lo(w[t])
        eu = np.abs(w[t].astype(np.float64) - (hu.astype(np.float64) + lu.astype(np.float64)))
        unscaled_tile = max(unscaled_tile, eu.sum() / mag.sum())
    assert worst_el <= 1.0, worst_el
    assert worst_tile <= 2.0 ** -21, worst_tile
    if stat_exp <= -24:
        # the unscaled split of such tiles is off by far more than 22 bits
        assert unscaled_tile > 2.0 ** -16, unscaled_tile
