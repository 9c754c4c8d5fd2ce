"""The decode kernels' hi/lo fp16 split of a weight, checked on the host.

A weight w (q_d s_gd for the keys, p_t s_tg for the values, fp32) enters the
fp16 tensor-core products as two halves: hi = fp16(w with its 13 low
mantissa bits cleared), exact in fp16 when w is a normal fp16 value, and
lo = fp16_rn(w - hi) (csrc/decode_mma.cuh, split_hi_lo).  The pair carries
about 22 significant bits: |w - (hi + lo)| <= 2^-22 |w| + 2^-24.  The last
term covers weights below the fp16 normal range (2^-14), where hi and lo
are each rounded to the subnormal spacing 2^-24 (half of it each).  The
kernels keep |w| below the fp16 maximum: q is scaled by a power of two to a maximum
in [1/2, 1), the softmax weights are at most 1, and a scale (max - min)/M of
fp16 data is below 65504.
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
