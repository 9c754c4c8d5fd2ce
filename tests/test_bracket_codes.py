"""The encode kernels' bracketed code test, checked on the host with exact
arithmetic.

The kernels round each code twice, t_lo = rn(a inv_lo + 1.5 2^23) and
t_hi = rn(a inv_hi + 1.5 2^23), with inv = rn(1/scale),
inv_lo = rn(inv (1 - 2^-21)) and inv_hi = rn(inv (1 + 2^-21)).  They take
t_lo - 1.5 2^23 as the code whenever t_lo == t_hi, and redo the division only
when the two differ.  The argument (kivi_device.cuh, bracket_code_bits) says
that agreement implies the code of the IEEE quotient rn(a / scale), and that
a code taken this way never exceeds M.  Here both sides are computed exactly
in numpy: products of two fp32 values are exact in fp64, and in [2^23, 2^24)
the fp32 rounding of p + 1.5 2^23 is 1.5 2^23 + rint(p).  The inputs are
random groups and, above all, values placed within a few fp16 ulps of every
half-integer quotient, where a wrong bracket would show.
"""
import numpy as np
import pytest

C23 = np.float64(1.5 * 2.0 ** 23)


def _fp16_neighbours(x, k):
    """fp16 values within k ulps of x (x fp16)."""
    bits = x.astype(np.float16).view(np.uint16).astype(np.int32)
    out = []
    for d in range(-k, k + 1):
        b = bits + np.where(x >= 0, d, -d)
        out.append((b & 0xFFFF).astype(np.uint16).view(np.float16))
    return np.concatenate(out)


def _check(mn16, mx16, xs16, bits):
    """Checks every x of one group [mn, mx]; returns the counts of codes the
    bracket takes, of codes it sends to the division, and of codes a single
    rounding with inv alone would get wrong (the inputs reach hard cases)."""
    M = (1 << bits) - 1
    mn, mx = np.float32(mn16), np.float32(mx16)
    rng_ = np.float32(mx - mn)                       # fp32 subtraction
    scale = np.float32(rng_ / np.float32(M))         # IEEE division
    if scale == 0:
        return 0, 0, 0
    xs = xs16.astype(np.float32)
    xs = xs[(xs >= mn) & (xs <= mx) & np.isfinite(xs)]
    a = (xs - mn).astype(np.float32)                 # rn32(x - min)
    q = (a / scale).astype(np.float32)               # IEEE quotient
    code = np.clip(np.rint(q), 0, M)                 # ties to even
    inv = np.float32(np.float32(1.0) / scale)
    inv_lo = np.float32(np.float64(inv) * np.float64(np.float32(1.0 - 2.0 ** -21)))
    inv_hi = np.float32(np.float64(inv) * np.float64(np.float32(1.0 + 2.0 ** -21)))
    p_lo = a.astype(np.float64) * np.float64(inv_lo)  # exact: 24 x 24 bits
    p_hi = a.astype(np.float64) * np.float64(inv_hi)
    assert (p_lo + C23 < 2.0 ** 24).all() and (p_lo >= 0).all()
    t_lo, t_hi = np.rint(p_lo), np.rint(p_hi)
    agree = t_lo == t_hi
    assert (t_lo[agree] == code[agree]).all(), (mn16, mx16, a[agree][t_lo[agree] != code[agree]][:4])
    assert (t_lo[agree] <= M).all()
    naive_wrong = np.rint(a.astype(np.float64) * np.float64(inv)) != code
    return int(agree.sum()), int((~agree).sum()), int(naive_wrong.sum())


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_bracket_agreement_gives_the_ieee_code(bits):
    rng = np.random.default_rng(1000 + bits)
    M = (1 << bits) - 1
    agreed = redone = naive_wrong = 0
    for _ in range(300):
        lo, hi = np.sort(rng.standard_normal(2) * rng.choice([1e-3, 0.1, 1.0, 30.0, 2000.0]))
        mn16, mx16 = np.float16(lo), np.float16(hi)
        if not (np.isfinite(mn16) and np.isfinite(mx16)) or mn16 >= mx16:
            continue
        mn, mx = np.float32(mn16), np.float32(mx16)
        scale = np.float32(np.float32(mx - mn) / np.float32(M))
        # near every half-integer quotient, a few fp16 ulps either side
        centres = (mn + (np.arange(M) + 0.5) * np.float64(scale)).astype(np.float16)
        xs = np.concatenate([_fp16_neighbours(centres, 3),
                             rng.uniform(mn, mx, 64).astype(np.float16), np.array([mn16, mx16])])
        ag, rd, nw = _check(mn16, mx16, xs, bits)
        agreed += ag
        redone += rd
        naive_wrong += nw
    assert agreed > 20000
    assert naive_wrong > 0  # one rounding with inv alone is not enough here
    # the exact division is rare even among near-ties (random inputs: ~2^(b-20))
    assert redone < 0.05 * agreed, (agreed, redone)
