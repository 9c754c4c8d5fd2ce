"""Pins of the CPU oracle against what the definitions and mathematics fix.

None of these tests compares the oracle with itself or with the CUDA path.
Each one checks the oracle against an independent statement: hand-worked
examples (tests/golden), numpy's IEEE binary16 conversion, exhaustive
enumeration of codes in numpy float32, exact rational arithmetic, closed
forms, textbook softmax attention in float64, and the streaming/prefix
equivalence of the append rule.  Together they are chosen so that a dropped
term, a wrong sign or index, a transposed layout or a wrong rounding mode in
the oracle fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

from conftest import golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f16(x):
    return np.asarray(x, dtype=np.float16)


def bits16(x):
    return f16(x).view(np.uint16)


# ------------------------------------------------------------ fp16 helpers --

def test_half_to_float_exhaustive(ref):
    """All 65536 binary16 patterns convert like numpy's float16 -> float32."""
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = pats.view(np.float16).astype(np.float32)
    got = np.array([ref.half_to_float(int(p)) for p in pats], dtype=np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_float_to_half_matches_numpy_rne(ref):
    """float32 -> binary16 rounds to nearest even exactly as numpy does, over
    random bit patterns, every fp16 value, and every fp16 midpoint."""
    rng = np.random.default_rng(123)
    r = rng.integers(0, 1 << 32, 60000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    r = r[np.isfinite(r)]
    small = rng.standard_normal(20000).astype(np.float32) * np.float32(1e-5)
    fp16vals = np.arange(0, 0x7C00, 7, dtype=np.uint16).view(np.float16).astype(np.float32)
    # midpoints between consecutive positive fp16 values (exact in fp32): ties
    a = np.arange(0, 0x7BFF, 5, dtype=np.uint16)
    lo = a.view(np.float16).astype(np.float64)
    hi = (a + 1).view(np.float16).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)
    xs = np.concatenate([r, small, fp16vals, -fp16vals, mids, -mids,
                         np.float32([65504, 65519.996, 65520, 65536, 1e-8, 2.0 ** -25,
                                     3 * 2.0 ** -25, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11])])
    want = xs.astype(np.float16).view(np.uint16)
    got = np.array([ref.float_to_half(float(x)) for x in xs], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(xs[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


# ---------------------------------------------------------- pack / unpack --

def test_pack_words_golden(ref):
    for bits, codes, word in golden("pack_words.txt"):
        bits = int(bits)
        codes = [int(c) for c in codes.split(",")]
        want = int(word, 16)
        got = ref.pack_word(codes, bits) & 0xFFFFFFFF
        assert got == want, (bits, codes, hex(got), word)
        assert list(ref.unpack_word(want, bits)) == codes


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_pack_unpack_identity(ref, bits):
    rng = np.random.default_rng(bits)
    P, M = 32 // bits, (1 << bits) - 1
    for _ in range(2000):
        codes = rng.integers(0, M + 1, P)
        w = ref.pack_word(codes, bits)
        assert list(ref.unpack_word(w, bits)) == list(codes)
        # the same word by plain integer arithmetic, code i weighted by 2^(i*b)
        assert (w & 0xFFFFFFFF) == sum(int(c) << (i * bits) for i, c in enumerate(codes))


# ------------------------------------------------------------------ groups --

def _rn16_of_fma(code, scale, zero) -> np.uint16:
    """fp16_rne(fmaf(code, scale, zero)) by exact rationals: one fp32 rounding
    of the exact c*s + z, then numpy's fp32 -> fp16 round to nearest even."""
    f = _rn32(Fraction(int(code)) * Fraction(float(scale)) + Fraction(float(zero)))
    return np.float32(f).astype(np.float16).view(np.uint16)


def test_groups_golden(ref):
    for bits, xs, scale_bits, zero, codes, xhat in golden("groups.txt"):
        bits = int(bits)
        x = f16([float(v) for v in xs.split(",")])
        s, z, c = ref.group_quantize(x, bits)
        assert np.float32(s).view(np.uint32) == np.uint32(int(scale_bits, 16)), (xs, s)
        assert np.float32(z).view(np.uint32) == np.float32(float(zero)).view(np.uint32), (xs, z)
        assert list(c) == [int(v) for v in codes.split(",")], (xs, list(c))
        # the fixture's x_hat column follows from its own codes / scale / zero
        want = bits16([float(v) for v in xhat.split(",")])
        got = np.array([_rn16_of_fma(ci, s, z) for ci in c], dtype=np.uint16)
        assert np.array_equal(got, want), (xs, got, want)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_decode_matches_exact_dequant(ref, bits):
    """Materialized keys and values equal fp16_rne(fmaf(code, scale, zero))
    formed with exact rationals, codes unpacked here by plain integer shifts
    (keys: word row t // P, code t % P; values: word d // P, code d % P)."""
    rng = np.random.default_rng(50 + bits)
    T, D, G, R = 96, 64, 32, 32
    K = f16(rng.standard_normal((1, 1, T, D)) * 4)
    V = f16(rng.standard_normal((1, 1, T, D)))
    rc = ref.RefCache(1, 1, D, bits, bits, G, R, 128).encode(K, V)
    P, M = 32 // bits, (1 << bits) - 1
    Tq = ref.quantized_tokens(T, G, R)
    dk, dv = rc.decode(0)[0, 0], rc.decode(1)[0, 0]
    for t in range(0, Tq, 5):
        for d in range(0, D, 3):
            wk = int(np.int32(rc.kq[0, 0, t // P, d]).view(np.uint32))
            ck = (wk >> ((t % P) * bits)) & M
            assert dk[t, d] == _rn16_of_fma(ck, rc.kscale[0, 0, t // G, d], rc.kzero[0, 0, t // G, d])
            wv = int(np.int32(rc.vq[0, 0, t, d // P]).view(np.uint32))
            cv = (wv >> ((d % P) * bits)) & M
            assert dv[t, d] == _rn16_of_fma(cv, rc.vscale[0, 0, t, d // G], rc.vzero[0, 0, t, d // G])


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_ramp_group_is_exact(ref, bits):
    """x = 0..M: scale 1, zero 0, codes equal x, reconstruction exact."""
    M = (1 << bits) - 1
    x = f16(np.arange(M + 1, dtype=np.float32))
    s, z, c = ref.group_quantize(x, bits)
    assert s == np.float32(1.0) and z == np.float32(0.0)
    assert list(c) == list(range(M + 1))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_codes_range_and_extremes(ref, bits):
    """Codes lie in [0, M]; the group minimum codes to 0 and the maximum to M."""
    rng = np.random.default_rng(bits + 10)
    M = (1 << bits) - 1
    for _ in range(300):
        x = f16(rng.standard_normal(32) * rng.uniform(0.01, 50))
        s, z, c = ref.group_quantize(x, bits)
        xf = x.astype(np.float32)
        assert c.min() >= 0 and c.max() <= M
        assert z == xf.min()
        if s > 0:
            assert c[np.argmin(xf)] == 0 and c[np.argmax(xf)] == M


def test_constant_group(ref):
    for bits in (2, 4, 8):
        for v in (0.0, -0.0, 1.5, -3.25, 60000.0):
            x = f16([v] * 32)
            s, z, c = ref.group_quantize(x, bits)
            assert s == 0.0 and (c == 0).all()
            assert np.float32(z).view(np.uint32) == np.float32(v + 0.0).view(np.uint32)


def test_round_half_even_ties(ref):
    """b=2, min 0, max 3 (scale exactly 1): 0.5 -> 0, 1.5 -> 2, 2.5 -> 2."""
    s, z, c = ref.group_quantize(f16([0.0, 3.0, 0.5, 1.5, 2.5]), 2)
    assert s == 1.0 and list(c) == [0, 3, 0, 2, 2]


# ------------------------------------------------------ brute-force encode --

def _rn32(fr: Fraction) -> np.float32:
    """Nearest float32 to an exact rational, ties to even."""
    f = np.float32(float(fr))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda v: (abs(Fraction(float(v)) - fr),
                                     int(np.array(v, dtype=np.float32).view(np.uint32)) & 1))


def _brute_group(x16, bits):
    """Re-derive one group in numpy float32: min/max scan, IEEE division, then
    the nearest code found by enumerating every candidate (ties to even)."""
    M = (1 << bits) - 1
    xf = x16.astype(np.float32) + np.float32(0.0)
    mn, mx = np.float32(xf.min()) + np.float32(0.0), np.float32(xf.max()) + np.float32(0.0)
    scale = np.float32(mx - mn) / np.float32(M)
    codes = []
    for v in xf:
        if scale == 0:
            codes.append(0)
            continue
        q = np.float32(np.float32(v - mn) / scale)
        cand = np.arange(M + 1)
        dist = np.abs(cand.astype(np.float64) - np.float64(q))
        best = cand[dist == dist.min()]
        codes.append(int(best[best % 2 == 0][0]) if best.size > 1 else int(best[0]))
    return np.float32(scale), np.float32(mn), codes


def _pack(codes, bits):
    out = 0
    for i, c in enumerate(codes):
        out |= int(c) << (i * bits)
    return np.uint32(out).view(np.int32)


@pytest.mark.parametrize("bits,G,R,T,D", [(2, 32, 0, 48, 32), (4, 32, 32, 47, 32),
                                          (8, 32, 0, 40, 64), (2, 64, 64, 200, 64)])
def test_encode_matches_brute_force(ref, bits, G, R, T, D):
    """Keys (per channel over G tokens) and values (per token over G channels)
    re-derived element by element in numpy float32 with exhaustive code search."""
    rng = np.random.default_rng(T + D + bits)
    K = f16(rng.standard_normal((1, 1, T, D)) * np.where(np.arange(D) % 7 == 3, 9.0, 1.0))
    V = f16(rng.standard_normal((1, 1, T, D)))
    Tmax = (T + G - 1) // G * G + G
    rc = ref.RefCache(1, 1, D, bits, bits, G, R, Tmax).encode(K, V)
    P, RG = 32 // bits, R + G
    Tq = max(0, (T - R) // G * G)
    Kf, Vf = K[0, 0], V[0, 0]
    for g in range(Tq // G):
        for d in range(D):
            s, z, codes = _brute_group(Kf[g * G:(g + 1) * G, d], bits)
            assert rc.kscale[0, 0, g, d] == s and rc.kzero[0, 0, g, d] == z
            for w in range(G // P):
                assert rc.kq[0, 0, g * (G // P) + w, d] == _pack(codes[w * P:(w + 1) * P], bits)
    for t in range(Tq):
        for g in range(D // G):
            s, z, codes = _brute_group(Vf[t, g * G:(g + 1) * G], bits)
            assert rc.vscale[0, 0, t, g] == s and rc.vzero[0, 0, t, g] == z
            for w in range(G // P):
                assert rc.vq[0, 0, t, g * (G // P) + w] == _pack(codes[w * P:(w + 1) * P], bits)
    for t in range(Tq, T):
        assert np.array_equal(rc.kres[0, 0, t % RG], Kf[t].view(np.uint16))
        assert np.array_equal(rc.vres[0, 0, t % RG], Vf[t].view(np.uint16))


def test_fp32_division_is_correctly_rounded(ref):
    """The quotients behind the codes are the correctly rounded fp32 values of
    (x - min) / scale, checked with exact rationals on sampled groups."""
    rng = np.random.default_rng(7)
    for bits in (2, 4, 8):
        M = (1 << bits) - 1
        for _ in range(40):
            x = f16(rng.standard_normal(32) * 3)
            s, z, c = ref.group_quantize(x, bits)
            exact_s = _rn32(Fraction(float(np.float32(x.astype(np.float32).max()) - z)) / M)
            assert np.float32(s) == exact_s
            for v, code in zip(x.astype(np.float32), c):
                a = np.float32(v - z)  # exact or correctly rounded fp32 subtraction
                assert a == _rn32(Fraction(float(v)) - Fraction(float(z)))
                q = _rn32(Fraction(float(a)) / Fraction(float(s)))
                fl = int(np.floor(q))
                frac = Fraction(float(q)) - fl
                want = fl + (1 if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and fl % 2) else 0)
                assert code == min(max(want, 0), M)


# ------------------------------------------------------------ error bound --

@pytest.mark.parametrize("bits", [2, 4, 8])
def test_dequant_error_bound(ref, bits):
    """|x - x_hat| <= scale/2 + half an fp16 ulp of x_hat + a few fp32 ulps."""
    rng = np.random.default_rng(bits + 99)
    T, D, G, R = 160, 64, 32, 32
    K = f16(rng.standard_normal((1, 2, T, D)) * np.where(np.arange(D) % 5 == 0, 15.0, 1.0))
    V = f16(rng.standard_normal((1, 2, T, D)))
    rc = ref.RefCache(1, 2, D, bits, bits, G, R, 192).encode(K, V)
    Tq = (T - R) // G * G
    M = (1 << bits) - 1
    for which, X in ((0, K), (1, V)):
        xh = rc.decode(which).view(np.float16).astype(np.float64)
        x = X.astype(np.float64)
        if which == 0:
            s = np.repeat(rc.kscale[:, :, :Tq // G], G, axis=2).astype(np.float64)
            z = np.repeat(rc.kzero[:, :, :Tq // G], G, axis=2).astype(np.float64)
        else:
            s = np.repeat(rc.vscale[:, :, :Tq], G, axis=3).astype(np.float64)
            z = np.repeat(rc.vzero[:, :, :Tq], G, axis=3).astype(np.float64)
        err = np.abs(x[:, :, :Tq] - xh[:, :, :Tq])
        ulp16 = np.spacing(np.abs(xh[:, :, :Tq]).astype(np.float16)).astype(np.float64)
        bound = s / 2 + ulp16 / 2 + 4 * 2.0 ** -24 * (np.abs(x[:, :, :Tq]) + np.abs(z) + s * M)
        assert (err <= bound).all()
        assert np.array_equal(xh[:, :, Tq:], x[:, :, Tq:])  # residual is verbatim


# ------------------------------------------------------------------ split --

def test_split_golden(ref):
    for T, G, R, Tq, res in golden("split.txt"):
        T, G, R, Tq, res = map(int, (T, G, R, Tq, res))
        assert ref.quantized_tokens(T, G, R) == Tq and T - Tq == res


# ------------------------------------------------------------------ bytes --

@pytest.mark.parametrize("T,bits,G,R", [(256, 4, 32, 32), (4096, 2, 32, 128), (2065, 4, 32, 0),
                                        (2065, 8, 32, 0), (100, 2, 32, 128), (1000, 2, 64, 64)])
def test_cache_bytes_closed_form(ref, T, bits, G, R):
    """Stored bytes = T.D.b/8 over the quantized tokens + fp32 (scale, zero)
    per group + 2 bytes per residual element, checked against the sizes of
    the arrays an encode actually writes."""
    D = 128
    rng = np.random.default_rng(T)
    K = f16(rng.standard_normal((1, 1, T, D)))
    rc = ref.RefCache(1, 1, D, bits, bits, G, R, (T + G - 1) // G * G + G).encode(K, K)
    Tq = ref.quantized_tokens(T, G, R)
    P = 32 // bits
    kbytes = (Tq // P) * D * 4 + 2 * (Tq // G) * D * 4 + (T - Tq) * D * 2
    vbytes = Tq * (D // P) * 4 + 2 * Tq * (D // G) * 4 + (T - Tq) * D * 2
    assert ref.cache_bytes(T, D, bits, G, R, 0) == kbytes
    assert ref.cache_bytes(T, D, bits, G, R, 1) == vbytes
    assert kbytes == Tq * D * bits // 8 + (Tq // G) * D * 8 + (T - Tq) * D * 2
    # the written rows are exactly those bytes: nothing past Tq is touched
    assert not rc.kq[0, 0, Tq // P:].any() and not rc.vq[0, 0, Tq:].any()


# ----------------------------------------------------- attention reduction --

def _exact_cache_tensor(rng, shape, axis, G):
    """Values (c - 128)/64 for c in 0..255 with every group along `axis`
    holding both 0 and 255: int8 quantization is then exact (scale 1/64,
    zero -2) and K_hat == K."""
    c = rng.integers(0, 256, shape)
    c = np.moveaxis(c, axis, -1).copy()
    c[..., 0::G] = 0
    c[..., 1::G] = 255
    c = np.moveaxis(c, -1, axis)
    return f16((c - 128) / 64.0)


@pytest.mark.parametrize("NQ", [1, 2])
def test_attention_reduces_to_textbook(ref, NQ):
    """With an exactly representable cache, decode attention equals
    softmax(q K^T * sm_scale) V computed by torch in float64."""
    import torch
    rng = np.random.default_rng(5 + NQ)
    B, H, D, G, R, T = 2, 2, 64, 32, 32, 150
    K = _exact_cache_tensor(rng, (B, H, T, D), axis=2, G=G)
    V = _exact_cache_tensor(rng, (B, H, T, D), axis=3, G=G)
    q = f16(rng.standard_normal((B, H * NQ, D)))
    rc = ref.RefCache(B, H, D, 8, 8, G, R, 192).encode(K, V)
    assert np.array_equal(rc.decode(0), K.view(np.uint16))
    sm = 0.125
    logits, out = rc.attention(q, sm_scale=sm)
    Kt = torch.from_numpy(K.astype(np.float64))
    Vt = torch.from_numpy(V.astype(np.float64))
    qt = torch.from_numpy(q.astype(np.float64)).view(B, H, NQ, D)
    s = torch.einsum("bhnd,bhtd->bhnt", qt, Kt) * sm
    o = torch.einsum("bhnt,bhtd->bhnd", torch.softmax(s, dim=-1), Vt)
    assert np.allclose(logits, s.reshape(B, H * NQ, T).numpy(), rtol=1e-6, atol=1e-6)
    assert np.allclose(out, o.reshape(B, H * NQ, D).numpy(), rtol=1e-6, atol=1e-6)
    # default scale: torch's scaled_dot_product_attention, whose own default
    # is 1/sqrt(D), with the KV head repeated for each of its query heads
    Kr = Kt.repeat_interleave(NQ, dim=1)
    Vr = Vt.repeat_interleave(NQ, dim=1)
    o_sdpa = torch.nn.functional.scaled_dot_product_attention(qt.reshape(B, H * NQ, 1, D), Kr, Vr)
    assert np.allclose(rc.attention(q)[1], o_sdpa.reshape(B, H * NQ, D).numpy(), rtol=1e-6, atol=1e-6)


def _exact_groups_tensor(rng, shape, axis, G, bits):
    """fp16 values z + c 2^e whose groups along `axis` (G elements) each have
    their own exponent e in {-8, -7, -6} and offset z (a multiple of 2^-8 in
    [-2, 2]), with codes c in [0, 2^b - 1] and both ends present.  Every value
    is exact in fp16 (|x| < 8, a multiple of 2^-8), the group's scale is
    exactly 2^e and its zero exactly z, so the b-bit codes reproduce the
    tensor exactly while the statistics differ from group to group."""
    M = (1 << bits) - 1
    x = np.moveaxis(np.empty(shape), axis, -1).copy()
    ng = x.shape[-1] // G
    lead = x.shape[:-1]
    e = rng.integers(-8, -5, lead + (ng,))
    z = rng.integers(-512, 513, lead + (ng,)) / 256.0
    c = rng.integers(0, M + 1, lead + (ng, G))
    c[..., 0] = 0
    c[..., 1] = M
    vals = z[..., None] + c * np.exp2(e)[..., None]
    x[...] = rng.integers(-512, 513, x.shape) / 256.0  # a ragged tail stays fp16
    x[..., :ng * G] = vals.reshape(lead + (ng * G,))
    out = f16(np.moveaxis(x, -1, axis))
    assert np.array_equal(out.astype(np.float64), np.moveaxis(x, -1, axis))
    return out


@pytest.mark.parametrize("bk,bv,NQ", [(8, 4, 1), (4, 8, 2), (2, 2, 3)])
def test_attention_with_per_group_statistics(ref, bk, bv, NQ):
    """Decode attention over a cache whose every key group (channel d, G
    tokens) and value group (token t, G channels) has its own exact scale and
    zero, at mixed widths: K_hat == K and V_hat == V exactly, so the result is
    textbook softmax attention in float64 -- but only if the dequantization
    inside the attention reads each element's own group statistics
    (CacheForge README, "How it works": per-channel key groups, per-token
    value groups)."""
    import torch
    rng = np.random.default_rng(40 + bk + 3 * bv + NQ)
    B, H, D, G, R, T = 2, 2, 64, 32, 32, 150
    K = _exact_groups_tensor(rng, (B, H, T, D), axis=2, G=G, bits=bk)
    V = _exact_groups_tensor(rng, (B, H, T, D), axis=3, G=G, bits=bv)
    q = f16(rng.standard_normal((B, H * NQ, D)))
    rc = ref.RefCache(B, H, D, bk, bv, G, R, 192).encode(K, V)
    Tq = ref.quantized_tokens(T, G, R)
    # the statistics really differ between neighbouring channels and groups
    assert not np.array_equal(rc.kscale[:, :, :Tq // G, 0::2], rc.kscale[:, :, :Tq // G, 1::2])
    assert not np.array_equal(rc.kzero[:, :, :Tq // G, 0::2], rc.kzero[:, :, :Tq // G, 1::2])
    assert not np.array_equal(rc.vscale[:, :, :Tq, 0], rc.vscale[:, :, :Tq, 1])
    assert np.array_equal(rc.decode(0), K.view(np.uint16))
    assert np.array_equal(rc.decode(1), V.view(np.uint16))
    sm = 0.125
    logits, out = rc.attention(q, sm_scale=sm)
    Kt = torch.from_numpy(K.astype(np.float64))
    Vt = torch.from_numpy(V.astype(np.float64))
    qt = torch.from_numpy(q.astype(np.float64)).view(B, H, NQ, D)
    s = torch.einsum("bhnd,bhtd->bhnt", qt, Kt) * sm
    o = torch.einsum("bhnt,bhtd->bhnd", torch.softmax(s, dim=-1), Vt)
    assert np.allclose(logits, s.reshape(B, H * NQ, T).numpy(), rtol=1e-6, atol=1e-6)
    assert np.allclose(out, o.reshape(B, H * NQ, D).numpy(), rtol=1e-6, atol=1e-6)


def test_ragged_lengths_equal_truncated_prefixes(ref):
    """Encoding a batch with seq_lens keeps, for each sequence b, what encoding
    its first seq_lens[b] tokens on their own gives: the codes and statistics
    of its quantized groups, the residual tokens in their ring slots, and the
    same materialized rows and attention (groups and sequences are
    independent)."""
    rng = np.random.default_rng(77)
    B, H, D, G, R, T, bk, bv = 4, 2, 64, 32, 32, 200, 4, 2
    lens = [200, 77, 5, 0]
    Pk, Pv, RG = 32 // bk, 32 // bv, R + G
    K = f16(rng.standard_normal((B, H, T, D)))
    V = f16(rng.standard_normal((B, H, T, D)))
    q = f16(rng.standard_normal((B, H, D)))
    rc = ref.RefCache(B, H, D, bk, bv, G, R, 224).encode(K, V, seq_lens=lens)
    dk, dv = rc.decode(0, T_out=T), rc.decode(1, T_out=T)
    lg, out = rc.attention(q)
    for b, n in enumerate(lens):
        one = ref.RefCache(1, H, D, bk, bv, G, R, 224).encode(K[b:b + 1, :, :n], V[b:b + 1, :, :n])
        Tq = ref.quantized_tokens(n, G, R)
        for name, rows in (("kq", Tq // Pk), ("kscale", Tq // G), ("kzero", Tq // G),
                           ("vq", Tq), ("vscale", Tq), ("vzero", Tq)):
            assert np.array_equal(getattr(rc, name)[b, :, :rows], getattr(one, name)[0, :, :rows]), (b, name)
        slots = [t % RG for t in range(Tq, n)]
        assert np.array_equal(rc.kres[b][:, slots], one.kres[0][:, slots]), b
        assert np.array_equal(rc.vres[b][:, slots], one.vres[0][:, slots]), b
        assert np.array_equal(dk[b, :, :n], one.decode(0, T_out=n)[0]), b
        assert np.array_equal(dv[b, :, :n], one.decode(1, T_out=n)[0]), b
        lg1, o1 = one.attention(q[b:b + 1])
        assert np.array_equal(lg[b, :, :n], lg1[0, :, :n]) and np.array_equal(out[b], o1[0]), b


def test_attention_gqa_mapping(ref):
    """Query head hq reads KV head hq // (Hq/H): permuting KV heads permutes
    the output blocks accordingly."""
    rng = np.random.default_rng(11)
    B, H, NQ, D, G, R, T = 1, 2, 2, 64, 32, 32, 100
    K = f16(rng.standard_normal((B, H, T, D)))
    V = f16(rng.standard_normal((B, H, T, D)))
    q = f16(rng.standard_normal((B, H * NQ, D)))
    a = ref.RefCache(B, H, D, 4, 4, G, R, 128).encode(K, V).attention(q)[1]
    b = ref.RefCache(B, H, D, 4, 4, G, R, 128).encode(K[:, ::-1].copy(), V[:, ::-1].copy())
    qs = np.concatenate([q[:, NQ:], q[:, :NQ]], axis=1)
    o = b.attention(qs)[1]
    assert np.array_equal(o[:, NQ:], a[:, :NQ]) and np.array_equal(o[:, :NQ], a[:, NQ:])


# ------------------------------------------------------ streaming append --

@pytest.mark.parametrize("bk,bv,G,R,T0,n", [(2, 2, 32, 128, 130, 100), (4, 8, 32, 0, 17, 80),
                                           (8, 4, 64, 64, 0, 200), (2, 4, 32, 32, 250, 33)])
def test_append_equals_prefix_encode(ref, bk, bv, G, R, T0, n):
    """Encoding T0 tokens and appending n one at a time gives the same cache
    (codes, stats, residual ring contents) as encoding the T0+n prefix."""
    rng = np.random.default_rng(T0 + n + G)
    B, H, D = 2, 2, 64
    T = T0 + n
    K = f16(rng.standard_normal((B, H, T, D)) * 3)
    V = f16(rng.standard_normal((B, H, T, D)))
    Tmax = (T + G - 1) // G * G + G
    a = ref.RefCache(B, H, D, bk, bv, G, R, Tmax).encode(K[:, :, :T0], V[:, :, :T0])
    for t in range(T0, T):
        assert not a.append(K[:, :, t], V[:, :, t]).any()
    b = ref.RefCache(B, H, D, bk, bv, G, R, Tmax).encode(K, V)
    Tq = ref.quantized_tokens(T, G, R)
    Pk, Pv, RG = 32 // bk, 32 // bv, R + G
    assert (a.lens == T).all()
    assert np.array_equal(a.kq[:, :, :Tq // Pk], b.kq[:, :, :Tq // Pk])
    assert np.array_equal(a.kscale[:, :, :Tq // G], b.kscale[:, :, :Tq // G])
    assert np.array_equal(a.kzero[:, :, :Tq // G], b.kzero[:, :, :Tq // G])
    assert np.array_equal(a.vq[:, :, :Tq], b.vq[:, :, :Tq])
    assert np.array_equal(a.vscale[:, :, :Tq], b.vscale[:, :, :Tq])
    assert np.array_equal(a.vzero[:, :, :Tq], b.vzero[:, :, :Tq])
    slots = [t % RG for t in range(Tq, T)]
    assert np.array_equal(a.kres[:, :, slots], b.kres[:, :, slots])
    assert np.array_equal(a.vres[:, :, slots], b.vres[:, :, slots])
    assert np.array_equal(a.decode(0), b.decode(0)) and np.array_equal(a.decode(1), b.decode(1))


def test_append_capacity(ref):
    """A full sequence is left untouched and reported; the others advance."""
    rng = np.random.default_rng(3)
    B, H, D, G, R = 2, 1, 64, 32, 0
    K = f16(rng.standard_normal((B, H, 64, D)))
    rc = ref.RefCache(B, H, D, 4, 4, G, R, 64).encode(K, K, seq_lens=[64, 10])
    over = rc.append(K[:, :, 0], K[:, :, 0])
    assert list(over) == [True, False] and list(rc.lens) == [64, 11]
