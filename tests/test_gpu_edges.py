"""GPU parity on the method's edge cases and on the extremes of fp16.

Each case runs the whole path through the C ABI -- prefix encode, both
materialize calls, the split decode (logits, then p . V) and the fused decode
attention -- and compares it with the CPU oracle on the same input bits:
codes, packed words, statistics and the residual ring bit for bit,
materialized fp16 exactly, logits and outputs within 2e-3 per row.

Cases (CacheForge README, "How it works": min/max statistics per key channel
and per value token; the arithmetic contract in include/kivi.h):
  - constant groups (scale 0, every code 0, reconstruction exact), among them
    an all-zero key channel, an all-zero token, and whole constant groups;
  - groups mixing -0 and +0, and groups holding only signed zeros;
  - groups that span the whole fp16 range, -65504 .. 65504;
  - keys and values scaled by 2^-12 (statistics and decode weights far below
    1) and by 2^6;
  - a zero query (uniform attention);
  - a long softmax tail: one token per sequence far above a few thousand
    tokens that each weigh about e^-9 but together carry a third of the mass.
"""
import numpy as np
import pytest
import torch

from _parity import (compare_attention, compare_dequant, compare_state, gpu_decode, gpu_encode,
                     new_cache, np16, roundup, state)
from kivi_bit_kv_gb300 import abi
from oracle import ref as R

pytestmark = pytest.mark.gpu


def _normal(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.float16)


def _run(cuda, K, V, q, bk, bv, G, Rr, seq_lens=None, sm_scale=None):
    B, H, T, D = K.shape
    Tmax = roundup(T + 40, G)
    cache = new_cache(B, H, D, bk, bv, G, Rr, Tmax, cuda)
    gpu_encode(cache, K, V, seq_lens)
    rc = R.RefCache(B, H, D, bk, bv, G, Rr, Tmax).encode(np16(K), np16(V), seq_lens=seq_lens)
    compare_state(state(cache), rc)
    for which in (0, 1):
        out = torch.zeros((B, H, T, D), dtype=torch.float16, device=cuda)
        abi.kivi_dequant(cache, which, out)
        torch.cuda.synchronize()
        ex, tot = compare_dequant(np16(out).view(np.uint16), rc.decode(which, T_out=T), rc.lens)
        assert ex == tot
    lg, o, fo = gpu_decode(cache, q, sm_scale)
    rlg, ro = rc.attention(np16(q), sm_scale=sm_scale)
    compare_attention(lg, o, rlg, ro, rc.lens, fused=fo)
    return rc, lg, o


WIDTHS = [(2, 2, 32, 128), (4, 4, 32, 32), (8, 8, 64, 64), (2, 4, 32, 128)]


@pytest.mark.parametrize("bk,bv,G,Rr", WIDTHS)
def test_constant_groups(cuda, bk, bv, G, Rr):
    B, H, Hq, D, T = 2, 2, 4, 128, 700
    K = _normal((B, H, T, D), 101, 2.0)
    V = _normal((B, H, T, D), 102)
    K[:, :, :, 5] = 0.0                       # an all-zero key channel
    K[:, :, :, 9] = 1.5                       # a constant key channel
    K[0, :, G:2 * G, :] = -3.25               # a whole constant key group row
    V[:, :, 7, :] = 0.0                       # an all-zero token
    V[:, :, 40, :] = 2.0                      # a constant token
    V[1, :, 100:140, 0:G] = 0.75              # constant value groups
    q = _normal((B, Hq, D), 103)
    rc, _, _ = _run(cuda, K, V, q, bk, bv, G, Rr)
    Tq = R.quantized_tokens(T, G, Rr)
    if Tq > 2 * G:
        # scale exactly 0 where the group is constant, and the zero point is the
        # value (group row 1 of sequence 0 is the constant -3.25 in every channel)
        assert (rc.kscale[:, :, :Tq // G, 5] == 0).all()
        assert (rc.kzero[1, :, :Tq // G, 5] == 0).all() and (rc.kzero[0, :, 0, 5] == 0).all()
        assert (rc.kscale[0, :, 1, :] == 0).all() and (rc.kzero[0, :, 1, :] == -3.25).all()
        assert (rc.vscale[:, :, 7, :] == 0).all()


@pytest.mark.parametrize("bk,bv,G,Rr", WIDTHS[:3])
def test_signed_zeros(cuda, bk, bv, G, Rr):
    B, H, Hq, D, T = 2, 2, 2, 128, 650
    g = np.random.default_rng(7)
    K = _normal((B, H, T, D), 111, 2.0).numpy()
    V = _normal((B, H, T, D), 112).numpy()
    for X in (K, V):
        z = g.random(X.shape) < 0.3
        X[z] = np.where(g.random(int(z.sum())) < 0.5, np.float16(-0.0), np.float16(0.0))
    K[:, :, 0:G, 3] = np.where(g.random((B, H, G)) < 0.5, np.float16(-0.0), np.float16(0.0))
    V[:, :, 11, 0:G] = np.where(g.random((B, H, G)) < 0.5, np.float16(-0.0), np.float16(0.0))
    assert np.signbit(K).any() and (np.signbit(K) & (K == 0)).any()
    q = _normal((B, Hq, D), 113)
    rc, _, _ = _run(cuda, torch.from_numpy(K), torch.from_numpy(V), q, bk, bv, G, Rr)
    # statistics never hold -0
    for name in ("kscale", "kzero", "vscale", "vzero"):
        a = getattr(rc, name)
        assert not (np.signbit(a) & (a == 0)).any(), name


@pytest.mark.parametrize("bk,bv,G,Rr", WIDTHS)
def test_fp16_extremes(cuda, bk, bv, G, Rr):
    """Groups spanning -65504 .. 65504 (the range 131008 is exact in fp32).
    The query is small so that the logits stay in a range where the softmax
    is not decided by single fp32 rounding steps."""
    B, H, Hq, D, T = 2, 2, 4, 128, 600
    g = torch.Generator().manual_seed(121)
    K = ((torch.rand((B, H, T, D), generator=g) * 2 - 1) * 65504).to(torch.float16)
    V = ((torch.rand((B, H, T, D), generator=g) * 2 - 1) * 65504).to(torch.float16)
    K[:, :, 0::G, :] = 65504.0
    K[:, :, 1::G, :] = -65504.0
    V[:, :, :, 0::G] = -65504.0
    V[:, :, :, 1::G] = 65504.0
    q = _normal((B, Hq, D), 123, 2.0 ** -12)
    _run(cuda, K, V, q, bk, bv, G, Rr)


@pytest.mark.parametrize("scale", [2.0 ** -12, 2.0 ** 6], ids=["x2^-12", "x2^6"])
@pytest.mark.parametrize("bk,bv,G,Rr", WIDTHS)
def test_scaled_inputs(cuda, bk, bv, G, Rr, scale):
    B, H, Hq, D, T = 2, 2, 4, 128, 1400
    K = _normal((B, H, T, D), 131, 2.0 * scale)
    V = _normal((B, H, T, D), 132, scale)
    q = _normal((B, Hq, D), 133)
    _run(cuda, K, V, q, bk, bv, G, Rr)


@pytest.mark.parametrize("bk,bv,G,Rr", WIDTHS[:2])
def test_zero_query(cuda, bk, bv, G, Rr):
    """q = 0: every logit is 0 and the output is the mean of V_hat."""
    B, H, Hq, D, T = 2, 2, 4, 128, 900
    K = _normal((B, H, T, D), 141, 2.0)
    V = _normal((B, H, T, D), 142)
    q = torch.zeros((B, Hq, D), dtype=torch.float16)
    _, lg, _ = _run(cuda, K, V, q, bk, bv, G, Rr)
    assert (lg[:, :, :T] == 0).all()


@pytest.mark.parametrize("bk,bv,G,Rr,Hq", [(2, 2, 32, 128, 2), (2, 2, 32, 128, 8), (4, 2, 32, 32, 4)])
def test_long_softmax_tail(cuda, bk, bv, G, Rr, Hq):
    """The query reads key channel 0 only.  One token per sequence sits about
    9 nats above all the others, which spread over half a nat: each tail token
    weighs about e^-9 of the peak, and the 4000 of them together about a third
    of the softmax mass.  Channel 0 of every key group holds only the peak
    value and tail values on a grid of 1/4, and the other channels do not
    reach the logits, so the whole tail lies deep in the small weights of the
    decode contractions."""
    B, H, D, T = 2, 2, 128, 4000
    g = torch.Generator().manual_seed(151)
    K = _normal((B, H, T, D), 152, 1.0)
    V = _normal((B, H, T, D), 153)
    tail = -15.5 + torch.randint(0, 3, (B, H, T), generator=g).to(torch.float32) / 4
    K[:, :, :, 0] = tail.to(torch.float16)
    K[0, :, 777, 0] = 10.0
    K[1, :, 3001, 0] = 10.0
    q = torch.zeros((B, Hq, D), dtype=torch.float16)
    q[:, :, 0] = 4.0
    _, lg, o = _run(cuda, K, V, q, bk, bv, G, Rr)
    s = lg[0, 0, :T].astype(np.float64)
    p = np.exp(s - s.max())
    assert 0.2 < (p.sum() - 1) / p.sum() < 0.5  # the tail carries a real share of the mass
