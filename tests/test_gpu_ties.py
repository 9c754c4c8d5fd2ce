"""GPU parity on inputs built to sit on or next to rounding boundaries: every
group's quotients (x - min) / scale lie at half-integers (exact ties, which
round to even) or a few fp16 ulps away from them, with scales of exactly 1 and
slightly off 1.  The kernels' fast codes must hand every such element to the
exact IEEE-quotient path; codes, statistics and rings must equal the oracle's
bit for bit -- for the staged key encode, the unstaged one (D = 256, G = 128),
the value encode and the append flush."""
import numpy as np
import pytest
import torch

from _parity import compare_state, gpu_encode, new_cache, np16, roundup, state
from kivi_bit_kv_gb300 import abi
from oracle import ref as R

pytestmark = pytest.mark.gpu

SCALES = (1.0, 1.0 + 2.0 ** -10, 1.0 - 2.0 ** -11, 0.75, 3.0)


def tie_groups(n_groups, G, bits, rng):
    """[n_groups, G] fp16 values: element 0 is 0 (the min), element 1 is
    M s (the max), the rest (k + 1/2) s shifted by -2..2 fp16 ulps."""
    M = (1 << bits) - 1
    s = np.asarray(SCALES)[rng.integers(0, len(SCALES), n_groups)][:, None]
    k = rng.integers(0, M, (n_groups, G))
    x = ((k + 0.5) * s).astype(np.float16)
    step = rng.integers(-2, 3, (n_groups, G)).astype(np.int16)
    x = (x.view(np.int16) + step).view(np.float16)
    x = np.clip(x, np.float16(0), (M * s).astype(np.float16))
    x[:, 0] = 0
    x[:, 1] = (M * s[:, 0]).astype(np.float16)
    return x


def tie_kv(B, H, T, D, bits_k, bits_v, G, seed):
    rng = np.random.default_rng(seed)
    ng = T // G
    # keys: groups of G tokens per channel
    kg = tie_groups(B * H * D * ng, G, bits_k, rng).reshape(B, H, D, ng, G)
    K = np.ascontiguousarray(kg.transpose(0, 1, 3, 4, 2).reshape(B, H, T, D))
    # values: groups of G channels per token
    vg = tie_groups(B * H * T * (D // G), G, bits_v, rng)
    V = np.ascontiguousarray(vg.reshape(B, H, T, D))
    return K, V


def count_near_ties(x, bits, G, axis_tokens):
    """Quotients within 1e-5 of a half-integer, from the oracle's own stats."""
    M = (1 << bits) - 1
    xf = x.astype(np.float64)
    if axis_tokens:  # keys: [.., T, D] -> groups over T
        g = xf.reshape(*xf.shape[:-2], -1, G, xf.shape[-1])
        mn, mx = g.min(axis=-2, keepdims=True), g.max(axis=-2, keepdims=True)
    else:
        g = xf.reshape(*xf.shape[:-1], -1, G)
        mn, mx = g.min(axis=-1, keepdims=True), g.max(axis=-1, keepdims=True)
    sc = np.float32(mx - mn) / np.float32(M)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (g - mn) / sc
    f = np.abs(q - np.floor(q) - 0.5)
    return int(np.nansum(f < 1e-5))


CASES = [  # B, H, D, bits_k, bits_v, G, R, T
    (2, 2, 128, 2, 2, 32, 0, 512),
    (1, 2, 128, 4, 4, 32, 32, 384),
    (1, 2, 128, 8, 8, 32, 0, 256),
    (1, 1, 256, 2, 4, 128, 0, 512),   # unstaged key encode (D = 256, G = 128)
    (1, 2, 64, 8, 2, 64, 64, 384),
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[3]}{c[4]}_D{c[2]}_G{c[5]}" for c in CASES])
def test_encode_ties_bit_exact(cuda, case):
    B, H, D, bk, bv, G, Rr, T = case
    K, V = tie_kv(B, H, T, D, bk, bv, G, seed=T + D)
    assert count_near_ties(K, bk, G, True) > 100 and count_near_ties(V, bv, G, False) > 100
    cache = new_cache(B, H, D, bk, bv, G, Rr, roundup(T + 2 * G, G), cuda)
    gpu_encode(cache, torch.from_numpy(K), torch.from_numpy(V))
    rc = R.RefCache(B, H, D, bk, bv, G, Rr, cache.Tmax).encode(K, V)
    compare_state(state(cache), rc)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_append_flush_ties_bit_exact(cuda, bits):
    """Tokens appended one at a time until groups flush through the append
    kernel's quantizers."""
    B, H, D, G, Rr = 2, 2, 128, 32, 32
    T0, n = 40, 3 * G
    K, V = tie_kv(B, H, T0 + n + G - (T0 + n) % G, D, bits, bits, G, seed=bits)
    K, V = K[:, :, :T0 + n], V[:, :, :T0 + n]
    cache = new_cache(B, H, D, bits, bits, G, Rr, roundup(T0 + n + G, G), cuda)
    gpu_encode(cache, torch.from_numpy(np.ascontiguousarray(K[:, :, :T0])),
               torch.from_numpy(np.ascontiguousarray(V[:, :, :T0])))
    rc = R.RefCache(B, H, D, bits, bits, G, Rr, cache.Tmax).encode(K[:, :, :T0], V[:, :, :T0])
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    for t in range(T0, T0 + n):
        kt = np.ascontiguousarray(K[:, :, t])
        vt = np.ascontiguousarray(V[:, :, t])
        abi.kivi_append_token(cache, torch.from_numpy(kt).to(cuda), torch.from_numpy(vt).to(cuda), status)
        rc.append(kt, vt)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare_state(state(cache), rc)
