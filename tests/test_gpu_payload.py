"""GPU parity of the compact payload (include/kivi.h): kivi_export writes the
oracle's payload byte for byte (to pinned host memory and to device memory),
kivi_import of the oracle's payload reproduces the oracle's cache state and
decode output, and every header / capacity / size error is reported through
the status word with the cache or the destination left as it was.  (CacheSeek
PR #4 change notes: the store keeps the codes, scales and offsets in host
memory, and its root hash covers a fingerprint of the quantization settings.)"""
import numpy as np
import pytest
import torch

from _parity import (compare_attention, compare_state, gpu_decode, gpu_encode, new_cache, np16,
                     roundup, state)
from kivi_bit_kv_gb300 import abi
from oracle import ref as R

pytestmark = pytest.mark.gpu

# name, B, H, D, bits_k, bits_v, G, R, T, seq_lens, appends
CASES = [
    ("int2_ragged", 3, 2, 128, 2, 2, 32, 128, 700, [700, 1, 160], 37),
    ("int4_int8_R0", 2, 3, 64, 4, 8, 32, 0, 530, [530, 0], 5),
    ("int8_G128_d256", 2, 2, 256, 8, 8, 128, 128, 900, [900, 300], 130),
]


def f16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.float16)


def build(case, cuda):
    name, B, H, D, bk, bv, G, Rr, T, sl, n_app = case
    Tmax = roundup(T + n_app + 8, G)
    K, V = f16((B, H, T, D), 1, 2.0), f16((B, H, T, D), 2)
    cache = new_cache(B, H, D, bk, bv, G, Rr, Tmax, cuda)
    gpu_encode(cache, K, V, sl)
    rc = R.RefCache(B, H, D, bk, bv, G, Rr, Tmax).encode(np16(K), np16(V), seq_lens=sl)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    kn, vn = f16((n_app, B, H, D), 3, 2.0), f16((n_app, B, H, D), 4)
    for s in range(n_app):  # ring positions and flushed groups of every phase
        abi.kivi_append_token(cache, kn[s].to(cuda), vn[s].to(cuda), status)
        rc.append(np16(kn[s]), np16(vn[s]))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare_state(state(cache), rc)
    return cache, rc


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("where", ["pinned", "device"])
def test_export_matches_oracle_bytes(cuda, case, where):
    cache, rc = build(case, cuda)
    want = rc.payload()
    n = abi.kivi_payload_bytes(cache.desc, rc.lens)
    assert n == len(want)
    kw = dict(pin_memory=True) if where == "pinned" else dict(device=cuda)
    dst = torch.full((n + 48,), 0xA5, dtype=torch.uint8, **kw)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    abi.kivi_export(cache, dst, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = dst.cpu().numpy()
    assert np.array_equal(got[:n], want), np.argwhere(got[:n] != want)[:5].tolist()
    assert (got[n:] == 0xA5).all()  # nothing past the payload


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_import_reproduces_oracle_state(cuda, case):
    _, rc = build(case, cuda)
    name, B, H, D, bk, bv, G, Rr = case[:8]
    payload = torch.from_numpy(rc.payload()).pin_memory()
    fresh = new_cache(B, H, D, bk, bv, G, Rr, rc.Tmax + G, cuda)  # another Tmax is fine
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    abi.kivi_import(fresh, payload, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare_state(state(fresh), rc)
    Hq = 2 * H
    q = f16((B, Hq, D), 9)
    lg, o, fo = gpu_decode(fresh, q)
    rlg, ro = rc.attention(np16(q))
    compare_attention(lg, o, rlg, ro, rc.lens, fused=fo)


def test_import_errors_leave_cache_unchanged(cuda):
    cache, rc = build(CASES[0], cuda)
    name, B, H, D, bk, bv, G, Rr = CASES[0][:8]
    good = rc.payload()
    before = state(cache)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)

    def attempt(buf, target=cache):
        status.zero_()
        abi.kivi_import(target, torch.from_numpy(np.ascontiguousarray(buf)).pin_memory(), status)
        torch.cuda.synchronize()
        return int(status.item())

    bad_fp = good.copy()
    bad_fp[8] ^= 1                       # fingerprint
    assert attempt(bad_fp) == abi.KIVI_EINVAL
    bad_magic = good.copy()
    bad_magic[0] ^= 0xFF
    assert attempt(bad_magic) == abi.KIVI_EINVAL
    bad_h = good.copy()
    bad_h[20] += 1                       # H
    assert attempt(bad_h) == abi.KIVI_EINVAL
    assert attempt(good[:len(good) - 16]) == abi.KIVI_EWORKSPACE  # truncated
    for k, v in before.items():
        assert np.array_equal(state(cache)[k], v), k
    # another codec (value width): the fingerprint differs
    other = new_cache(B, H, D, bk, 4, G, Rr, rc.Tmax, cuda)
    assert attempt(good, other) == abi.KIVI_EINVAL
    # a sequence longer than the target's Tmax
    small = new_cache(B, H, D, bk, bv, G, Rr, roundup(int(rc.lens.max()) - 1, G) - G, cuda)
    small_before = state(small)
    assert attempt(good, small) == abi.KIVI_ECAPACITY
    for k, v in small_before.items():
        assert np.array_equal(state(small)[k], v), k


def test_export_into_short_buffer_writes_nothing(cuda):
    cache, rc = build(CASES[1], cuda)
    n = len(rc.payload())
    dst = torch.full((n - 16,), 0x5A, dtype=torch.uint8, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    abi.kivi_export(cache, dst, status)
    torch.cuda.synchronize()
    assert int(status.item()) == abi.KIVI_EWORKSPACE
    assert (dst.cpu().numpy() == 0x5A).all()


def test_payload_buffers_must_be_device_or_pinned(cuda):
    cache, _ = build(CASES[1], cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    with pytest.raises(ValueError):
        abi.kivi_export(cache, torch.zeros(1 << 16, dtype=torch.uint8), status)  # pageable
    buf = np.zeros(1 << 16, np.uint8)  # pageable host memory, through the C ABI directly
    L = abi.load()
    import ctypes as C
    st = L.kivi_export(C.byref(cache.desc), buf.ctypes.data, buf.nbytes, status.data_ptr(),
                       torch.cuda.current_stream().cuda_stream)
    assert st == abi.KIVI_EINVAL
    assert "pinned" in abi.kivi_last_error()
