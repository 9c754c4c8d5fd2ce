"""Compact payload and codec fingerprint, host side (no GPU): the FNV-1a hash
against the specification's test vectors, the library's fingerprint and
payload size against the oracle's, the oracle's payload layout and its round
trip, and the export / import argument checks that return before any CUDA
call.  (CacheSeek PR #4 change notes: a quantized layer is stored in host
memory as its codes, scales and offsets, and a fingerprint of the quantization
settings enters the prefix root hash.)"""
import ctypes as C
import struct

import numpy as np
import pytest

from conftest import golden

CODECS = [(128, 2, 2, 32, 128), (128, 4, 4, 32, 0), (128, 8, 8, 32, 0), (64, 4, 4, 32, 32),
          (256, 4, 4, 64, 64), (128, 2, 4, 32, 32), (128, 8, 2, 128, 128)]


def test_fnv1a64_specification_vectors(ref):
    rows = golden("fnv1a64.txt")
    assert len(rows) == 3
    for text, want in rows:
        assert ref.fnv1a64(text.encode()) == int(want, 16)


def test_fingerprint_matches_oracle_and_separates_codecs(kivi_lib, ref):
    from kivi_bit_kv_gb300 import abi
    seen = set()
    for D, bk, bv, G, R in CODECS:
        d = abi.kivi_cache(B=3, H=2, D=D, bits_k=bk, bits_v=bv, G=G, R=R, Tmax=4096)
        fp = abi.kivi_codec_fingerprint(d)
        assert fp == ref.codec_fingerprint(D, bk, bv, G, R)
        # B, H and Tmax are not part of the codec
        d2 = abi.kivi_cache(B=1, H=7, D=D, bits_k=bk, bits_v=bv, G=G, R=R, Tmax=G)
        assert abi.kivi_codec_fingerprint(d2) == fp
        seen.add(fp)
    assert len(seen) == len(CODECS)
    bad = abi.kivi_cache(B=1, H=1, D=96, bits_k=2, bits_v=2, G=32, R=0, Tmax=64)
    assert abi.kivi_codec_fingerprint(bad) == 0


@pytest.mark.parametrize("codec", CODECS)
def test_payload_bytes_match_oracle(kivi_lib, ref, codec):
    from kivi_bit_kv_gb300 import abi
    D, bk, bv, G, R = codec
    B, H, Tmax = 5, 3, 4096
    lens = [0, 1, R + G - 1, 2049, Tmax]
    d = abi.kivi_cache(B=B, H=H, D=D, bits_k=bk, bits_v=bv, G=G, R=R, Tmax=Tmax)
    n = abi.kivi_payload_bytes(d, lens)
    assert n == ref.payload_bytes(B, H, D, bk, bv, G, R, lens)
    per_slice = sum(abi.kivi_cache_bytes(t, D, bk, G, R, 0) + abi.kivi_cache_bytes(t, D, bv, G, R, 1)
                    for t in lens)
    assert n == 64 + 32 + H * per_slice
    assert abi.kivi_payload_bytes(d, [0, 1, 2, 3, Tmax + 1]) == 0
    assert abi.kivi_payload_bytes(d, [0, 1, 2, -1, 3]) == 0


def _encoded(ref, B=3, H=2, D=64, bk=2, bv=4, G=32, R=32, Tmax=320, T=300, lens=(300, 77, 0), seed=0):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((B, H, T, D)).astype(np.float16)
    V = rng.standard_normal((B, H, T, D)).astype(np.float16)
    return ref.RefCache(B, H, D, bk, bv, G, R, Tmax).encode(K, V, seq_lens=list(lens))


def test_oracle_payload_layout(ref):
    rc = _encoded(ref)
    p = rc.payload()
    assert bytes(p[:4]) == b"KIVP"
    magic, fmt, fp = struct.unpack_from("<IIQ", p, 0)
    assert (magic, fmt, fp) == (0x5056494B, 1, ref.codec_fingerprint(64, 2, 4, 32, 32))
    assert struct.unpack_from("<7i5i", p, 16) == (3, 2, 64, 2, 4, 32, 32, 0, 0, 0, 0, 0)
    assert struct.unpack_from("<4i", p, 64) == (300, 77, 0, 0)  # padded to 4 entries
    # first slice (b=0, h=0): kq rows of the Tq = 256 quantized tokens, then kscale
    o = 80
    Tq = 256
    kq = np.frombuffer(p[o:o + Tq // 16 * 64 * 4].tobytes(), "<i4").reshape(Tq // 16, 64)
    assert np.array_equal(kq, rc.kq[0, 0, :Tq // 16])
    o += kq.nbytes
    ks = np.frombuffer(p[o:o + Tq // 32 * 64 * 4].tobytes(), "<f4").reshape(Tq // 32, 64)
    assert np.array_equal(ks, rc.kscale[0, 0, :Tq // 32])
    assert len(p) == ref.payload_bytes(3, 2, 64, 2, 4, 32, 32, [300, 77, 0])


def test_oracle_payload_round_trip(ref):
    rc = _encoded(ref)
    rng = np.random.default_rng(1)
    for s in range(40):  # appends move the ring and flush groups
        rc.append(rng.standard_normal((3, 2, 64)).astype(np.float16),
                  rng.standard_normal((3, 2, 64)).astype(np.float16))
    p = rc.payload()
    rc2 = ref.RefCache.from_payload(p, 512)
    assert np.array_equal(rc2.lens, rc.lens)
    for which in (0, 1):
        assert np.array_equal(rc2.decode(which), rc.decode(which))
    q = rng.standard_normal((3, 4, 64)).astype(np.float16)
    for a, b in zip(rc.attention(q), rc2.attention(q)):
        assert np.array_equal(a, b)
    assert np.array_equal(rc2.payload(), p)


def test_export_import_reject_bad_buffers_before_launch(kivi_lib):
    """Argument errors that return before any CUDA call."""
    from kivi_bit_kv_gb300 import abi
    L = kivi_lib
    d = abi.kivi_cache(B=2, H=4, D=128, bits_k=2, bits_v=2, G=32, R=128, Tmax=4096)
    for i, name in enumerate(["kq", "kscale", "kzero", "vq", "vscale", "vzero", "kres", "vres", "len"]):
        setattr(d, name, 0x10000 + 0x100000 * (i + 1))
    ref = C.byref(d)
    assert L.kivi_export(ref, None, 1 << 20, 0x30000, None) == abi.KIVI_EINVAL
    assert L.kivi_export(ref, 0x20008, 1 << 20, 0x30000, None) == abi.KIVI_EINVAL   # misaligned
    assert L.kivi_export(ref, 0x20000, 64 + 15, 0x30000, None) == abi.KIVI_EINVAL   # < header + lens
    assert "header" in abi.kivi_last_error()
    assert L.kivi_import(ref, 0x20000, 1 << 20, None, None) == abi.KIVI_EINVAL      # status NULL
    assert L.kivi_import(ref, None, 1 << 20, 0x30000, None) == abi.KIVI_EINVAL
