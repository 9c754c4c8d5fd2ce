"""ctypes front end of the CPU oracle, over numpy arrays.

TEST INFRASTRUCTURE ONLY.  Every function here marshals numpy arrays into the
plain C oracle (kivi_ref.c) one (batch, head) slice at a time; none of the
method's arithmetic lives in Python.  ``RefCache`` mirrors the device cache
layout so that its arrays can be compared with the CUDA library's buffers
element by element:

    kq   int32 [B, H, Tmax/Pk, D]     kscale, kzero  fp32 [B, H, Tmax/G, D]
    vq   int32 [B, H, Tmax, D/Pv]     vscale, vzero  fp32 [B, H, Tmax, D/G]
    kres, vres  fp16 bits (uint16) [B, H, R+G, D]
    lens int32 [B]

Slices are independent, so a thread pool may run them on several host cores;
ctypes releases the GIL for the duration of each C call.
"""
from __future__ import annotations

import ctypes as C
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

_LIB = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_VP = C.c_void_p


def lib():
    """Load the oracle library, building it first if it is missing or stale.

    KIVI_REF_LIB, when set, names another build of kivi_ref.c to load instead:
    the planted-mistake tests point it at deliberately broken copies to show
    that the pins reject them."""
    global _LIB
    if _LIB is None:
        path = os.environ.get("KIVI_REF_LIB") or _build.build()
        L = C.CDLL(path)
        L.kref_half_to_float.argtypes = [C.c_uint16]
        L.kref_half_to_float.restype = C.c_float
        L.kref_float_to_half.argtypes = [C.c_float]
        L.kref_float_to_half.restype = C.c_uint16
        L.kref_quantized_tokens.argtypes = [C.c_int] * 3
        L.kref_quantized_tokens.restype = C.c_int
        L.kref_group_quantize.argtypes = [_u16p, C.c_int, C.c_long, C.c_int,
                                          C.POINTER(C.c_float), C.POINTER(C.c_float), _i32p]
        L.kref_group_quantize.restype = None
        L.kref_pack_word.argtypes = [_i32p, C.c_int]
        L.kref_pack_word.restype = C.c_int32
        L.kref_unpack_word.argtypes = [C.c_int32, C.c_int, _i32p]
        L.kref_unpack_word.restype = None
        enc = [_VP, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, _VP, _VP, _VP, _VP]
        L.kref_encode_keys.argtypes = enc
        L.kref_encode_values.argtypes = enc
        dec = [_VP, _VP, _VP, _VP, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, _VP]
        L.kref_decode_keys.argtypes = dec
        L.kref_decode_values.argtypes = dec
        L.kref_append.argtypes = [_VP] * 8 + [C.c_int, _VP, _VP] + [C.c_int] * 6
        L.kref_append.restype = C.c_int
        L.kref_attention.argtypes = ([_VP, C.c_int, C.c_float, C.c_int, C.c_int,
                                      C.c_int, C.c_int, C.c_int, C.c_int]
                                     + [_VP] * 8 + [_VP, _VP])
        L.kref_attention.restype = None
        L.kref_cache_bytes.argtypes = [C.c_int] * 6
        L.kref_cache_bytes.restype = C.c_size_t
        L.kref_fnv1a64.argtypes = [_VP, C.c_size_t]
        L.kref_fnv1a64.restype = C.c_uint64
        L.kref_codec_fingerprint.argtypes = [C.c_int] * 5
        L.kref_codec_fingerprint.restype = C.c_uint64
        L.kref_payload_header.argtypes = [_VP] + [C.c_int] * 7 + [_VP]
        L.kref_payload_header.restype = C.c_size_t
        io = [_VP] + [C.c_int] * 6 + [_VP] * 8
        L.kref_payload_put_slice.argtypes = io
        L.kref_payload_put_slice.restype = C.c_size_t
        L.kref_payload_get_slice.argtypes = io
        L.kref_payload_get_slice.restype = C.c_size_t
        _LIB = L
    return _LIB


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(C.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


# ---------------------------------------------------------------- scalars --

def half_to_float(h: int) -> float:
    return float(lib().kref_half_to_float(int(h)))


def float_to_half(f: float) -> int:
    return int(lib().kref_float_to_half(float(f)))


def quantized_tokens(T: int, G: int, R: int) -> int:
    return int(lib().kref_quantized_tokens(T, G, R))


def group_quantize(x, bits: int):
    """Quantize one group of fp16 values; returns (scale, zero, codes)."""
    x = _u16(x).ravel()
    s, z = C.c_float(), C.c_float()
    codes = np.zeros(x.size, np.int32)
    lib().kref_group_quantize(x, x.size, 1, bits, C.byref(s), C.byref(z), codes)
    return np.float32(s.value), np.float32(z.value), codes


def pack_word(codes, bits: int) -> int:
    c = np.ascontiguousarray(codes, dtype=np.int32)
    assert c.size == 32 // bits
    return int(lib().kref_pack_word(c, bits))


def unpack_word(word: int, bits: int) -> np.ndarray:
    out = np.zeros(32 // bits, np.int32)
    lib().kref_unpack_word(np.int32(np.uint32(word & 0xFFFFFFFF).view(np.int32)), bits, out)
    return out


def cache_bytes(T: int, D: int, bits: int, G: int, R: int, which: int) -> int:
    return int(lib().kref_cache_bytes(T, D, bits, G, R, which))


# ------------------------------------------------------------------ cache --

def _pool_map(fn, items, threads: int):
    if threads <= 1:
        for it in items:
            fn(it)
        return
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fn, items))


class RefCache:
    """Host copy of a KIVI cache in the device layout (see module docstring)."""

    def __init__(self, B, H, D, bits_k, bits_v, G, R, Tmax):
        assert Tmax % G == 0
        self.B, self.H, self.D = B, H, D
        self.bits_k, self.bits_v, self.G, self.R, self.Tmax = bits_k, bits_v, G, R, Tmax
        Pk, Pv, RG = 32 // bits_k, 32 // bits_v, R + G
        self.kq = np.zeros((B, H, Tmax // Pk, D), np.int32)
        self.kscale = np.zeros((B, H, Tmax // G, D), np.float32)
        self.kzero = np.zeros((B, H, Tmax // G, D), np.float32)
        self.vq = np.zeros((B, H, Tmax, D // Pv), np.int32)
        self.vscale = np.zeros((B, H, Tmax, D // G), np.float32)
        self.vzero = np.zeros((B, H, Tmax, D // G), np.float32)
        self.kres = np.zeros((B, H, RG, D), np.uint16)
        self.vres = np.zeros((B, H, RG, D), np.uint16)
        self.lens = np.zeros((B,), np.int32)

    # -- prefix encode ------------------------------------------------------
    def encode(self, K, V, seq_lens=None, threads: int = 1, slices=None):
        """Encode a prefix K, V [B, H, T, D] (fp16); seq_lens[b] <= T tokens
        of sequence b are kept (all T when None).  ``slices`` restricts the
        work to a list of (b, h) pairs (the others are left untouched)."""
        K, V = _u16(K), _u16(V)
        B, H, T, D = K.shape
        assert (B, H, D) == (self.B, self.H, self.D) and V.shape == K.shape
        lens = np.full(B, T, np.int32) if seq_lens is None else np.asarray(seq_lens, np.int32)
        assert (lens <= T).all() and (lens <= self.Tmax).all()
        self.lens[:] = lens
        L = lib()

        def one(bh):
            b, h = bh
            Tb = int(lens[b])
            kin = np.ascontiguousarray(K[b, h, :Tb])
            vin = np.ascontiguousarray(V[b, h, :Tb])
            L.kref_encode_keys(_p(kin), Tb, D, self.bits_k, self.G, self.R,
                               _p(self.kq[b, h]), _p(self.kscale[b, h]),
                               _p(self.kzero[b, h]), _p(self.kres[b, h]))
            L.kref_encode_values(_p(vin), Tb, D, self.bits_v, self.G, self.R,
                                 _p(self.vq[b, h]), _p(self.vscale[b, h]),
                                 _p(self.vzero[b, h]), _p(self.vres[b, h]))

        items = slices if slices is not None else [(b, h) for b in range(B) for h in range(H)]
        _pool_map(one, items, threads)
        return self

    # -- materialize --------------------------------------------------------
    def decode(self, which: int, T_out: int | None = None, threads: int = 1, slices=None):
        """Materialize keys (which=0) or values (which=1) as fp16 bits
        [B, H, T_out, D]; rows at or past lens[b] are left zero."""
        T_out = int(self.lens.max()) if T_out is None else T_out
        out = np.zeros((self.B, self.H, T_out, self.D), np.uint16)
        L = lib()

        def one(bh):
            b, h = bh
            n = int(self.lens[b])
            o = np.zeros((max(n, 1), self.D), np.uint16)
            if which == 0:
                L.kref_decode_keys(_p(self.kq[b, h]), _p(self.kscale[b, h]), _p(self.kzero[b, h]),
                                   _p(self.kres[b, h]), n, self.D, self.bits_k, self.G, self.R, _p(o))
            else:
                L.kref_decode_values(_p(self.vq[b, h]), _p(self.vscale[b, h]), _p(self.vzero[b, h]),
                                     _p(self.vres[b, h]), n, self.D, self.bits_v, self.G, self.R, _p(o))
            out[b, h, :n] = o[:n]

        items = slices if slices is not None else [(b, h) for b in range(self.B) for h in range(self.H)]
        _pool_map(one, items, threads)
        return out

    # -- append -------------------------------------------------------------
    def append(self, k, v):
        """Append one token k, v [B, H, D] (fp16) to every sequence.  Returns a
        bool array [B]: True where the sequence was full and nothing changed."""
        k, v = _u16(k), _u16(v)
        assert k.shape == (self.B, self.H, self.D) and v.shape == k.shape
        L = lib()
        overflow = np.zeros(self.B, bool)
        for b in range(self.B):
            n = int(self.lens[b])
            new = n
            for h in range(self.H):
                kin = np.ascontiguousarray(k[b, h])
                vin = np.ascontiguousarray(v[b, h])
                new = L.kref_append(_p(self.kq[b, h]), _p(self.kscale[b, h]), _p(self.kzero[b, h]),
                                    _p(self.kres[b, h]), _p(self.vq[b, h]), _p(self.vscale[b, h]),
                                    _p(self.vzero[b, h]), _p(self.vres[b, h]), n, _p(kin), _p(vin),
                                    self.D, self.bits_k, self.bits_v, self.G, self.R, self.Tmax)
            if new < 0:
                overflow[b] = True
            else:
                self.lens[b] = new
        return overflow

    # -- decode attention ---------------------------------------------------
    def attention(self, q, sm_scale: float | None = None, threads: int = 1, slices=None):
        """Decode attention for q [B, Hq, D] (fp16), Hq a multiple of H; query
        head hq reads KV head hq // (Hq // H).  Returns (logits, out): logits
        fp32 [B, Hq, max(lens)] (zero past lens[b]) and out fp32 [B, Hq, D].
        ``slices`` restricts the work to a list of (b, h) KV slices."""
        q = _u16(q)
        B, Hq, D = q.shape
        assert B == self.B and D == self.D and Hq % self.H == 0
        NQ = Hq // self.H
        sm = float(1.0 / np.sqrt(D)) if sm_scale is None else float(sm_scale)
        Tl = max(int(self.lens.max()), 1)
        logits = np.zeros((B, Hq, Tl), np.float32)
        out = np.zeros((B, Hq, D), np.float32)
        L = lib()

        def one(bh):
            b, h = bh
            n = int(self.lens[b])
            qs = np.ascontiguousarray(q[b, h * NQ:(h + 1) * NQ])
            lg = np.zeros((NQ, max(n, 1)), np.float32)
            o = np.zeros((NQ, D), np.float32)
            L.kref_attention(_p(qs), NQ, C.c_float(sm), n, D, self.bits_k, self.bits_v, self.G, self.R,
                             _p(self.kq[b, h]), _p(self.kscale[b, h]), _p(self.kzero[b, h]), _p(self.kres[b, h]),
                             _p(self.vq[b, h]), _p(self.vscale[b, h]), _p(self.vzero[b, h]), _p(self.vres[b, h]),
                             _p(lg), _p(o))
            logits[b, h * NQ:(h + 1) * NQ, :n] = lg[:, :n]
            out[b, h * NQ:(h + 1) * NQ] = o

        items = slices if slices is not None else [(b, h) for b in range(B) for h in range(self.H)]
        _pool_map(one, items, threads)
        return logits, out


def fnv1a64(data: bytes) -> int:
    """FNV-1a 64 of a byte string (the C oracle's kref_fnv1a64)."""
    buf = np.frombuffer(bytes(data) or b"\0", np.uint8).copy()
    return int(lib().kref_fnv1a64(_p(buf), len(data)))


def codec_fingerprint(D: int, bits_k: int, bits_v: int, G: int, R: int) -> int:
    return int(lib().kref_codec_fingerprint(D, bits_k, bits_v, G, R))


def payload_bytes(B, H, D, bits_k, bits_v, G, R, lens) -> int:
    """Size of the compact payload: header, padded len table, slices."""
    L = lib()
    n = 64 + (B + 3) // 4 * 16
    for b in range(B):
        t = int(lens[b])
        n += H * (L.kref_cache_bytes(t, D, bits_k, G, R, 0) + L.kref_cache_bytes(t, D, bits_v, G, R, 1))
    return n


def _payload(self) -> np.ndarray:
    """The cache's compact payload (kref_payload_header, then the slices in
    (b, h) order through kref_payload_put_slice) as a uint8 array."""
    L = lib()
    B, H = self.B, self.H
    total = payload_bytes(B, H, self.D, self.bits_k, self.bits_v, self.G, self.R, self.lens)
    out = np.zeros(total, np.uint8)
    lens = np.ascontiguousarray(self.lens, np.int32)
    o = L.kref_payload_header(_p(out), B, H, self.D, self.bits_k, self.bits_v, self.G, self.R, _p(lens))
    for b in range(B):
        for h in range(H):
            o += L.kref_payload_put_slice(
                out.ctypes.data + o, int(lens[b]), self.D, self.bits_k, self.bits_v, self.G, self.R,
                _p(self.kq[b, h]), _p(self.kscale[b, h]), _p(self.kzero[b, h]), _p(self.kres[b, h]),
                _p(self.vq[b, h]), _p(self.vscale[b, h]), _p(self.vzero[b, h]), _p(self.vres[b, h]))
    assert o == total
    return out


def _from_payload(cls, buf, Tmax: int) -> "RefCache":
    """A RefCache of capacity Tmax holding the payload `buf` (header fields
    unpacked here; the slices through kref_payload_get_slice)."""
    import struct
    buf = np.ascontiguousarray(np.frombuffer(bytes(buf), np.uint8))
    magic, fmt, fp = struct.unpack_from("<IIQ", buf, 0)
    B, H, D, bits_k, bits_v, G, R = struct.unpack_from("<7i", buf, 16)
    assert magic == 0x5056494B and fmt == 1, (hex(magic), fmt)
    assert fp == codec_fingerprint(D, bits_k, bits_v, G, R)
    lens = np.frombuffer(buf[64:64 + 4 * B].tobytes(), "<i4").astype(np.int32)
    rc = cls(B, H, D, bits_k, bits_v, G, R, Tmax)
    rc.lens[:] = lens
    L = lib()
    o = 64 + (B + 3) // 4 * 16
    for b in range(B):
        for h in range(H):
            o += L.kref_payload_get_slice(
                buf.ctypes.data + o, int(lens[b]), D, bits_k, bits_v, G, R,
                _p(rc.kq[b, h]), _p(rc.kscale[b, h]), _p(rc.kzero[b, h]), _p(rc.kres[b, h]),
                _p(rc.vq[b, h]), _p(rc.vscale[b, h]), _p(rc.vzero[b, h]), _p(rc.vres[b, h]))
    assert o == len(buf), (o, len(buf))
    return rc


RefCache.payload = _payload
RefCache.from_payload = classmethod(_from_payload)


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
