"""ctypes binding of libkivi (include/kivi.h), one Python function per C entry point.

Argument marshalling only: tensors are checked for dtype, device, shape and
contiguity, their device pointers and the current CUDA stream are passed to the
C library, and a non-zero status raises :class:`KiviError`.  Every step of the
method runs in the library's CUDA kernels; there is no Python or CPU fallback,
and a missing library is an error.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# KIVI_LIB selects another in-tree build of the library (the bounds-checked
# one, libkivi_checked.so); by default libkivi.so next to this file.
LIB_PATH = os.environ.get("KIVI_LIB") or os.path.join(HERE, "libkivi.so")

KIVI_OK = 0
KIVI_EINVAL = 1
KIVI_ECAPACITY = 2
KIVI_ECUDA = 3
KIVI_ETIMEOUT = 4
KIVI_EWORKSPACE = 5
KIVI_ECHECK = 6

(KIVI_BUF_KQ, KIVI_BUF_KSCALE, KIVI_BUF_KZERO, KIVI_BUF_VQ, KIVI_BUF_VSCALE, KIVI_BUF_VZERO,
 KIVI_BUF_KRES, KIVI_BUF_VRES, KIVI_BUF_LEN) = range(9)

# Every symbol include/kivi.h declares.
EXPORTS = (
    "kivi_abi_version", "kivi_status_string", "kivi_last_error", "kivi_cache_validate",
    "kivi_buffer_bytes", "kivi_cache_bytes", "kivi_quant_keys", "kivi_quant_values",
    "kivi_dequant", "kivi_append_token", "kivi_decode_qk", "kivi_decode_pv",
    "kivi_workspace_bytes", "kivi_decode_pv_noalloc", "kivi_decode_attention",
    "kivi_codec_fingerprint", "kivi_payload_bytes", "kivi_export", "kivi_import",
    "kivi_check_status",
)

KIVI_PAYLOAD_MAGIC = 0x5056494B
KIVI_PAYLOAD_VERSION = 1
KIVI_PAYLOAD_HEADER_BYTES = 64

KIVI_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


class KiviError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {message} (status {status})")
        self.status = status


class kivi_cache(C.Structure):
    """Mirror of the C struct ``kivi_cache``."""
    _fields_ = [
        ("B", C.c_int32), ("H", C.c_int32), ("D", C.c_int32),
        ("bits_k", C.c_int32), ("bits_v", C.c_int32),
        ("G", C.c_int32), ("R", C.c_int32), ("Tmax", C.c_int32),
        ("kq", C.c_void_p), ("kscale", C.c_void_p), ("kzero", C.c_void_p),
        ("vq", C.c_void_p), ("vscale", C.c_void_p), ("vzero", C.c_void_p),
        ("kres", C.c_void_p), ("vres", C.c_void_p), ("len", C.c_void_p),
    ]


_LIB = None


def load(path: str | None = None):
    """Load libkivi.so (built in-tree by ``kivi_bit_kv_gb300.build``)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it with kivi_bit_kv_gb300.build.build(); "
                          "there is no fallback path")
    L = C.CDLL(p)
    vp, i32, f32, sz = C.c_void_p, C.c_int32, C.c_float, C.c_size_t
    cp = C.POINTER(kivi_cache)
    sig = {
        "kivi_abi_version": ([], i32),
        "kivi_status_string": ([i32], C.c_char_p),
        "kivi_last_error": ([], C.c_char_p),
        "kivi_cache_validate": ([cp], i32),
        "kivi_buffer_bytes": ([cp, i32], sz),
        "kivi_cache_bytes": ([i32] * 6, sz),
        "kivi_quant_keys": ([cp, vp, i32, vp, vp], i32),
        "kivi_quant_values": ([cp, vp, i32, vp, vp], i32),
        "kivi_dequant": ([cp, i32, vp, i32, vp], i32),
        "kivi_append_token": ([cp, vp, vp, vp, vp], i32),
        "kivi_decode_qk": ([cp, vp, i32, f32, vp, i32, vp], i32),
        "kivi_decode_pv": ([cp, vp, i32, i32, vp, vp, sz, vp], i32),
        "kivi_workspace_bytes": ([cp, i32], sz),
        "kivi_decode_pv_noalloc": ([cp, vp, i32, i32, vp, vp], i32),
        "kivi_decode_attention": ([cp, vp, i32, f32, vp, vp, sz, vp], i32),
        "kivi_codec_fingerprint": ([cp], C.c_uint64),
        "kivi_payload_bytes": ([cp, vp], sz),
        "kivi_export": ([cp, vp, sz, vp, vp], i32),
        "kivi_import": ([cp, vp, sz, vp, vp], i32),
        "kivi_check_status": ([C.POINTER(i32)], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _LIB = L
    return L


def _check(status: int, where: str):
    if status != KIVI_OK:
        L = load()
        msg = L.kivi_last_error().decode() or L.kivi_status_string(status).decode()
        raise KiviError(status, where, msg)


def _stream(stream, device) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, dtype, name: str, device=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, cache is on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


# ------------------------------------------------------------ host-only ---

def kivi_abi_version() -> int:
    return int(load().kivi_abi_version())


def kivi_status_string(status: int) -> str:
    return load().kivi_status_string(status).decode()


def kivi_last_error() -> str:
    return load().kivi_last_error().decode()


def kivi_cache_validate(desc: kivi_cache) -> int:
    return int(load().kivi_cache_validate(C.byref(desc)))


def kivi_buffer_bytes(desc: kivi_cache, buffer: int) -> int:
    return int(load().kivi_buffer_bytes(C.byref(desc), buffer))


def kivi_cache_bytes(T: int, D: int, bits: int, G: int, R: int, which: int) -> int:
    return int(load().kivi_cache_bytes(T, D, bits, G, R, which))


def kivi_codec_fingerprint(desc: kivi_cache) -> int:
    """FNV-1a 64 fingerprint of the codec (D, bits, G, R) of a descriptor."""
    return int(load().kivi_codec_fingerprint(C.byref(desc)))


def kivi_payload_bytes(desc: kivi_cache, lens) -> int:
    """Bytes of the compact payload when sequence b holds lens[b] tokens."""
    arr = (C.c_int32 * desc.B)(*[int(x) for x in lens])
    return int(load().kivi_payload_bytes(C.byref(desc), C.cast(arr, C.c_void_p)))


def kivi_workspace_bytes(cache, Hq: int) -> int:
    return int(load().kivi_workspace_bytes(C.byref(cache.desc), Hq))


# ---------------------------------------------------------- device calls ---

def kivi_quant_keys(cache, K: torch.Tensor, seq_lens: torch.Tensor | None = None, stream=None):
    """Prefix-encode keys K fp16 [B, H, T, D] into ``cache``."""
    B, H, T, D = K.shape
    if (B, H, D) != (cache.B, cache.H, cache.D):
        raise ValueError(f"K shape {tuple(K.shape)} does not match cache (B, H, D)="
                         f"{(cache.B, cache.H, cache.D)}")
    kp = _dev(K, torch.float16, "K", cache.device)
    lp = None if seq_lens is None else _dev(seq_lens, torch.int32, "seq_lens", cache.device)
    _check(load().kivi_quant_keys(C.byref(cache.desc), kp, T, lp, _stream(stream, cache.device)),
           "kivi_quant_keys")


def kivi_quant_values(cache, V: torch.Tensor, seq_lens: torch.Tensor | None = None, stream=None):
    """Prefix-encode values V fp16 [B, H, T, D] into ``cache``."""
    B, H, T, D = V.shape
    if (B, H, D) != (cache.B, cache.H, cache.D):
        raise ValueError(f"V shape {tuple(V.shape)} does not match cache (B, H, D)="
                         f"{(cache.B, cache.H, cache.D)}")
    vp = _dev(V, torch.float16, "V", cache.device)
    lp = None if seq_lens is None else _dev(seq_lens, torch.int32, "seq_lens", cache.device)
    _check(load().kivi_quant_values(C.byref(cache.desc), vp, T, lp, _stream(stream, cache.device)),
           "kivi_quant_values")


def kivi_dequant(cache, which: int, out: torch.Tensor, stream=None):
    """Materialize keys (which=0) or values (which=1) into out fp16 [B, H, T_out, D]."""
    B, H, T_out, D = out.shape
    if (B, H, D) != (cache.B, cache.H, cache.D):
        raise ValueError(f"out shape {tuple(out.shape)} does not match cache")
    op = _dev(out, torch.float16, "out", cache.device)
    _check(load().kivi_dequant(C.byref(cache.desc), which, op, T_out, _stream(stream, cache.device)),
           "kivi_dequant")


def kivi_append_token(cache, k: torch.Tensor, v: torch.Tensor, status: torch.Tensor, stream=None):
    """Append one token k, v fp16 [B, H, D] (or [B, H, 1, D]) to every sequence."""
    shape = (cache.B, cache.H, cache.D)
    for name, t in (("k", k), ("v", v)):
        if tuple(t.shape) not in (shape, (cache.B, cache.H, 1, cache.D)):
            raise ValueError(f"{name} shape {tuple(t.shape)}; expected {shape}")
    if status.numel() < 1:
        raise ValueError("status must hold one int32")
    _check(load().kivi_append_token(C.byref(cache.desc), _dev(k, torch.float16, "k", cache.device),
                                    _dev(v, torch.float16, "v", cache.device),
                                    _dev(status, torch.int32, "status", cache.device),
                                    _stream(stream, cache.device)), "kivi_append_token")


def kivi_decode_qk(cache, q: torch.Tensor, logits: torch.Tensor, sm_scale: float | None = None,
                   stream=None):
    """logits fp32 [B, Hq, ld] <- sm_scale * q . K_hat^T for q fp16 [B, Hq, D] (or [B, Hq, 1, D])."""
    B, Hq = q.shape[0], q.shape[1]
    if B != cache.B or q.shape[-1] != cache.D or q.numel() != B * Hq * cache.D:
        raise ValueError(f"q shape {tuple(q.shape)} does not match cache")
    if logits.dim() != 3 or tuple(logits.shape[:2]) != (B, Hq):
        raise ValueError(f"logits must be [B, Hq, ld], got {tuple(logits.shape)}")
    sm = float(cache.D ** -0.5) if sm_scale is None else float(sm_scale)
    _check(load().kivi_decode_qk(C.byref(cache.desc), _dev(q, torch.float16, "q", cache.device), Hq,
                                 sm, _dev(logits, torch.float32, "logits", cache.device),
                                 logits.shape[2], _stream(stream, cache.device)), "kivi_decode_qk")


def kivi_decode_pv(cache, logits: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, stream=None):
    """out fp32 [B, Hq, D] <- softmax(logits) . V_hat, with ws a device workspace."""
    B, Hq, ld = logits.shape
    if tuple(out.shape) not in ((B, Hq, cache.D), (B, Hq, 1, cache.D)):
        raise ValueError(f"out shape {tuple(out.shape)}; expected {(B, Hq, cache.D)}")
    wp = _dev(ws, ws.dtype, "ws", cache.device)
    _check(load().kivi_decode_pv(C.byref(cache.desc), _dev(logits, torch.float32, "logits", cache.device),
                                 ld, Hq, _dev(out, torch.float32, "out", cache.device), wp,
                                 ws.numel() * ws.element_size(), _stream(stream, cache.device)),
           "kivi_decode_pv")


def kivi_decode_pv_noalloc(cache, logits: torch.Tensor, out: torch.Tensor, stream=None):
    """kivi_decode_pv without a workspace argument, for callers that cannot
    allocate device memory: the library's fixed 16 MiB per-device scratch
    holds the partial results.  Calls sharing a device must not overlap on
    the GPU (order them on one stream); the first call on a device should
    come before any stream capture."""
    B, Hq, ld = logits.shape
    if tuple(out.shape) not in ((B, Hq, cache.D), (B, Hq, 1, cache.D)):
        raise ValueError(f"out shape {tuple(out.shape)}; expected {(B, Hq, cache.D)}")
    _check(load().kivi_decode_pv_noalloc(C.byref(cache.desc),
                                         _dev(logits, torch.float32, "logits", cache.device), ld, Hq,
                                         _dev(out, torch.float32, "out", cache.device),
                                         _stream(stream, cache.device)), "kivi_decode_pv_noalloc")


def kivi_decode_attention(cache, q: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                          sm_scale: float | None = None, stream=None):
    """out fp32 [B, Hq, D] <- softmax(sm_scale q . K_hat^T) . V_hat in one fused
    pass (logits stay on chip); q fp16 [B, Hq, D] (or [B, Hq, 1, D]), ws a
    device workspace of at least kivi_workspace_bytes(cache, Hq) bytes."""
    B, Hq = q.shape[0], q.shape[1]
    if B != cache.B or q.shape[-1] != cache.D or q.numel() != B * Hq * cache.D:
        raise ValueError(f"q shape {tuple(q.shape)} does not match cache")
    if tuple(out.shape) not in ((B, Hq, cache.D), (B, Hq, 1, cache.D)):
        raise ValueError(f"out shape {tuple(out.shape)}; expected {(B, Hq, cache.D)}")
    sm = float(cache.D ** -0.5) if sm_scale is None else float(sm_scale)
    wp = _dev(ws, ws.dtype, "ws", cache.device)
    _check(load().kivi_decode_attention(C.byref(cache.desc), _dev(q, torch.float16, "q", cache.device),
                                        Hq, sm, _dev(out, torch.float32, "out", cache.device), wp,
                                        ws.numel() * ws.element_size(), _stream(stream, cache.device)),
           "kivi_decode_attention")


def _payload_buf(t: torch.Tensor, name: str, device) -> int:
    """A uint8 payload buffer: a CUDA tensor on the cache's device or a pinned
    CPU tensor (read and written by the kernels over the CPU-GPU link)."""
    if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8:
        raise TypeError(f"{name} must be a torch.uint8 tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.is_cuda:
        if t.device != device:
            raise ValueError(f"{name} is on {t.device}, cache is on {device}")
    elif not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory (pin_memory=True)")
    return t.data_ptr()


def kivi_export(cache, dst: torch.Tensor, status: torch.Tensor, stream=None):
    """Write the cache's compact payload (include/kivi.h) into dst (uint8,
    CUDA or pinned host).  A payload larger than dst sets status[0] to
    KIVI_EWORKSPACE on the device and writes nothing."""
    _check(load().kivi_export(C.byref(cache.desc), _payload_buf(dst, "dst", cache.device), dst.numel(),
                              _dev(status, torch.int32, "status", cache.device),
                              _stream(stream, cache.device)), "kivi_export")


def kivi_import(cache, src: torch.Tensor, status: torch.Tensor, stream=None):
    """Read a compact payload from src (uint8, CUDA or pinned host) into the
    cache.  A header that does not match the cache's codec sets status[0] to
    KIVI_EINVAL on the device (KIVI_ECAPACITY for a sequence longer than
    Tmax, KIVI_EWORKSPACE for a truncated payload) and the cache is left as
    it was."""
    _check(load().kivi_import(C.byref(cache.desc), _payload_buf(src, "src", cache.device), src.numel(),
                              _dev(status, torch.int32, "status", cache.device),
                              _stream(stream, cache.device)), "kivi_import")


def kivi_check_status() -> int:
    """Status of the first failed device bounds check since the previous call
    (KIVI_ECHECK) or KIVI_OK; always KIVI_OK in a library built without
    KIVI_CHECKS.  Synchronizes the device."""
    out = C.c_int32(-1)
    _check(load().kivi_check_status(C.byref(out)), "kivi_check_status")
    return int(out.value)
