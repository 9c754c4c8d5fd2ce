"""Helpers for the GPU parity tests: run the CUDA path through the C ABI, run
the oracle on the same input bits, and compare with the stated tolerances.

Tolerances:
  codes, packed words, fp32 scale / zero, residual ring, lengths: bit-exact;
  materialized fp16: within 1 fp16 ulp (the arithmetic is the same fmaf +
      fp16 rounding on both sides, so equality is expected and counted);
  logits and attention output: per (b, hq) row, max|gpu - ref| / max|ref|
      <= 2e-3, the GPU accumulating in fp32 and the oracle in float64.
"""
from __future__ import annotations

import numpy as np
import torch

from kivi_bit_kv_gb300 import KiviCache, abi
from oracle import ref as R

ATTN_RTOL = 2e-3


def roundup(x, m):
    return (x + m - 1) // m * m


def np16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def new_cache(B, H, D, bk, bv, G, Rr, Tmax, device):
    return KiviCache(B, H, D, bk, bv, G, Rr, Tmax, device=device)


def gpu_encode(cache: KiviCache, K: torch.Tensor, V: torch.Tensor, seq_lens=None):
    dev = cache.device
    sl = None if seq_lens is None else torch.as_tensor(np.asarray(seq_lens, np.int32), device=dev)
    abi.kivi_quant_keys(cache, K.to(dev), sl)
    abi.kivi_quant_values(cache, V.to(dev), sl)
    torch.cuda.synchronize(dev)


def gpu_decode(cache: KiviCache, q: torch.Tensor, sm_scale=None):
    """Two-kernel decode (logits, out) and the fused kivi_decode_attention
    output."""
    B, Hq, D = q.shape
    ld = roundup(cache.Tmax, 4)
    logits = torch.zeros((B, Hq, ld), dtype=torch.float32, device=cache.device)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=cache.device)
    ws = cache.workspace(Hq)
    qd = q.to(cache.device)
    abi.kivi_decode_qk(cache, qd, logits, sm_scale)
    abi.kivi_decode_pv(cache, logits, out, ws)
    fused = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=cache.device)
    abi.kivi_decode_attention(cache, qd, fused, cache.workspace(Hq), sm_scale)
    torch.cuda.synchronize(cache.device)
    return logits.cpu().numpy(), out.cpu().numpy(), fused.cpu().numpy()


def state(cache: KiviCache, rows=None) -> dict:
    """Host copy of the cache buffers (optionally only batch rows `rows`)."""
    names = ["kq", "kscale", "kzero", "vq", "vscale", "vzero", "kres", "vres", "lens"]
    out = {}
    for n in names:
        t = getattr(cache, n)
        if rows is not None:
            t = t[torch.as_tensor(rows, device=t.device)]
        out[n] = t.cpu().numpy()
    out["kres"] = out["kres"].view(np.uint16)
    out["vres"] = out["vres"].view(np.uint16)
    return out


def compare_state(st: dict, rc: "R.RefCache"):
    """Bit-exact comparison of every byte the cache holds for rc.lens tokens."""
    assert np.array_equal(st["lens"], rc.lens), (st["lens"], rc.lens)
    Pk, Pv, G, RG = 32 // rc.bits_k, 32 // rc.bits_v, rc.G, rc.R + rc.G
    for b in range(rc.B):
        n = int(rc.lens[b])
        Tq = R.quantized_tokens(n, G, rc.R)
        for name, rows in (("kq", Tq // Pk), ("kscale", Tq // G), ("kzero", Tq // G),
                           ("vq", Tq), ("vscale", Tq), ("vzero", Tq)):
            a = st[name][b, :, :rows]
            e = getattr(rc, name)[b, :, :rows]
            if a.dtype == np.float32:
                a, e = a.view(np.uint32), e.view(np.uint32)
            if not np.array_equal(a, e):
                idx = np.argwhere(a != e)[:5]
                raise AssertionError(f"{name} differs for b={b} (len {n}, Tq {Tq}) at {idx.tolist()}: "
                                     f"gpu {a[tuple(idx[0])]} ref {e[tuple(idx[0])]}")
        slots = [t % RG for t in range(Tq, n)]
        assert np.array_equal(st["kres"][b][:, slots], rc.kres[b][:, slots]), f"kres b={b}"
        assert np.array_equal(st["vres"][b][:, slots], rc.vres[b][:, slots]), f"vres b={b}"


def ulp_diff16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in fp16 ulps between two arrays of fp16 bit patterns."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return np.abs(ordered(a) - ordered(b))


def compare_dequant(gpu_bits: np.ndarray, ref_bits: np.ndarray, lens):
    """<= 1 fp16 ulp on every materialized element; returns the exact count."""
    exact = total = 0
    for b, n in enumerate(lens):
        n = int(n)
        d = ulp_diff16(gpu_bits[b, :, :n], ref_bits[b, :, :n])
        assert d.max(initial=0) <= 1, f"b={b}: {int(d.max())} ulp"
        exact += int((d == 0).sum())
        total += d.size
    return exact, total


def row_rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    den = np.abs(ref).max()
    num = np.abs(gpu - ref).max()
    return float(num / den) if den > 0 else float(num)


def compare_attention(lg, out, ref_lg, ref_out, lens, heads=None, rtol=ATTN_RTOL, fused=None):
    """Per-row relative error of logits and outputs; rows of empty sequences
    must be exactly zero.  The fused kernel's output (which merges per-warp
    softmax partials, a different rounding order) is held to the same bound
    against the oracle.  Returns the worst (logit, output) errors."""
    worst_l = worst_o = 0.0
    B, Hq = out.shape[:2]
    for b in range(B):
        n = int(lens[b])
        for h in range(Hq) if heads is None else heads:
            if n == 0:
                assert (out[b, h] == 0).all()
                assert fused is None or (fused[b, h] == 0).all()
                continue
            el = row_rel_err(lg[b, h, :n], ref_lg[b, h, :n])
            eo = row_rel_err(out[b, h], ref_out[b, h])
            assert el <= rtol, f"logits b={b} hq={h}: rel err {el:.3g}"
            assert eo <= rtol, f"out b={b} hq={h}: rel err {eo:.3g}"
            if fused is not None:
                ef = row_rel_err(fused[b, h], ref_out[b, h])
                assert ef <= rtol, f"fused out b={b} hq={h}: rel err {ef:.3g}"
                eo = max(eo, ef)
            worst_l, worst_o = max(worst_l, el), max(worst_o, eo)
    return worst_l, worst_o
