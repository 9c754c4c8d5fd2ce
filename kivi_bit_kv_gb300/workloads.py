"""Seeded synthetic inputs for the KIVI hot path (no quantization arithmetic here).

The pages run KIVI inside Llama-2-7B and Mistral-7B (CacheForge README,
"Example" and "Evaluate CacheForge on LongBench") and inside an exact-prefix
store (CacheSeek PR #4); no model weights or datasets are used here.  Instead
K, V and q are drawn from N(0, 1) in fp16 with the shapes of those models'
attention layers, and a few key channels are scaled up to mimic the
per-channel outliers that motivate quantizing keys per channel (CacheForge
README, "How it works").  Every tensor is a pure function of (shape, seed), so
the CUDA library and the CPU oracle can be fed identical bits.

Both the tests and the benchmark import this module; the oracle does not.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int              # batch (for prefix-store workloads: layers x batch)
    H: int              # KV heads
    Hq: int             # query heads
    T: int              # prefix tokens (max length when ragged)
    D: int              # head dim
    bits_k: int
    bits_v: int
    G: int
    R: int
    seed: int = 0
    outliers: tuple = ("frac", 0.04, 5.0, 20.0)   # or ("fixed", (3, 17), 10.0)
    steps: int = 0                                 # decode steps (streaming)
    ragged: tuple | None = None                    # (min_len, max_len) per sequence
    layers: int = 1                                # layers folded into B
    note: str = field(default="", compare=False)

    @property
    def Tmax(self) -> int:
        t = self.T + self.steps + 1
        return (t + self.G - 1) // self.G * self.G


WORKLOADS = {
    "tiny": Workload(
        "tiny", B=1, H=4, Hq=4, T=256, D=64, bits_k=4, bits_v=4, G=32, R=32, seed=0,
        outliers=("fixed", (3, 17), 10.0),
        note="single layer [1,4,256,64], int4, G=32, R=32: 224 quantized tokens, 7 key groups"),
    "llama2_7b_layer": Workload(
        "llama2_7b_layer", B=8, H=32, Hq=32, T=4096, D=128, bits_k=2, bits_v=2, G=32, R=128,
        seed=1, note="Llama-2-7B-shaped layer [8,32,4096,128], int2 K and V, G=32, R=128"),
    "prefix_store_int4": Workload(
        "prefix_store_int4", B=32, H=32, Hq=32, T=2065, D=128, bits_k=4, bits_v=4, G=32, R=0,
        seed=2, layers=32,
        note="32 layers x [1,32,2065,128] folded into B=32, int4, R=0, 17-token fp16 tail"),
    "prefix_store_int8": Workload(
        "prefix_store_int8", B=32, H=32, Hq=32, T=2065, D=128, bits_k=8, bits_v=8, G=32, R=0,
        seed=3, layers=32,
        note="32 layers x [1,32,2065,128] folded into B=32, int8, R=0, 17-token fp16 tail"),
    "mistral_gqa": Workload(
        "mistral_gqa", B=4, H=8, Hq=32, T=32768, D=128, bits_k=2, bits_v=2, G=32, R=128, seed=4,
        note="Mistral-7B-shaped GQA decode, K/V [4,8,32768,128], q [4,32,1,128], int2"),
    "streaming": Workload(
        "streaming", B=64, H=32, Hq=32, T=8192, D=128, bits_k=2, bits_v=2, G=32, R=128, seed=5,
        steps=256, ragged=(1024, 8192),
        note="B=64 streaming decode, lengths U[1024,8192], 256 append+decode steps, int2"),
}


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=torch.device(device)).manual_seed(int(seed))


def outlier_scales(H: int, D: int, seed: int, spec) -> torch.Tensor:
    """Per (head, channel) multipliers for the keys: fp32 [H, D] on the CPU.

    ("fixed", channels, s): those channels of every head times s.
    ("frac", f, lo, hi): round(f*D) channels per head, chosen by seed, each
    times its own U(lo, hi) factor."""
    sc = torch.ones((H, D), dtype=torch.float32)
    if spec[0] == "fixed":
        _, chans, s = spec
        sc[:, list(chans)] = float(s)
    elif spec[0] == "frac":
        _, f, lo, hi = spec
        n = max(1, int(round(f * D)))
        g = _gen(seed * 7919 + 17, "cpu")
        for h in range(H):
            idx = torch.randperm(D, generator=g)[:n]
            sc[h, idx] = lo + (hi - lo) * torch.rand(n, generator=g)
    return sc


def normal_f16(shape, seed: int, device="cpu", chunk_rows: int = 1 << 26) -> torch.Tensor:
    """fp16 N(0,1) tensor of `shape`; drawn in fp32 slabs to bound memory."""
    out = torch.empty(shape, dtype=torch.float16, device=device)
    flat = out.view(shape[0], -1)
    g = _gen(seed, device)
    per = max(1, chunk_rows // max(1, flat.shape[1]))
    for i in range(0, flat.shape[0], per):
        flat[i:i + per] = torch.randn(flat[i:i + per].shape, generator=g, device=device,
                                      dtype=torch.float32).to(torch.float16)
    return out


def make_kv(w: Workload, device="cpu", T: int | None = None, seed_offset: int = 0):
    """K, V fp16 [B, H, T, D]; keys carry the workload's outlier channels."""
    T = w.T if T is None else T
    shape = (w.B, w.H, T, w.D)
    K = normal_f16(shape, w.seed * 1000 + 11 + seed_offset, device)
    V = normal_f16(shape, w.seed * 1000 + 13 + seed_offset, device)
    sc = outlier_scales(w.H, w.D, w.seed, w.outliers).to(device)
    for b in range(w.B):  # per batch row, to keep the fp32 temporary small
        K[b] = (K[b].float() * sc[:, None, :]).to(torch.float16)
    return K, V


def make_q(w: Workload, device="cpu", step: int = 0) -> torch.Tensor:
    """Decode queries q fp16 [B, Hq, D] for decode step `step`."""
    return normal_f16((w.B, w.Hq, w.D), w.seed * 1000 + 17 + 7 * step, device)


def make_lengths(w: Workload) -> torch.Tensor:
    """Per-sequence prefix lengths int32 [B] (all T unless the workload is ragged)."""
    if w.ragged is None:
        return torch.full((w.B,), w.T, dtype=torch.int32)
    lo, hi = w.ragged
    g = _gen(w.seed * 7919 + 29, "cpu")
    return torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int32)


def make_step_tokens(w: Workload, steps: int, device="cpu"):
    """New tokens for `steps` decode steps: k, v fp16 [steps, B, H, D]."""
    k = normal_f16((steps, w.B, w.H, w.D), w.seed * 1000 + 19, device)
    v = normal_f16((steps, w.B, w.H, w.D), w.seed * 1000 + 23, device)
    sc = outlier_scales(w.H, w.D, w.seed, w.outliers).to(device)
    k = (k.float() * sc[None, None]).to(torch.float16)
    return k, v
