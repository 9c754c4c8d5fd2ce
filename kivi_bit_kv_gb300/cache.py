"""Device cache allocation for libkivi: torch owns the memory, the C library
gets a ``kivi_cache`` descriptor of raw device pointers.

Layouts (P = 32 / bits; see include/kivi.h):
    kq      int32 [B, H, Tmax/Pk, D]     kscale, kzero  fp32 [B, H, Tmax/G, D]
    vq      int32 [B, H, Tmax, D/Pv]     vscale, vzero  fp32 [B, H, Tmax, D/G]
    kres, vres  fp16 [B, H, R+G, D]      lens  int32 [B]
"""
from __future__ import annotations

import torch

from . import abi


class KiviCache:
    """A KIVI KV cache for one attention layer, resident on one GPU."""

    def __init__(self, B: int, H: int, D: int, bits_k: int, bits_v: int, G: int, R: int,
                 Tmax: int, device="cuda"):
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.B, self.H, self.D = B, H, D
        self.bits_k, self.bits_v, self.G, self.R, self.Tmax = bits_k, bits_v, G, R, Tmax
        desc = abi.kivi_cache(B=B, H=H, D=D, bits_k=bits_k, bits_v=bits_v, G=G, R=R, Tmax=Tmax)
        # sizes come from the library, so a bad configuration fails here
        nbytes = [abi.kivi_buffer_bytes(desc, i) for i in range(9)]
        if min(nbytes) == 0:
            st = abi.kivi_cache_validate(desc)
            raise abi.KiviError(st, "KiviCache", abi.kivi_last_error())
        Pk, Pv, RG = 32 // bits_k, 32 // bits_v, R + G
        kw = dict(device=self.device)
        self.kq = torch.zeros((B, H, Tmax // Pk, D), dtype=torch.int32, **kw)
        self.kscale = torch.zeros((B, H, Tmax // G, D), dtype=torch.float32, **kw)
        self.kzero = torch.zeros_like(self.kscale)
        self.vq = torch.zeros((B, H, Tmax, D // Pv), dtype=torch.int32, **kw)
        self.vscale = torch.zeros((B, H, Tmax, D // G), dtype=torch.float32, **kw)
        self.vzero = torch.zeros_like(self.vscale)
        self.kres = torch.zeros((B, H, RG, D), dtype=torch.float16, **kw)
        self.vres = torch.zeros_like(self.kres)
        self.lens = torch.zeros((B,), dtype=torch.int32, **kw)
        bufs = [self.kq, self.kscale, self.kzero, self.vq, self.vscale, self.vzero,
                self.kres, self.vres, self.lens]
        for t, nb in zip(bufs, nbytes):
            assert t.numel() * t.element_size() == nb, (t.shape, nb)
        desc.kq, desc.kscale, desc.kzero = (t.data_ptr() for t in bufs[0:3])
        desc.vq, desc.vscale, desc.vzero = (t.data_ptr() for t in bufs[3:6])
        desc.kres, desc.vres, desc.len = (t.data_ptr() for t in bufs[6:9])
        self.desc = desc

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in
                   (self.kq, self.kscale, self.kzero, self.vq, self.vscale, self.vzero,
                    self.kres, self.vres, self.lens))

    def workspace(self, Hq: int) -> torch.Tensor:
        """A decode workspace large enough for ``kivi_decode_pv`` with Hq query heads."""
        n = abi.kivi_workspace_bytes(self, Hq)
        return torch.empty((max(n, 16) + 15) // 16 * 4, dtype=torch.float32, device=self.device)
