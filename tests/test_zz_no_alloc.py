"""kivi_decode_pv_noalloc: the decode p.V entry point for callers that cannot
allocate device memory (an engine that keeps all of HBM for its own KV pool, a
custom op that must stay inside its host runtime's memory accounting, a
decode loop that must not call cudaMalloc because it can synchronize the
device).  Its partial results live in the library's fixed 16 MiB per-device
scratch instead of a caller workspace.

Checked through the C ABI against kivi_decode_pv with a caller workspace, on
two calls in a row (the second call finds the first call's partials still in
the shared scratch), within the attention tolerance the other parity tests
use.  This file is collected last so that a run stopping at the first failure
has already run every other test."""
import ctypes as C

import numpy as np
import pytest
import torch

from _parity import ATTN_RTOL, new_cache, roundup, row_rel_err
from kivi_bit_kv_gb300 import abi

pytestmark = pytest.mark.gpu


def _filled_cache(cuda, B, H, Hq, D, T, seed):
    g = torch.Generator().manual_seed(seed)
    K = (torch.randn((B, H, T, D), generator=g) * 2).to(torch.float16).to(cuda)
    V = torch.randn((B, H, T, D), generator=g).to(torch.float16).to(cuda)
    cache = new_cache(B, H, D, 2, 2, 32, 128, roundup(T + 1, 32), cuda)
    abi.kivi_quant_keys(cache, K)
    abi.kivi_quant_values(cache, V)
    return cache, g


def test_noalloc_matches_workspace_entry_point_two_calls(cuda):
    B, H, Hq, D, T = 4, 4, 8, 128, 3000
    cache, g = _filled_cache(cuda, B, H, Hq, D, T, 31)
    assert abi.kivi_workspace_bytes(cache, Hq) <= abi.KIVI_NOALLOC_SCRATCH_BYTES
    ld = roundup(cache.Tmax, 4)
    ws = cache.workspace(Hq)
    for call in range(2):
        q = torch.randn((B, Hq, D), generator=g).to(torch.float16).to(cuda)
        logits = torch.zeros((B, Hq, ld), dtype=torch.float32, device=cuda)
        abi.kivi_decode_qk(cache, q, logits)
        want = torch.zeros((B, Hq, D), dtype=torch.float32, device=cuda)
        got = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=cuda)
        abi.kivi_decode_pv(cache, logits, want, ws)
        abi.kivi_decode_pv_noalloc(cache, logits, got)
        torch.cuda.synchronize()
        w, o = want.cpu().numpy(), got.cpu().numpy()
        assert np.isfinite(o).all(), f"call {call}"
        for b in range(B):
            for h in range(Hq):
                assert row_rel_err(o[b, h], w[b, h]) <= ATTN_RTOL, (call, b, h)


def test_noalloc_rejects_shapes_beyond_the_scratch(cuda):
    """A shape whose workspace exceeds the fixed scratch is refused with
    KIVI_EWORKSPACE and a message, before anything is launched."""
    L = abi.load()
    d = abi.kivi_cache(B=64, H=8, D=128, bits_k=2, bits_v=2, G=32, R=128, Tmax=65536)
    for i, name in enumerate(["kq", "kscale", "kzero", "vq", "vscale", "vzero", "kres", "vres", "len"]):
        setattr(d, name, 0x100000 * (i + 1))  # never dereferenced: rejected on the host
    Hq = 64
    assert L.kivi_workspace_bytes(C.byref(d), Hq) > abi.KIVI_NOALLOC_SCRATCH_BYTES
    st = L.kivi_decode_pv_noalloc(C.byref(d), 0x2000000, 65536, Hq, 0x3000000, None)
    assert st == abi.KIVI_EWORKSPACE
    assert "16 MiB" in abi.kivi_last_error()
