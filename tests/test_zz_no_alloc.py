"""kivi_decode_pv_noalloc: the decode p.V entry point for callers that cannot
allocate device memory (an engine that keeps all of HBM for its own KV pool, a
custom op that must stay inside its host runtime's memory accounting, a
decode loop that must not call cudaMalloc because it can synchronize the
device).  Its partial results live in the library's fixed 16 MiB per-device
scratch instead of a caller workspace.

Checked through the C ABI against kivi_decode_pv with a fresh, NaN-filled
caller workspace: the same kernels run on the same inputs, so the outputs
must be bit-identical.  Two calls in a row share the scratch: the first one
on long sequences, the second on a cache whose sequences are much shorter, so
the scratch still holds partials of chunks the second call does not have,
and the result must not depend on them.  Device memory in use must not change
from call to call.  This file is collected last so that a run stopping at the
first failure has already run every other test."""
import ctypes as C

import numpy as np
import pytest
import torch

from _parity import new_cache, roundup
from kivi_bit_kv_gb300 import abi

pytestmark = pytest.mark.gpu

B, H, HQ, D, T = 4, 4, 8, 128, 3000


def _filled_cache(cuda, seed, seq_lens=None):
    g = torch.Generator().manual_seed(seed)
    K = (torch.randn((B, H, T, D), generator=g) * 2).to(torch.float16).to(cuda)
    V = torch.randn((B, H, T, D), generator=g).to(torch.float16).to(cuda)
    cache = new_cache(B, H, D, 2, 2, 32, 128, roundup(T + 1, 32), cuda)
    sl = None if seq_lens is None else torch.tensor(seq_lens, dtype=torch.int32, device=cuda)
    abi.kivi_quant_keys(cache, K, sl)
    abi.kivi_quant_values(cache, V, sl)
    q = torch.randn((B, HQ, D), generator=g).to(torch.float16).to(cuda)
    logits = torch.zeros((B, HQ, roundup(cache.Tmax, 4)), dtype=torch.float32, device=cuda)
    abi.kivi_decode_qk(cache, q, logits)
    return cache, logits


def _reference(cache, logits, cuda):
    """kivi_decode_pv with a fresh caller workspace filled with NaN."""
    ws = cache.workspace(HQ)  # fp32
    ws.fill_(float("nan"))
    want = torch.full((B, HQ, D), float("nan"), dtype=torch.float32, device=cuda)
    abi.kivi_decode_pv(cache, logits, want, ws)
    return want


def test_noalloc_matches_workspace_entry_point_two_calls(cuda):
    long_cache, long_logits = _filled_cache(cuda, 31)
    short_cache, short_logits = _filled_cache(cuda, 32, seq_lens=[700, 64, 1500, 0])
    for cache in (long_cache, short_cache):
        assert abi.kivi_workspace_bytes(cache, HQ) <= abi.KIVI_NOALLOC_SCRATCH_BYTES
    want_long = _reference(long_cache, long_logits, cuda)
    want_short = _reference(short_cache, short_logits, cuda)
    got = [torch.full((B, HQ, D), float("nan"), dtype=torch.float32, device=cuda) for _ in range(3)]
    torch.cuda.synchronize()

    abi.kivi_decode_pv_noalloc(long_cache, long_logits, got[0])
    torch.cuda.synchronize()
    # after the first call (which may load the library's scratch module)
    free_after_first = torch.cuda.mem_get_info()[0]
    torch_after_first = torch.cuda.memory_allocated()
    abi.kivi_decode_pv_noalloc(short_cache, short_logits, got[1])
    abi.kivi_decode_pv_noalloc(long_cache, long_logits, got[2])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_after_first, "device memory changed across calls"
    assert torch.cuda.memory_allocated() == torch_after_first

    for i, want in ((0, want_long), (1, want_short), (2, want_long)):
        o, w = got[i].cpu().numpy(), want.cpu().numpy()
        assert np.isfinite(o).all(), f"call {i}"
        assert np.array_equal(o.view(np.uint32), w.view(np.uint32)), f"call {i} differs from kivi_decode_pv"
    # the empty sequence of the short cache gets zeros
    assert (got[1][3] == 0).all()


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
    # a bad Hq on the same large cache is an argument error, not a size error
    st = L.kivi_decode_pv_noalloc(C.byref(d), 0x2000000, 65536, 12, 0x3000000, None)
    assert st == abi.KIVI_EINVAL
    assert "Hq=12" in abi.kivi_last_error()
