"""GPU parity: libkivi's CUDA kernels, called through the C ABI, against the
CPU oracle on identical seeded inputs.

Small shapes span several tiles, decode chunks and ragged tails and cover the
edge cases (empty sequences, T < R, T == R, T == R+G-1, T == R+G, tails that
do not fill a group, every bit width and group size, mixed key/value widths,
grouped-query ratios 1..8, capacity overflow).  The named workloads run at
full size in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

from _parity import (compare_attention, compare_dequant, compare_state, gpu_decode, gpu_encode,
                     new_cache, np16, roundup, state)
from kivi_bit_kv_gb300 import abi
from kivi_bit_kv_gb300 import workloads as W
from oracle import ref as R

pytestmark = pytest.mark.gpu

THREADS = R.host_threads()


def f16_host(shape, seed, scale=1.0, outlier_every=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g)
    if outlier_every:
        mult = torch.ones(shape[-1])
        mult[::outlier_every] = 12.0
        x = x * mult
    return (x * scale).to(torch.float16)


# name, B, H, Hq, D, bits_k, bits_v, G, R, T, seq_lens
SMALL = [
    ("d64_int4", 1, 4, 4, 64, 4, 4, 32, 32, 256, None),
    ("d128_int2", 2, 2, 2, 128, 2, 2, 32, 128, 1500, None),
    ("d128_int8_tail", 2, 2, 2, 128, 8, 8, 32, 0, 1100, None),
    ("d256_int4_G64", 1, 2, 4, 256, 4, 4, 64, 64, 700, None),
    ("k2v4_gqa4", 2, 2, 8, 128, 2, 4, 32, 32, 1300, None),
    ("k8v2_G128_gqa3", 1, 2, 6, 128, 8, 2, 128, 128, 2100, None),
    ("d64_G64_gqa8", 1, 1, 8, 64, 2, 2, 64, 0, 900, None),
    ("d256_int2_gqa2", 1, 2, 4, 256, 2, 2, 32, 32, 600, None),
    ("ragged", 4, 2, 4, 128, 2, 2, 32, 128, 1200, [0, 1, 159, 1200]),
    ("T_lt_R", 1, 2, 2, 128, 2, 2, 32, 128, 100, None),
    ("T_eq_R", 1, 2, 2, 128, 4, 4, 32, 128, 128, None),
    ("T_eq_R_G_1", 1, 2, 2, 128, 4, 4, 32, 128, 159, None),
    ("T_eq_R_G", 1, 2, 2, 128, 4, 4, 32, 128, 160, None),
    ("T1", 1, 1, 1, 64, 2, 2, 32, 0, 1, None),
    ("multi_chunk", 1, 1, 2, 128, 2, 2, 32, 128, 5000, None),
    ("int8_gqa4_multi", 1, 2, 8, 128, 8, 8, 32, 64, 3000, None),
    # the largest grouped-query ratio, 16 query heads per KV head: four passes
    ("gqa16_4pass", 1, 2, 32, 128, 2, 2, 32, 128, 1200, None),
    # a sequence's last chunk absorbs a tail of up to min(R, TC/4) tokens
    ("slack_tail", 4, 1, 1, 128, 2, 2, 32, 128, 1160, [1025, 1152, 1153, 640]),
    ("slack_R32", 4, 1, 2, 128, 4, 4, 32, 32, 1100, [512, 543, 544, 1056]),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_encode_dequant_decode_small(cuda, case):
    name, B, H, Hq, D, bk, bv, G, Rr, T, sl = case
    Tmax = roundup(T + 40, G)
    K = f16_host((B, H, T, D), 1 + T, 2.0, outlier_every=13)
    V = f16_host((B, H, T, D), 2 + T)
    q = f16_host((B, Hq, D), 3 + T)
    cache = new_cache(B, H, D, bk, bv, G, Rr, Tmax, cuda)
    gpu_encode(cache, K, V, sl)
    rc = R.RefCache(B, H, D, bk, bv, G, Rr, Tmax).encode(np16(K), np16(V), seq_lens=sl)
    compare_state(state(cache), rc)

    lens = rc.lens
    for which in (0, 1):
        out = torch.zeros((B, H, T, D), dtype=torch.float16, device=cuda)
        abi.kivi_dequant(cache, which, out)
        torch.cuda.synchronize()
        ex, tot = compare_dequant(np16(out).view(np.uint16), rc.decode(which, T_out=T), lens)
        assert ex == tot  # same fmaf + fp16 rounding on both sides

    lg, o, fo = gpu_decode(cache, q)
    rlg, ro = rc.attention(np16(q))
    compare_attention(lg, o, rlg, ro, lens, fused=fo)


def test_decode_many_chunks(cuda):
    """A capacity of 2^24 tokens in 256-token chunks: 65536 chunk partials per
    row, more weights than the combine kernel keeps in shared memory, so it
    recomputes them where it uses them.  Results as for any other shape."""
    B, H, Hq, D, bits, G, Rr, T = 1, 1, 2, 64, 8, 32, 0, 3000
    K = f16_host((B, H, T, D), 21, 2.0)
    V = f16_host((B, H, T, D), 22)
    q = f16_host((B, Hq, D), 23)
    cache = new_cache(B, H, D, bits, bits, G, Rr, 1 << 24, cuda)
    gpu_encode(cache, K, V)
    rc = R.RefCache(B, H, D, bits, bits, G, Rr, roundup(T, G)).encode(np16(K), np16(V))
    lg, o, fo = gpu_decode(cache, q)
    rlg, ro = rc.attention(np16(q))
    compare_attention(lg[:, :, :T], o, rlg, ro, rc.lens, fused=fo)
    del cache
    torch.cuda.empty_cache()


def test_more_slices_than_a_grid_dimension(cuda):
    """66000 (b, h) slices, more than one grid dimension holds (65535): the
    encode and materialize kernels loop over slices, decode runs on a 1-D
    grid.  Sampled batch rows are compared with the oracle run on those rows
    alone (slices are independent)."""
    B, H, Hq, D, bits, G, Rr, T = 33000, 2, 4, 64, 4, 32, 0, 70
    Tmax = roundup(T + 8, G)
    K = f16_host((B, H, T, D), 31, 2.0)
    V = f16_host((B, H, T, D), 32)
    q = f16_host((B, Hq, D), 33)
    cache = new_cache(B, H, D, bits, bits, G, Rr, Tmax, cuda)
    gpu_encode(cache, K, V)
    rows = [0, 1, 16383, 32767, 32768, B - 1]
    rc = R.RefCache(len(rows), H, D, bits, bits, G, Rr, Tmax).encode(np16(K[rows]), np16(V[rows]))
    compare_state(state(cache, rows), rc)
    out = torch.zeros((B, H, T, D), dtype=torch.float16, device=cuda)
    abi.kivi_dequant(cache, 1, out)
    torch.cuda.synchronize()
    ex, tot = compare_dequant(np16(out[rows]).view(np.uint16), rc.decode(1, T_out=T), rc.lens)
    assert ex == tot
    lg, o, fo = gpu_decode(cache, q)
    rlg, ro = rc.attention(np16(q[rows]))
    compare_attention(lg[rows][:, :, :T], o[rows], rlg, ro, rc.lens, fused=fo[rows])
    # compact payload round trip on the device: every slice's offset
    n = abi.kivi_payload_bytes(cache.desc, cache.lens.cpu().tolist())
    buf = torch.empty(n, dtype=torch.uint8, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    abi.kivi_export(cache, buf, status)
    fresh = new_cache(B, H, D, bits, bits, G, Rr, Tmax, cuda)
    abi.kivi_import(fresh, buf, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Tq = R.quantized_tokens(T, G, Rr)
    for name, used in (("kq", Tq * bits // 32), ("kscale", Tq // G), ("kzero", Tq // G), ("vq", Tq),
                       ("vscale", Tq), ("vzero", Tq)):
        assert torch.equal(getattr(fresh, name)[:, :, :used], getattr(cache, name)[:, :, :used]), name
    assert torch.equal(fresh.lens, cache.lens)
    compare_state(state(fresh, rows), rc)
    del cache, out, fresh, buf
    torch.cuda.empty_cache()


def test_fused_decode_many_ragged_sequences(cuda):
    """More sequences than the fused decode's CTA has threads (1000 > 384),
    ragged from 0 to 300 tokens with empty ones among them: the tile split
    then scans the lengths in several passes carrying running totals, many
    ranges hold several short rows and some rows are cut between CTAs.  Every
    row is compared with the oracle (empty sequences must give zeros)."""
    B, H, Hq, D, bk, bv, G, Rr = 1000, 1, 2, 64, 2, 4, 32, 32
    g = np.random.default_rng(41)
    lens = g.integers(0, 301, size=B)
    lens[g.choice(B, 40, replace=False)] = 0
    T = int(lens.max())
    Tmax = roundup(T + 8, G)
    K = f16_host((B, H, T, D), 42, 2.0)
    V = f16_host((B, H, T, D), 43)
    q = f16_host((B, Hq, D), 44)
    cache = new_cache(B, H, D, bk, bv, G, Rr, Tmax, cuda)
    gpu_encode(cache, K, V, lens.tolist())
    rc = R.RefCache(B, H, D, bk, bv, G, Rr, Tmax).encode(np16(K), np16(V), seq_lens=lens.tolist())
    lg, o, fo = gpu_decode(cache, q)
    rlg, ro = rc.attention(np16(q))
    compare_attention(lg[:, :, :T], o, rlg, ro, rc.lens, fused=fo)
    del cache
    torch.cuda.empty_cache()


def test_decode_is_deterministic(cuda):
    B, H, Hq, D, T = 2, 2, 4, 128, 3000
    K, V = f16_host((B, H, T, D), 5, 2.0), f16_host((B, H, T, D), 6)
    q = f16_host((B, Hq, D), 7)
    cache = new_cache(B, H, D, 2, 2, 32, 128, roundup(T, 32), cuda)
    gpu_encode(cache, K, V)
    a = gpu_decode(cache, q)
    b = gpu_decode(cache, q)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("bk,bv,G,Rr,T0,n", [(2, 2, 32, 128, 100, 300), (4, 8, 32, 0, 17, 150),
                                            (8, 4, 64, 64, 0, 260), (2, 4, 128, 128, 250, 140)])
def test_append_stream_small(cuda, bk, bv, G, Rr, T0, n):
    """Append n tokens one at a time (flushes at different steps for
    different sequences) and compare cache state and decode output."""
    B, H, Hq, D = 3, 2, 4, 128
    lens0 = [T0, max(0, T0 - 37), T0 + 45]
    Tmax = roundup(max(lens0) + n + 1, G)
    Tpad = max(lens0)
    K = f16_host((B, H, Tpad, D), 11, 2.0, outlier_every=9)
    V = f16_host((B, H, Tpad, D), 12)
    kn = f16_host((n, B, H, D), 13, 2.0)
    vn = f16_host((n, B, H, D), 14)
    cache = new_cache(B, H, D, bk, bv, G, Rr, Tmax, cuda)
    gpu_encode(cache, K, V, lens0)
    rc = R.RefCache(B, H, D, bk, bv, G, Rr, Tmax).encode(np16(K), np16(V), seq_lens=lens0)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    knd, vnd = kn.to(cuda), vn.to(cuda)
    check_at = {0, 1, n // 3, n - 1}
    for s in range(n):
        abi.kivi_append_token(cache, knd[s], vnd[s], status)
        rc.append(np16(kn[s]), np16(vn[s]))
        if s in check_at:
            q = f16_host((B, Hq, D), 100 + s)
            lg, o, fo = gpu_decode(cache, q)
            rlg, ro = rc.attention(np16(q))
            compare_attention(lg, o, rlg, ro, rc.lens, fused=fo)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare_state(state(cache), rc)


def test_append_capacity_status(cuda):
    """A full sequence is left unchanged and flagged; the others advance."""
    B, H, D, G = 2, 2, 64, 32
    cache = new_cache(B, H, D, 4, 4, G, 0, 64, cuda)
    K = f16_host((B, H, 64, D), 21)
    gpu_encode(cache, K, K, [64, 10])
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    k = f16_host((B, H, D), 22).to(cuda)
    abi.kivi_append_token(cache, k, k, status)
    torch.cuda.synchronize()
    assert int(status.item()) == abi.KIVI_ECAPACITY
    assert cache.lens.cpu().tolist() == [64, 11]


def test_binding_rejects_bad_tensors(cuda):
    cache = new_cache(1, 2, 64, 2, 2, 32, 32, 256, cuda)
    with pytest.raises(TypeError):
        abi.kivi_quant_keys(cache, torch.zeros((1, 2, 64, 64), dtype=torch.float32, device=cuda))
    with pytest.raises(ValueError):
        abi.kivi_quant_keys(cache, torch.zeros((1, 2, 64, 64), dtype=torch.float16))
    with pytest.raises(abi.KiviError) as e:
        abi.kivi_quant_keys(cache, torch.zeros((1, 2, 300, 64), dtype=torch.float16, device=cuda))
    assert e.value.status == abi.KIVI_EINVAL


# ------------------------------------------------------- named workloads --

def _workload_encode(w, cuda, rows=None):
    """Encode workload w on the GPU; oracle-encode batch rows `rows`."""
    K, V = W.make_kv(w, device=cuda)
    lens = W.make_lengths(w)
    Tmax = roundup(w.T + w.steps + 1, w.G)
    cache = new_cache(w.B, w.H, w.D, w.bits_k, w.bits_v, w.G, w.R, Tmax, cuda)
    gpu_encode(cache, K, V, None if w.ragged is None else lens.tolist())
    rows = list(range(w.B)) if rows is None else rows
    Kh = np16(K[rows]).view(np.uint16)
    Vh = np16(V[rows]).view(np.uint16)
    rc = R.RefCache(len(rows), w.H, w.D, w.bits_k, w.bits_v, w.G, w.R, Tmax)
    rc.encode(Kh, Vh, seq_lens=lens[rows].numpy(), threads=THREADS)
    return cache, rc, K, V, rows


def test_workload_tiny(cuda):
    w = W.WORKLOADS["tiny"]
    cache, rc, K, V, rows = _workload_encode(w, cuda)
    assert R.quantized_tokens(w.T, w.G, w.R) == 224
    compare_state(state(cache), rc)
    for which in (0, 1):
        out = torch.zeros((w.B, w.H, w.T, w.D), dtype=torch.float16, device=cuda)
        abi.kivi_dequant(cache, which, out)
        ex, tot = compare_dequant(np16(out).view(np.uint16), rc.decode(which), rc.lens)
        assert ex == tot
    q = W.make_q(w, cuda)
    lg, o, fo = gpu_decode(cache, q)
    rlg, ro = rc.attention(np16(q))
    compare_attention(lg, o, rlg, ro, rc.lens, fused=fo)


@pytest.mark.slow
def test_workload_llama2_layer_full(cuda):
    """[8,32,4096,128] int2: every code, stat and residual byte, every
    materialized element and every decode row against the oracle."""
    w = W.WORKLOADS["llama2_7b_layer"]
    cache, rc, K, V, rows = _workload_encode(w, cuda)
    compare_state(state(cache), rc)
    for which in (0, 1):
        out = torch.empty((w.B, w.H, w.T, w.D), dtype=torch.float16, device=cuda)
        abi.kivi_dequant(cache, which, out)
        ex, tot = compare_dequant(np16(out).view(np.uint16), rc.decode(which, threads=THREADS), rc.lens)
        assert ex == tot
    q = W.make_q(w, cuda)
    lg, o, fo = gpu_decode(cache, q)
    rlg, ro = rc.attention(np16(q), threads=THREADS)
    compare_attention(lg, o, rlg, ro, rc.lens, fused=fo)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefix_store_int4", "prefix_store_int8"])
def test_workload_prefix_store(cuda, name):
    """32 layers x [1,32,2065,128] (layers folded into the batch axis), R=0:
    encode the whole prefix, materialize it back; sampled layers compared
    completely (2048 quantized tokens + a 17-token fp16 tail each)."""
    w = W.WORKLOADS[name]
    rows = [0, 7, 19, 31]
    cache, rc, K, V, rows = _workload_encode(w, cuda, rows)
    assert R.quantized_tokens(w.T, w.G, w.R) == 2048
    compare_state(state(cache, rows), rc)
    for which in (0, 1):
        out = torch.empty((w.B, w.H, w.T, w.D), dtype=torch.float16, device=cuda)
        abi.kivi_dequant(cache, which, out)
        got = np16(out[rows]).view(np.uint16)
        ex, tot = compare_dequant(got, rc.decode(which, threads=THREADS), rc.lens)
        assert ex == tot
        # the fp16 tail comes back verbatim
        src = K if which == 0 else V
        assert torch.equal(out[:, :, 2048:], src[:, :, 2048:])


@pytest.mark.slow
def test_workload_mistral_gqa(cuda):
    """K/V [4,8,32768,128], q [4,32,1,128]: every row of the GQA decode."""
    w = W.WORKLOADS["mistral_gqa"]
    cache, rc, K, V, rows = _workload_encode(w, cuda)
    compare_state(state(cache), rc)
    q = W.make_q(w, cuda)
    lg, o, fo = gpu_decode(cache, q)
    rlg, ro = rc.attention(np16(q), threads=THREADS)
    compare_attention(lg, o, rlg, ro, rc.lens, fused=fo)


@pytest.mark.slow
def test_workload_streaming(cuda):
    """B=64 ragged lengths U[1024,8192], 256 append+decode steps on all 64
    sequences; 6 sampled sequences are followed by the oracle step by step."""
    w = W.WORKLOADS["streaming"]
    rows = [0, 9, 22, 37, 50, 63]
    cache, rc, K, V, rows = _workload_encode(w, cuda, rows)
    del K, V
    compare_state(state(cache, rows), rc)
    kn, vn = W.make_step_tokens(w, w.steps, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    check = {0, 1, 31, 32, 100, 200, 255}
    ld = roundup(cache.Tmax, 4)
    logits = torch.zeros((w.B, w.Hq, ld), dtype=torch.float32, device=cuda)
    out = torch.zeros((w.B, w.Hq, w.D), dtype=torch.float32, device=cuda)
    ws = cache.workspace(w.Hq)
    fused = torch.zeros((w.B, w.Hq, w.D), dtype=torch.float32, device=cuda)
    ws2 = cache.workspace(w.Hq)
    for s in range(w.steps):
        abi.kivi_append_token(cache, kn[s], vn[s], status)
        rc.append(np16(kn[s][rows]), np16(vn[s][rows]))
        q = W.make_q(w, cuda, step=s)
        abi.kivi_decode_qk(cache, q, logits)
        abi.kivi_decode_pv(cache, logits, out, ws)
        abi.kivi_decode_attention(cache, q, fused, ws2)
        if s in check:
            torch.cuda.synchronize()
            rlg, ro = rc.attention(np16(q[rows]), threads=THREADS)
            compare_attention(logits[rows].cpu().numpy(), out[rows].cpu().numpy(), rlg, ro, rc.lens,
                              fused=fused[rows].cpu().numpy())
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare_state(state(cache, rows), rc)
