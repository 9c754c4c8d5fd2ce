// decode.cu -- decode attention over the packed KIVI cache plus the fp16
// residual, with dequantization fused into the loads (the decode-time consumer
// of the cache: q . K_hat^T, softmax, p . V_hat).
//
// Three entry kernels share the tiles of decode_mma.cuh:
//   decode_qk_kernel         logits to global memory (kivi_decode_qk)
//   decode_pv_kernel         softmax + p . V from given logits (kivi_decode_pv)
//   decode_attention_kernel  both, logits kept in shared memory
//                            (kivi_decode_attention)
// Each CTA owns one KV head and one chunk of tokens (decode_chunk_plan),
// staged into shared memory at launch; the pv and fused kernels leave
// per-chunk (o, m, l) partials that decode_combine_kernel merges.
#include <math.h>

#include "decode_mma.cuh"
#include "kivi_launch.h"

namespace kivi {

// Per-CTA coordinates of decode chunk ci: TC tokens, or up to TC + S for the
// last chunk of a sequence (decode_chunks).  Chunks run in reverse order of
// blockIdx.y, so the last chunks of the sequences, which also carry the
// residual tokens, are dispatched first and full chunks fill the tail.
struct ChunkRange {
    int b, h, n, ci, t_begin, t_end, Tq, tq_end;
};

__device__ __forceinline__ bool chunk_range(const kivi_cache& c, int TC, int S, ChunkRange& r)
{
    const int bh = (int)blockIdx.x;
    r.b = bh / c.H;
    r.h = bh - r.b * c.H;
    r.n = c.len[r.b];
    const int nch = decode_chunks(r.n, TC, S);
    r.ci = (int)(gridDim.y - 1 - blockIdx.y);
    if (r.ci >= nch)
        return false;
    r.t_begin = r.ci * TC;
    r.t_end = r.ci == nch - 1 ? r.n : r.t_begin + TC;
    r.Tq = quantized_tokens(r.n, c.G, c.R);
    r.tq_end = max(r.t_begin, min(r.t_end, r.Tq));
    return true;
}

// Pointers into the dynamic shared memory of a decode kernel (decode_layout).
struct DecodeSmem {
    uint32_t *kw, *vw;
    float *ks, *kz, *vs, *vz, *p, *part, *zs;
    uint2* bb;
};

__device__ __forceinline__ DecodeSmem carve(float* base, const DecodeLayout& L)
{
    DecodeSmem m;
    m.kw = reinterpret_cast<uint32_t*>(base + L.kw);
    m.ks = base + L.ks;
    m.kz = base + L.kz;
    m.vw = reinterpret_cast<uint32_t*>(base + L.vw);
    m.vs = base + L.vs;
    m.vz = base + L.vz;
    m.p = base + L.p;
    m.bb = reinterpret_cast<uint2*>(base + L.bb);
    m.part = base + L.part;
    m.zs = base + L.zs;
    return m;
}


// ---------------------------------------------------------------- q . K ---

template <int BITS, int NQB>
__global__ void __launch_bounds__(kDecodeThreads, 3)
decode_qk_kernel(kivi_cache c, const uint16_t* __restrict__ q, int Hq, float sm_scale,
                 float* __restrict__ logits, int ldl, int TC, int S, const DecodeLayout L)
{
    extern __shared__ __align__(16) float dsm[];
    __shared__ __align__(16) float qs[NQB * qstride_of(256)];
    __shared__ float fac[NQB];
    using T = KeyTile<BITS, NQB>;
    ChunkRange r;
    if (!chunk_range(c, TC, S, r))
        return;
    const size_t bh = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DecodeSmem m = carve(dsm, L);
    stage_keys<BITS, T::TOK>(c, bh, r.t_begin, r.tq_end, m.kw, m.ks, m.kz);
    cp_async_commit();
    const int NQ = Hq / c.H;
    const int rows = 32 / (c.D / 32);  // residual tokens per warp step
    for (int pass = 0; pass < NQ / NQB; ++pass) {
        const int hq0 = r.h * NQ + pass * NQB;
        __syncthreads();
        stage_q<NQB>(q + ((size_t)r.b * Hq + hq0) * c.D, c.D, sm_scale, qs, fac);
        cp_async_wait_all();
        __syncthreads();
        float* out = logits + ((size_t)r.b * Hq + hq0) * ldl;
        auto sink = [&](int h, int t, float s) { out[(size_t)h * ldl + t] = s; };
        float lmax[2], rmax[NQB];  // unused here
        qk_quantized<BITS, NQB>(c.D, c.G, r.t_begin, r.tq_end, r.t_begin + warp * T::TOK, r.tq_end,
                                kDecodeWarps * T::TOK, m.kw, m.ks, m.kz, qs, fac, sink, lmax);
        qk_residual<NQB>(c, bh, r.tq_end + warp * rows, kDecodeWarps * rows, r.t_end, qs, fac, sink, rmax);
        (void)lane;
    }
}

// ---------------------------------------------------------------- p . V ---

// B fragments (with the softmax numerators) and the weighted value sum of
// one pass: p_sm holds the chunk's logits, mx their per-head maxima; then
// the chunk's partials.  Whole CTA.
template <int BITS, int NQB>
__device__ __forceinline__ void pv_pass(const kivi_cache& c, size_t bh, int TX, const ChunkRange& r,
                                        const DecodeSmem& m, const float (&mx)[NQB], size_t row0,
                                        int nchunks, float* ws_o, float* ws_m, float* ws_l, bool first_pass)
{
    const int ps = prob_stride(TX), NGv = c.D >> ilog2(c.G);
    const int n = r.t_end - r.t_begin, nq = r.tq_end - r.t_begin;
    if (first_pass) {
        cp_async_wait_all();  // the staged values
        __syncthreads();
    }
    pv_weights<NQB>(n, nq, NGv, threadIdx.x, pv_pairs(n, nq), kDecodeThreads, 0, m.p, ps, mx, m.vs, m.vz,
                    m.bb, bb_stride(TX), m.zs);
    __syncthreads();
    pv_chunk<BITS, NQB>(c, bh, TX, r.t_begin, r.tq_end, r.t_end, m.vw, m.bb, m.part);
    __syncthreads();
    write_partials<NQB>(c.D, c.G, pv_splits(pv_seg_groups<BITS>(c.D)), m.part, m.zs, mx, row0, nchunks,
                        ws_o, ws_m, ws_l);
}

template <int BITS, int NQB>
__global__ void __launch_bounds__(kDecodeThreads, 3)
decode_pv_kernel(kivi_cache c, const float* __restrict__ logits, int ldl, int Hq,
                 float* __restrict__ ws_o, float* __restrict__ ws_m, float* __restrict__ ws_l,
                 int nchunks, int TC, int S, const DecodeLayout L)
{
    extern __shared__ __align__(16) float dsm[];
    __shared__ float red[kDecodeWarps * NQB];
    ChunkRange r;
    if (!chunk_range(c, TC, S, r))
        return;
    const size_t bh = blockIdx.x;
    const DecodeSmem m = carve(dsm, L);
    stage_values<BITS>(c, bh, r.t_begin, r.tq_end, m.vw, m.vs, m.vz);
    cp_async_commit();
    const int NQ = Hq / c.H;
    const int n = r.t_end - r.t_begin;
    const int ps = prob_stride(TC + S);
    for (int pass = 0; pass < NQ / NQB; ++pass) {
        const int hq0 = r.h * NQ + pass * NQB;
        __syncthreads();
        float mx[NQB];
#pragma unroll
        for (int h = 0; h < NQB; ++h) {
            const float* lrow = logits + ((size_t)r.b * Hq + hq0 + h) * ldl + r.t_begin;
            mx[h] = -INFINITY;
            for (int t = threadIdx.x; t < n; t += kDecodeThreads) {
                const float x = lrow[t];
                m.p[h * ps + t] = x;
                mx[h] = fmaxf(mx[h], x);
            }
        }
        chunk_max<NQB>(mx, red);
        pv_pass<BITS, NQB>(c, bh, TC + S, r, m, mx, ((size_t)r.b * Hq + hq0) * nchunks + r.ci, nchunks,
                           ws_o, ws_m, ws_l, pass == 0);
    }
}

// ------------------------------------------------------------ attention ---

// One CTA per (KV head, chunk): the chunk's keys and values are staged at
// launch (two cp.async groups, keys first); q . K_hat^T runs as soon as the
// keys have landed and leaves the logits in shared memory, then the softmax,
// the B fragments and p . V_hat run as in decode_pv_kernel.  The logits never
// reach HBM.
template <int BITS, int NQB>
__global__ void __launch_bounds__(kDecodeThreads, 3)
decode_attention_kernel(kivi_cache c, const uint16_t* __restrict__ q, int Hq, float sm_scale,
                        float* __restrict__ ws_o, float* __restrict__ ws_m,
                        float* __restrict__ ws_l, int nchunks, int TC, int S, const DecodeLayout L)
{
    extern __shared__ __align__(16) float dsm[];
    __shared__ __align__(16) float qs[NQB * qstride_of(256)];
    __shared__ float fac[NQB];
    __shared__ float red[kDecodeWarps * NQB];
    using T = KeyTile<BITS, NQB>;
    ChunkRange r;
    if (!chunk_range(c, TC, S, r))
        return;
    const size_t bh = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int NQ = Hq / c.H;
    const DecodeSmem m = carve(dsm, L);
    stage_keys<BITS, T::TOK>(c, bh, r.t_begin, r.tq_end, m.kw, m.ks, m.kz);
    cp_async_commit();
    stage_values<BITS>(c, bh, r.t_begin, r.tq_end, m.vw, m.vs, m.vz);
    cp_async_commit();
    const int ps = prob_stride(TC + S);
    const int rows = 32 / (c.D / 32);  // residual tokens per warp step
    for (int pass = 0; pass < NQ / NQB; ++pass) {
        const int hq0 = r.h * NQ + pass * NQB;
        __syncthreads();
        if (pass > 0 && L.bb_on_keys) {
            // the previous pass's B fragments overwrote the staged keys
            stage_keys<BITS, T::TOK>(c, bh, r.t_begin, r.tq_end, m.kw, m.ks, m.kz);
            cp_async_commit();
        }
        stage_q<NQB>(q + ((size_t)r.b * Hq + hq0) * c.D, c.D, sm_scale, qs, fac);
        if (pass == 0)
            cp_async_wait_prior();  // the keys have landed; the values may still be in flight
        else
            cp_async_wait_all();
        __syncthreads();
        auto sink = [&](int h, int t, float s) { m.p[h * ps + t - r.t_begin] = s; };
        float lmax[2] = {-INFINITY, -INFINITY}, mx[NQB];
#pragma unroll
        for (int h = 0; h < NQB; ++h)
            mx[h] = -INFINITY;
        qk_quantized<BITS, NQB>(c.D, c.G, r.t_begin, r.tq_end, r.t_begin + warp * T::TOK, r.tq_end,
                                kDecodeWarps * T::TOK, m.kw, m.ks, m.kz, qs, fac, sink, lmax);
        qk_residual<NQB>(c, bh, r.tq_end + warp * rows, kDecodeWarps * rows, r.t_end, qs, fac, sink, mx);
#pragma unroll
        for (int slot = 0; slot < 2; ++slot) {
            const int hs = qk_slot_head<BITS, NQB>(slot);
#pragma unroll
            for (int h = 0; h < NQB; ++h)
                if (hs == h)
                    mx[h] = fmaxf(mx[h], lmax[slot]);
        }
        chunk_max<NQB>(mx, red);  // also publishes the logits
        pv_pass<BITS, NQB>(c, bh, TC + S, r, m, mx, ((size_t)r.b * Hq + hq0) * nchunks + r.ci, nchunks,
                           ws_o, ws_m, ws_l, pass == 0);
    }
}

// out[b][hq][d] = sum_c o_c[d] e^(m_c - M) / sum_c l_c e^(m_c - M), M = max m_c
// over the chunks c that hold tokens of sequence b.  One CTA per (b, hq): the
// chunk weights go to shared memory, each warp sums a quarter of the chunks
// with 16-byte loads, and the four warp sums are added in a fixed order.
constexpr int kCombineThreads = 128;

__global__ void __launch_bounds__(kCombineThreads)
decode_combine_kernel(const int32_t* __restrict__ len, int Hq, int D, int nchunks, int TC, int S,
                      const float* __restrict__ ws_o, const float* __restrict__ ws_m,
                      const float* __restrict__ ws_l, float* __restrict__ out)
{
    extern __shared__ __align__(16) float cmb[];  // e[nchunks], then [4][D] warp sums
    __shared__ float red[kDecodeWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t bhq = blockIdx.x;
    const int n = len[bhq / Hq];
    const int nv = decode_chunks(n, TC, S);
    const float* mrow = ws_m + bhq * nchunks;
    const float* lrow = ws_l + bhq * nchunks;
    float mx = -INFINITY;
    for (int k = threadIdx.x; k < nv; k += kCombineThreads)
        mx = fmaxf(mx, mrow[k]);
    for (int m = 16; m > 0; m >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    if (lane == 0)
        red[warp] = mx;
    __syncthreads();
    const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    float L = 0.0f;
    for (int k = threadIdx.x; k < nv; k += kCombineThreads) {
        const float e = expf(mrow[k] - M);
        cmb[k] = e;
        L = fmaf(lrow[k], e, L);
    }
    for (int m = 16; m > 0; m >>= 1)
        L += __shfl_xor_sync(0xffffffffu, L, m);
    if (lane == 0)
        red[warp] = L;
    __syncthreads();  // also publishes cmb[0 .. nv)
    L = (red[0] + red[1]) + (red[2] + red[3]);
    float* wsum = cmb + ((nchunks + 3) & ~3);
    const float4* o4 = reinterpret_cast<const float4*>(ws_o + bhq * nchunks * D);
    for (int d4 = lane; d4 < D / 4; d4 += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int k = warp; k < nv; k += kDecodeWarps) {
            const float4 o = o4[(size_t)k * (D / 4) + d4];
            const float e = cmb[k];
            acc.x = fmaf(o.x, e, acc.x);
            acc.y = fmaf(o.y, e, acc.y);
            acc.z = fmaf(o.z, e, acc.z);
            acc.w = fmaf(o.w, e, acc.w);
        }
        reinterpret_cast<float4*>(wsum + warp * D)[d4] = acc;
    }
    __syncthreads();
    for (int d = threadIdx.x; d < D; d += kCombineThreads) {
        const float o = (wsum[d] + wsum[D + d]) + (wsum[2 * D + d] + wsum[3 * D + d]);
        out[bhq * D + d] = nv > 0 ? o / L : 0.0f;
    }
}

// ---------------------------------------------------------------- launch ---

static ChunkPlan plan(const kivi_cache& c, int Hq)
{
    return decode_chunk_plan(c.D, c.bits_k, c.bits_v, c.G, c.R, Hq / c.H);
}
int chunk_tokens(const kivi_cache& c, int Hq) { return plan(c, Hq).TC; }
int pv_chunks(const kivi_cache& c, int Hq)
{
    const ChunkPlan cp = plan(c, Hq);
    return decode_chunks(c.Tmax, cp.TC, cp.S);
}

static cudaError_t combine(const kivi_cache& c, int Hq, const float* ws_o, const float* ws_m,
                           const float* ws_l, float* out, cudaStream_t s)
{
    const int nch = pv_chunks(c, Hq);
    const size_t smem = (((size_t)nch + 3) / 4 * 4 + (size_t)kDecodeWarps * c.D) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(decode_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    const ChunkPlan cp = plan(c, Hq);
    decode_combine_kernel<<<c.B * Hq, kCombineThreads, smem, s>>>(c.len, Hq, c.D, nch, cp.TC, cp.S,
                                                                  ws_o, ws_m, ws_l, out);
    return cudaGetLastError();
}

template <class K>
static cudaError_t set_smem(K kern, size_t bytes)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

static DecodeLayout cta_layout(const kivi_cache& c, int Hq, bool keys, bool values)
{
    const int NQ = Hq / c.H, NQB = heads_per_pass(NQ);
    const ChunkPlan cp = plan(c, Hq);
    return decode_layout(cp.TC, cp.TC + cp.S, c.D, c.bits_k, c.bits_v, c.G, NQB, NQ > NQB, keys,
                         values);
}

template <int BITS, int NQB>
static cudaError_t qk_launch(const kivi_cache& c, const uint16_t* q, int Hq, float sm,
                             float* logits, int ldl, cudaStream_t s)
{
    auto kern = decode_qk_kernel<BITS, NQB>;
    const DecodeLayout L = cta_layout(c, Hq, true, false);
    const size_t smem = 4 * L.total;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess)
        return e;
    kern<<<dim3(c.B * c.H, pv_chunks(c, Hq)), kDecodeThreads, smem, s>>>(c, q, Hq, sm, logits, ldl,
                                                                        plan(c, Hq).TC, plan(c, Hq).S, L);
    return cudaGetLastError();
}

template <int BITS>
static cudaError_t qk_bits(const kivi_cache& c, const uint16_t* q, int Hq, float sm,
                           float* logits, int ldl, cudaStream_t s)
{
    switch (heads_per_pass(Hq / c.H)) {
    case 4: return qk_launch<BITS, 4>(c, q, Hq, sm, logits, ldl, s);
    case 2: return qk_launch<BITS, 2>(c, q, Hq, sm, logits, ldl, s);
    default: return qk_launch<BITS, 1>(c, q, Hq, sm, logits, ldl, s);
    }
}

cudaError_t launch_decode_qk(const kivi_cache& c, const uint16_t* q, int Hq, float sm_scale,
                             float* logits, int ld_logits, cudaStream_t s)
{
    switch (c.bits_k) {
    case 2: return qk_bits<2>(c, q, Hq, sm_scale, logits, ld_logits, s);
    case 4: return qk_bits<4>(c, q, Hq, sm_scale, logits, ld_logits, s);
    default: return qk_bits<8>(c, q, Hq, sm_scale, logits, ld_logits, s);
    }
}

template <int BITS, int NQB>
static cudaError_t pv_launch(const kivi_cache& c, const float* logits, int ldl, int Hq,
                             float* ws_o, float* ws_m, float* ws_l, cudaStream_t s)
{
    auto kern = decode_pv_kernel<BITS, NQB>;
    const DecodeLayout L = cta_layout(c, Hq, false, true);
    const size_t smem = 4 * L.total;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess)
        return e;
    const int nch = pv_chunks(c, Hq);
    kern<<<dim3(c.B * c.H, nch), kDecodeThreads, smem, s>>>(c, logits, ldl, Hq, ws_o, ws_m, ws_l, nch,
                                                           plan(c, Hq).TC, plan(c, Hq).S, L);
    return cudaGetLastError();
}

template <int BITS>
static cudaError_t pv_bits(const kivi_cache& c, const float* logits, int ldl, int Hq, float* ws_o,
                           float* ws_m, float* ws_l, cudaStream_t s)
{
    switch (heads_per_pass(Hq / c.H)) {
    case 4: return pv_launch<BITS, 4>(c, logits, ldl, Hq, ws_o, ws_m, ws_l, s);
    case 2: return pv_launch<BITS, 2>(c, logits, ldl, Hq, ws_o, ws_m, ws_l, s);
    default: return pv_launch<BITS, 1>(c, logits, ldl, Hq, ws_o, ws_m, ws_l, s);
    }
}

cudaError_t launch_decode_pv(const kivi_cache& c, const float* logits, int ld_logits, int Hq,
                             float* out, float* ws_o, float* ws_m, float* ws_l, cudaStream_t s)
{
    cudaError_t e;
    switch (c.bits_v) {
    case 2: e = pv_bits<2>(c, logits, ld_logits, Hq, ws_o, ws_m, ws_l, s); break;
    case 4: e = pv_bits<4>(c, logits, ld_logits, Hq, ws_o, ws_m, ws_l, s); break;
    default: e = pv_bits<8>(c, logits, ld_logits, Hq, ws_o, ws_m, ws_l, s); break;
    }
    if (e != cudaSuccess)
        return e;
    return combine(c, Hq, ws_o, ws_m, ws_l, out, s);
}

template <int BITS, int NQB>
static cudaError_t attn_launch(const kivi_cache& c, const uint16_t* q, int Hq, float sm,
                               float* ws_o, float* ws_m, float* ws_l, cudaStream_t s)
{
    auto kern = decode_attention_kernel<BITS, NQB>;
    const DecodeLayout L = cta_layout(c, Hq, true, true);
    const size_t smem = 4 * L.total;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess)
        return e;
    const int nch = pv_chunks(c, Hq);
    kern<<<dim3(c.B * c.H, nch), kDecodeThreads, smem, s>>>(c, q, Hq, sm, ws_o, ws_m, ws_l, nch,
                                                           plan(c, Hq).TC, plan(c, Hq).S, L);
    return cudaGetLastError();
}

template <int BITS>
static cudaError_t attn_bits(const kivi_cache& c, const uint16_t* q, int Hq, float sm,
                             float* ws_o, float* ws_m, float* ws_l, cudaStream_t s)
{
    switch (heads_per_pass(Hq / c.H)) {
    case 4: return attn_launch<BITS, 4>(c, q, Hq, sm, ws_o, ws_m, ws_l, s);
    case 2: return attn_launch<BITS, 2>(c, q, Hq, sm, ws_o, ws_m, ws_l, s);
    default: return attn_launch<BITS, 1>(c, q, Hq, sm, ws_o, ws_m, ws_l, s);
    }
}

cudaError_t launch_decode_attention(const kivi_cache& c, const uint16_t* q, int Hq, float sm_scale,
                                    float* out, float* ws_o, float* ws_m, float* ws_l,
                                    cudaStream_t s)
{
    cudaError_t e;
    switch (c.bits_k) {  // the fused kernel needs bits_k == bits_v (checked by the caller)
    case 2: e = attn_bits<2>(c, q, Hq, sm_scale, ws_o, ws_m, ws_l, s); break;
    case 4: e = attn_bits<4>(c, q, Hq, sm_scale, ws_o, ws_m, ws_l, s); break;
    default: e = attn_bits<8>(c, q, Hq, sm_scale, ws_o, ws_m, ws_l, s); break;
    }
    if (e != cudaSuccess)
        return e;
    return combine(c, Hq, ws_o, ws_m, ws_l, out, s);
}

}  // namespace kivi
