// decode_kernels.cuh -- the decode-attention kernels over the packed KIVI
// cache plus the fp16 residual, with dequantization fused into the loads (the
// decode-time consumer of the cache: q . K_hat^T, softmax, p . V_hat), and
// their launchers for one head dimension D (a template parameter, so every
// tile's index arithmetic is resolved at compile time).  decode_d64.cu,
// decode_d128.cu and decode_d256.cu instantiate them; decode.cu dispatches.
//
// Two entry kernels share the tiles of decode_mma.cuh:
//   decode_qk_kernel         logits to global memory (kivi_decode_qk)
//   decode_pv_kernel         softmax + p . V from given logits (kivi_decode_pv)
// Each CTA owns one KV head and one chunk of tokens (decode_chunk_plan),
// staged into shared memory at launch; the pv kernel leaves per-chunk
// (o, m, l) partials that decode_combine_kernel (decode.cu) merges.  The fused
// kivi_decode_attention runs the streamed kernel of decode_stream.cuh.
#pragma once

#include <math.h>

#include "decode_mma.cuh"
#include "kivi_launch.h"

namespace kivi {

// Per-CTA coordinates of decode chunk ci of slice bh: TC tokens, or up to
// TC + S for the last chunk of a sequence (decode_chunks).  The 1-D grid holds
// B H nchunks CTAs, slice fastest; chunks run in reverse order, so the last
// chunks of the sequences, which also carry the residual tokens, are
// dispatched first and full chunks fill the tail.
struct ChunkRange {
    int bh, b, h, n, ci, t_begin, t_end, Tq, tq_end;
};

__device__ __forceinline__ bool chunk_range(const kivi_cache& c, int TC, int S, ChunkRange& r)
{
    const int BH = c.B * c.H;
    const int y = (int)(blockIdx.x / BH);
    const int bh = (int)blockIdx.x - y * BH;
    r.bh = bh;
    r.b = bh / c.H;
    r.h = bh - r.b * c.H;
    r.n = ld_checked(c.len + r.b);
    const int nch = decode_chunks(r.n, TC, S);
    r.ci = (int)(gridDim.x / BH) - 1 - y;
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
    bool zs_on_p;  // the zero terms overlay the logits
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
    m.zs_on_p = L.zs_on_p;
    return m;
}


// ---------------------------------------------------------------- q . K ---

template <int BITS, int NQB, int D>
__global__ void __launch_bounds__(kDecodeThreads, 3)
decode_qk_kernel(kivi_cache c, const uint16_t* __restrict__ q, int Hq, float sm_scale,
                 float* __restrict__ logits, int ldl, int TC, int S, const DecodeLayout L)
{
    extern __shared__ __align__(16) float dsm[];
    __shared__ __align__(16) float qs[NQB * qstride_of(D)];
    __shared__ float fac[NQB];
    __shared__ float red[kDecodeWarps];
    using T = KeyTile<BITS, NQB>;
    ChunkRange r;
    if (!chunk_range(c, TC, S, r))
        return;
    const size_t bh = r.bh;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DecodeSmem m = carve(dsm, L);
    stage_keys<BITS, T::TOK, D>(c, bh, r.t_begin, r.tq_end, m.kw, m.ks, m.kz);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    const float fk = weight_scale_pow2(cta_max_stat(m.ks, ((r.tq_end - r.t_begin) / c.G) * D, red));
    const int NQ = Hq / c.H;
    constexpr int rows = 32 / (D / 32);  // residual tokens per warp step
    for (int pass = 0; pass < NQ / NQB; ++pass) {
        const int hq0 = r.h * NQ + pass * NQB;
        __syncthreads();
        stage_q<NQB, D>(q + ((size_t)r.b * Hq + hq0) * D, sm_scale, fk, qs, fac);
        __syncthreads();
        float* out = logits + ((size_t)r.b * Hq + hq0) * ldl;
        auto sink = [&](int h, int t, float s) { st_checked(out + (size_t)h * ldl + t, s); };
        float lmax[2], rmax[NQB];  // unused here
        qk_quantized<BITS, NQB, D>(c.G, r.t_begin, r.tq_end, r.t_begin + warp * T::TOK, r.tq_end,
                                kDecodeWarps * T::TOK, m.kw, m.ks, m.kz, qs, fac, sink, lmax);
        qk_residual<NQB, D>(c, bh, r.tq_end + warp * rows, kDecodeWarps * rows, r.t_end, qs, fac, sink, rmax);
        (void)lane;
    }
}

// ---------------------------------------------------------------- p . V ---

// B fragments (with the softmax numerators) and the weighted value sum of
// one pass: p_sm holds the chunk's logits, mx their per-head maxima; then
// the chunk's partials.  Whole CTA.
// fv: the chunk's value weight scale, set on the first pass (red:
// kDecodeWarps floats of shared memory).
template <int BITS, int NQB, int D>
__device__ __forceinline__ void pv_pass(const kivi_cache& c, size_t bh, int TX, const ChunkRange& r,
                                        const DecodeSmem& m, const float (&mx)[NQB], size_t row0,
                                        int nchunks, float* ws_o, float* ws_m, float* ws_l, bool first_pass,
                                        float& fv, float* red)
{
    const int ps = prob_stride(TX), NGv = D >> ilog2(c.G);
    const int n = r.t_end - r.t_begin, nq = r.tq_end - r.t_begin;
    if (first_pass) {
        cp_async_wait_all();  // the staged values
        __syncthreads();
        fv = weight_scale_pow2(cta_max_stat(m.vs, nq * NGv, red));
    }
    pv_weights<NQB>(n, nq, NGv, threadIdx.x, pv_pairs(n, nq), kDecodeThreads, m.p, ps, mx, m.vs, m.vz, fv,
                    m.bb, bb_stride(TX), m.zs, m.zs_on_p);
    __syncthreads();
    pv_chunk<BITS, NQB, D>(c, bh, TX, r.t_begin, r.tq_end, r.t_end, m.vw, m.bb, __frcp_rn(fv), m.part);
    __syncthreads();
    write_partials<NQB, D>(c.G, pv_splits(pv_seg_groups<BITS>(D)), m.part, m.zs, mx, row0, nchunks, ws_o,
                           ws_m, ws_l);
}

template <int BITS, int NQB, int D>
__global__ void __launch_bounds__(kDecodeThreads, 3)
decode_pv_kernel(kivi_cache c, const float* __restrict__ logits, int ldl, int Hq,
                 float* __restrict__ ws_o, float* __restrict__ ws_m, float* __restrict__ ws_l,
                 int nchunks, int TC, int S, const DecodeLayout L)
{
    extern __shared__ __align__(16) float dsm[];
    __shared__ float red[kDecodeWarps * NQB];
    // the combine kernel may launch once every chunk CTA has started: it waits
    // for this grid's results in griddepcontrol.wait
    asm volatile("griddepcontrol.launch_dependents;");
    ChunkRange r;
    if (!chunk_range(c, TC, S, r))
        return;
    const size_t bh = r.bh;
    const DecodeSmem m = carve(dsm, L);
    stage_values<BITS, D>(c, bh, r.t_begin, r.tq_end, m.vw, m.vs, m.vz);
    cp_async_commit();
    const int NQ = Hq / c.H;
    const int n = r.t_end - r.t_begin;
    const int ps = prob_stride(TC + S);
    float fv = 1.0f;
    for (int pass = 0; pass < NQ / NQB; ++pass) {
        const int hq0 = r.h * NQ + pass * NQB;
        __syncthreads();
        float mx[NQB];
#pragma unroll
        for (int h = 0; h < NQB; ++h) {
            const float* lrow = logits + ((size_t)r.b * Hq + hq0 + h) * ldl + r.t_begin;
            mx[h] = -INFINITY;
            for (int t = threadIdx.x; t < n; t += kDecodeThreads) {
                const float x = ld_checked(lrow + t);
                m.p[h * ps + t] = x;
                mx[h] = fmaxf(mx[h], x);
            }
        }
        chunk_max<NQB>(mx, red);
        pv_pass<BITS, NQB, D>(c, bh, TC + S, r, m, mx, ((size_t)r.b * Hq + hq0) * nchunks + r.ci, nchunks,
                           ws_o, ws_m, ws_l, pass == 0, fv, red);
    }
}

// ---------------------------------------------------------------- launch ---

inline DecodeLayout cta_layout(const kivi_cache& c, int Hq, bool keys, bool values)
{
    const int NQ = Hq / c.H, NQB = heads_per_pass(NQ);
    const ChunkPlan cp = chunk_plan(c, Hq);
    return decode_layout(cp.TC, cp.TC + cp.S, c.D, c.bits_k, c.bits_v, c.G, NQB, NQ > NQB, keys, values,
                         cp.zs_on_p);
}

template <class K>
inline cudaError_t set_smem(K kern, size_t bytes)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Grid of the decode kernels: one CTA per (KV head, chunk), 1-D (the host
// keeps B H nchunks below 2^31).
inline dim3 decode_grid(const kivi_cache& c, int Hq) { return dim3((unsigned)(c.B * c.H * pv_chunks(c, Hq))); }

template <int D, int BITS, int NQB>
cudaError_t qk_launch(const kivi_cache& c, const uint16_t* q, int Hq, float sm, float* logits, int ldl,
                      cudaStream_t s)
{
    auto kern = decode_qk_kernel<BITS, NQB, D>;
    const DecodeLayout L = cta_layout(c, Hq, true, false);
    const ChunkPlan cp = chunk_plan(c, Hq);
    cudaError_t e = set_smem(kern, 4 * L.total);
    if (e != cudaSuccess)
        return e;
    kern<<<decode_grid(c, Hq), kDecodeThreads, 4 * L.total, s>>>(c, q, Hq, sm, logits, ldl, cp.TC, cp.S, L);
    return cudaGetLastError();
}

template <int D, int BITS, int NQB>
cudaError_t pv_launch(const kivi_cache& c, const float* logits, int ldl, int Hq, float* ws_o, float* ws_m,
                      float* ws_l, cudaStream_t s)
{
    auto kern = decode_pv_kernel<BITS, NQB, D>;
    const DecodeLayout L = cta_layout(c, Hq, false, true);
    const ChunkPlan cp = chunk_plan(c, Hq);
    cudaError_t e = set_smem(kern, 4 * L.total);
    if (e != cudaSuccess)
        return e;
    kern<<<decode_grid(c, Hq), kDecodeThreads, 4 * L.total, s>>>(c, logits, ldl, Hq, ws_o, ws_m, ws_l,
                                                                pv_chunks(c, Hq), cp.TC, cp.S, L);
    return cudaGetLastError();
}

// Dispatch of the code width (bits) and the query heads per pass (NQB) for
// head dimension D; `launch` is one of the launchers above.
#define KIVI_DECODE_DISPATCH(bits, NQ, launch, ...)                              \
    switch (bits) {                                                              \
    case 2:                                                                      \
        switch (heads_per_pass(NQ)) {                                            \
        case 4: return launch<D, 2, 4>(__VA_ARGS__);                             \
        case 2: return launch<D, 2, 2>(__VA_ARGS__);                             \
        default: return launch<D, 2, 1>(__VA_ARGS__);                            \
        }                                                                        \
    case 4:                                                                      \
        switch (heads_per_pass(NQ)) {                                            \
        case 4: return launch<D, 4, 4>(__VA_ARGS__);                             \
        case 2: return launch<D, 4, 2>(__VA_ARGS__);                             \
        default: return launch<D, 4, 1>(__VA_ARGS__);                            \
        }                                                                        \
    default:                                                                     \
        switch (heads_per_pass(NQ)) {                                            \
        case 4: return launch<D, 8, 4>(__VA_ARGS__);                             \
        case 2: return launch<D, 8, 2>(__VA_ARGS__);                             \
        default: return launch<D, 8, 1>(__VA_ARGS__);                            \
        }                                                                        \
    }

template <int D>
cudaError_t launch_decode_qk_d(const kivi_cache& c, const uint16_t* q, int Hq, float sm_scale, float* logits,
                               int ld_logits, cudaStream_t s)
{
    KIVI_SET_CHECK_RANGES(c, s, {{q, (size_t)c.B * Hq * D * 2}, {logits, (size_t)c.B * Hq * ld_logits * 4}});
    KIVI_DECODE_DISPATCH(c.bits_k, Hq / c.H, qk_launch, c, q, Hq, sm_scale, logits, ld_logits, s)
}

template <int D>
cudaError_t launch_decode_pv_d(const kivi_cache& c, const float* logits, int ld_logits, int Hq, float* ws_o,
                               float* ws_m, float* ws_l, cudaStream_t s)
{
    KIVI_SET_CHECK_RANGES(c, s, {{logits, (size_t)c.B * Hq * ld_logits * 4},
                                 {ws_o, (size_t)c.B * Hq * pv_chunks(c, Hq) * D * 4},
                                 {ws_m, (size_t)c.B * Hq * pv_chunks(c, Hq) * 4},
                                 {ws_l, (size_t)c.B * Hq * pv_chunks(c, Hq) * 4}});
    KIVI_DECODE_DISPATCH(c.bits_v, Hq / c.H, pv_launch, c, logits, ld_logits, Hq, ws_o, ws_m, ws_l, s)
}

#undef KIVI_DECODE_DISPATCH

// Instantiates the two launchers for one head dimension.
#define KIVI_DECODE_INSTANTIATE(DIM)                                                                      \
    template cudaError_t launch_decode_qk_d<DIM>(const kivi_cache&, const uint16_t*, int, float, float*, \
                                                 int, cudaStream_t);                                      \
    template cudaError_t launch_decode_pv_d<DIM>(const kivi_cache&, const float*, int, int, float*,      \
                                                 float*, float*, cudaStream_t);

}  // namespace kivi
