// decode.cu -- decode attention over the packed KIVI cache plus the fp16
// residual, with dequantization fused into the loads (the decode-time consumer
// of the cache: q . K_hat^T, softmax, p . V_hat).
//
// Three entry kernels share the tiles of decode_mma.cuh:
//   decode_qk_kernel         logits to global memory (kivi_decode_qk)
//   decode_pv_kernel         softmax + p . V from given logits (kivi_decode_pv)
//   decode_attention_kernel  both, logits kept in shared memory
//                            (kivi_decode_attention)
// Each CTA owns one KV head and one 1024-token chunk; the pv and fused kernels
// leave per-chunk (o, m, l) partials that decode_combine_kernel merges.
#include <math.h>

#include "decode_mma.cuh"
#include "kivi_launch.h"

namespace kivi {

// Per-CTA coordinates of a decode chunk.
struct ChunkRange {
    int b, h, n, t_begin, t_end, Tq, tq_end;
};

__device__ __forceinline__ bool chunk_range(const kivi_cache& c, ChunkRange& r)
{
    const size_t bh = blockIdx.x;
    r.b = (int)(bh / c.H);
    r.h = (int)(bh % c.H);
    r.n = c.len[r.b];
    r.t_begin = blockIdx.y * kChunkTokens;
    if (r.t_begin >= r.n)
        return false;
    r.t_end = min(r.t_begin + kChunkTokens, r.n);
    r.Tq = quantized_tokens(r.n, c.G, c.R);
    r.tq_end = max(r.t_begin, min(r.t_end, r.Tq));
    return true;
}

// ---------------------------------------------------------------- q . K ---

template <int BITS, int NQB>
__global__ void __launch_bounds__(kDecodeThreads)
decode_qk_kernel(kivi_cache c, const uint16_t* __restrict__ q, int Hq, float sm_scale,
                 float* __restrict__ logits, int ldl)
{
    __shared__ __align__(16) float qs[NQB * qstride_of(256)];
    __shared__ float fac[NQB];
    ChunkRange r;
    if (!chunk_range(c, r))
        return;
    const size_t bh = blockIdx.x;
    const int NQ = Hq / c.H;
    for (int pass = 0; pass < NQ / NQB; ++pass) {
        const int hq0 = r.h * NQ + pass * NQB;
        __syncthreads();
        stage_q<NQB>(q + ((size_t)r.b * Hq + hq0) * c.D, c.D, sm_scale, qs, fac);
        __syncthreads();
        float* out = logits + ((size_t)r.b * Hq + hq0) * ldl;
        auto sink = [&](int h, int t, float s) { out[(size_t)h * ldl + t] = s; };
        qk_quantized<BITS, NQB>(c, bh, r.t_begin, r.tq_end, qs, fac, sink);
        qk_residual<NQB>(c, bh, r.tq_end, r.t_end, qs, fac, sink);
    }
}

// ---------------------------------------------------------------- p . V ---

// Dynamic shared memory of the pv / fused kernels: p [NQB][1024], then the
// split partials.
__host__ __device__ constexpr size_t pv_smem_bytes(int NQB, int D, int G)
{
    return ((size_t)NQB * kChunkTokens + pv_part_floats(NQB, D, G)) * sizeof(float);
}

template <int BITS, int NQB>
__global__ void __launch_bounds__(kDecodeThreads)
decode_pv_kernel(kivi_cache c, const float* __restrict__ logits, int ldl, int Hq,
                 float* __restrict__ ws_o, float* __restrict__ ws_m, float* __restrict__ ws_l,
                 int nchunks)
{
    extern __shared__ __align__(16) float pv_smem[];
    __shared__ float red[kDecodeWarps * NQB];
    float* p_sm = pv_smem;
    float* o_part = p_sm + NQB * kChunkTokens;
    float* z_part = o_part + kDecodeWarps * NQB * c.D;
    ChunkRange r;
    if (!chunk_range(c, r))
        return;
    const size_t bh = blockIdx.x;
    const int NQ = Hq / c.H;
    const int n = r.t_end - r.t_begin;
    const int NCB = (c.D / (32 / BITS)) / ValTile<BITS, NQB>::WC;
    for (int pass = 0; pass < NQ / NQB; ++pass) {
        const int hq0 = r.h * NQ + pass * NQB;
        __syncthreads();
        for (int i = threadIdx.x; i < NQB * n; i += kDecodeThreads) {
            const int h = i / n, t = i % n;
            p_sm[h * kChunkTokens + t] = logits[((size_t)r.b * Hq + hq0 + h) * ldl + r.t_begin + t];
        }
        __syncthreads();
        float m[NQB], l[NQB];
        chunk_softmax<NQB>(p_sm, n, m, l, red);
        pv_chunk<BITS, NQB>(c, bh, r.t_begin, r.tq_end, r.t_end, p_sm, o_part, z_part);
        __syncthreads();
        const size_t row0 = ((size_t)r.b * Hq + hq0) * nchunks + blockIdx.y;
        write_partials<NQB>(c.D, c.G, pv_splits(NCB), o_part, z_part, m, l, row0, nchunks, ws_o,
                            ws_m, ws_l);
    }
}

// ------------------------------------------------------------ attention ---

template <int BITS, int NQB>
__global__ void __launch_bounds__(kDecodeThreads)
decode_attention_kernel(kivi_cache c, const uint16_t* __restrict__ q, int Hq, float sm_scale,
                        float* __restrict__ ws_o, float* __restrict__ ws_m,
                        float* __restrict__ ws_l, int nchunks)
{
    extern __shared__ __align__(16) float pv_smem[];
    __shared__ __align__(16) float qs[NQB * qstride_of(256)];
    __shared__ float fac[NQB];
    __shared__ float red[kDecodeWarps * NQB];
    float* p_sm = pv_smem;
    float* o_part = p_sm + NQB * kChunkTokens;
    float* z_part = o_part + kDecodeWarps * NQB * c.D;
    ChunkRange r;
    if (!chunk_range(c, r))
        return;
    const size_t bh = blockIdx.x;
    const int NQ = Hq / c.H;
    const int NCB = (c.D / (32 / BITS)) / ValTile<BITS, NQB>::WC;
    for (int pass = 0; pass < NQ / NQB; ++pass) {
        const int hq0 = r.h * NQ + pass * NQB;
        __syncthreads();
        stage_q<NQB>(q + ((size_t)r.b * Hq + hq0) * c.D, c.D, sm_scale, qs, fac);
        __syncthreads();
        auto sink = [&](int h, int t, float s) { p_sm[h * kChunkTokens + t - r.t_begin] = s; };
        qk_quantized<BITS, NQB>(c, bh, r.t_begin, r.tq_end, qs, fac, sink);
        qk_residual<NQB>(c, bh, r.tq_end, r.t_end, qs, fac, sink);
        __syncthreads();
        float m[NQB], l[NQB];
        chunk_softmax<NQB>(p_sm, r.t_end - r.t_begin, m, l, red);
        pv_chunk<BITS, NQB>(c, bh, r.t_begin, r.tq_end, r.t_end, p_sm, o_part, z_part);
        __syncthreads();
        const size_t row0 = ((size_t)r.b * Hq + hq0) * nchunks + blockIdx.y;
        write_partials<NQB>(c.D, c.G, pv_splits(NCB), o_part, z_part, m, l, row0, nchunks, ws_o,
                            ws_m, ws_l);
    }
}

// out[b][hq][d] = sum_c o_c[d] e^(m_c - M) / sum_c l_c e^(m_c - M), M = max m_c.
__global__ void __launch_bounds__(256)
decode_combine_kernel(const int32_t* __restrict__ len, int Hq, int D, int nchunks,
                      const float* __restrict__ ws_o, const float* __restrict__ ws_m,
                      const float* __restrict__ ws_l, float* __restrict__ out)
{
    const size_t bhq = blockIdx.x;
    const int b = (int)(bhq / Hq);
    const int n = len[b];
    const int nv = (n + kChunkTokens - 1) / kChunkTokens;
    const float* mrow = ws_m + bhq * nchunks;
    const float* lrow = ws_l + bhq * nchunks;
    float M = -INFINITY;
    for (int k = 0; k < nv; ++k)
        M = fmaxf(M, mrow[k]);
    float L = 0.0f;
    for (int k = 0; k < nv; ++k)
        L += lrow[k] * expf(mrow[k] - M);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float o = 0.0f;
        for (int k = 0; k < nv; ++k)
            o = fmaf(ws_o[(bhq * nchunks + k) * D + d], expf(mrow[k] - M), o);
        out[bhq * D + d] = nv > 0 ? o / L : 0.0f;
    }
}

// ---------------------------------------------------------------- launch ---

int pv_chunk_tokens(int) { return kChunkTokens; }
int qk_chunk_tokens(int) { return kChunkTokens; }
int pv_chunks(const kivi_cache& c) { return (c.Tmax + kChunkTokens - 1) / kChunkTokens; }

static cudaError_t combine(const kivi_cache& c, int Hq, int nch, const float* ws_o,
                           const float* ws_m, const float* ws_l, float* out, cudaStream_t s)
{
    decode_combine_kernel<<<c.B * Hq, c.D < 256 ? c.D : 256, 0, s>>>(c.len, Hq, c.D, nch, ws_o,
                                                                     ws_m, ws_l, out);
    return cudaGetLastError();
}

template <int BITS, int NQB>
static cudaError_t qk_launch(const kivi_cache& c, const uint16_t* q, int Hq, float sm,
                             float* logits, int ldl, cudaStream_t s)
{
    const dim3 grid(c.B * c.H, pv_chunks(c));
    decode_qk_kernel<BITS, NQB><<<grid, kDecodeThreads, 0, s>>>(c, q, Hq, sm, logits, ldl);
    return cudaGetLastError();
}

template <int BITS>
static cudaError_t qk_bits(const kivi_cache& c, const uint16_t* q, int Hq, float sm,
                           float* logits, int ldl, cudaStream_t s)
{
    switch (heads_per_pass(Hq / c.H)) {
    case 8: return qk_launch<BITS, 8>(c, q, Hq, sm, logits, ldl, s);
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
    const size_t smem = pv_smem_bytes(NQB, c.D, c.G);
    auto kern = decode_pv_kernel<BITS, NQB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const int nch = pv_chunks(c);
    kern<<<dim3(c.B * c.H, nch), kDecodeThreads, smem, s>>>(c, logits, ldl, Hq, ws_o, ws_m, ws_l, nch);
    return cudaGetLastError();
}

template <int BITS>
static cudaError_t pv_bits(const kivi_cache& c, const float* logits, int ldl, int Hq, float* ws_o,
                           float* ws_m, float* ws_l, cudaStream_t s)
{
    switch (heads_per_pass(Hq / c.H)) {
    case 8: return pv_launch<BITS, 8>(c, logits, ldl, Hq, ws_o, ws_m, ws_l, s);
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
    return combine(c, Hq, pv_chunks(c), ws_o, ws_m, ws_l, out, s);
}

template <int BITS, int NQB>
static cudaError_t attn_launch(const kivi_cache& c, const uint16_t* q, int Hq, float sm,
                               float* ws_o, float* ws_m, float* ws_l, cudaStream_t s)
{
    const size_t smem = pv_smem_bytes(NQB, c.D, c.G);
    auto kern = decode_attention_kernel<BITS, NQB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const int nch = pv_chunks(c);
    kern<<<dim3(c.B * c.H, nch), kDecodeThreads, smem, s>>>(c, q, Hq, sm, ws_o, ws_m, ws_l, nch);
    return cudaGetLastError();
}

template <int BITS>
static cudaError_t attn_bits(const kivi_cache& c, const uint16_t* q, int Hq, float sm,
                             float* ws_o, float* ws_m, float* ws_l, cudaStream_t s)
{
    switch (heads_per_pass(Hq / c.H)) {
    case 8: return attn_launch<BITS, 8>(c, q, Hq, sm, ws_o, ws_m, ws_l, s);
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
    return combine(c, Hq, pv_chunks(c), ws_o, ws_m, ws_l, out, s);
}

}  // namespace kivi
