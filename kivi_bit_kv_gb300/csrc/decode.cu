// decode.cu -- host side of decode attention: the chunk plan, the dispatch
// to the kernels of the head dimension (decode_kernels.cuh, instantiated by
// decode_d64.cu / decode_d128.cu / decode_d256.cu), and the kernel that
// merges the per-chunk (o, m, l) partials.
#include <math.h>

#include "decode_mma.cuh"
#include "kivi_launch.h"

namespace kivi {

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

int chunk_tokens(const kivi_cache& c, int Hq) { return chunk_plan(c, Hq).TC; }
int pv_chunks(const kivi_cache& c, int Hq)
{
    const ChunkPlan cp = chunk_plan(c, Hq);
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
    const ChunkPlan cp = chunk_plan(c, Hq);
    decode_combine_kernel<<<c.B * Hq, kCombineThreads, smem, s>>>(c.len, Hq, c.D, nch, cp.TC, cp.S,
                                                                  ws_o, ws_m, ws_l, out);
    return cudaGetLastError();
}

cudaError_t launch_decode_qk(const kivi_cache& c, const uint16_t* q, int Hq, float sm_scale,
                             float* logits, int ld_logits, cudaStream_t s)
{
    switch (c.D) {
    case 64: return launch_decode_qk_d<64>(c, q, Hq, sm_scale, logits, ld_logits, s);
    case 128: return launch_decode_qk_d<128>(c, q, Hq, sm_scale, logits, ld_logits, s);
    default: return launch_decode_qk_d<256>(c, q, Hq, sm_scale, logits, ld_logits, s);
    }
}

cudaError_t launch_decode_pv(const kivi_cache& c, const float* logits, int ld_logits, int Hq,
                             float* out, float* ws_o, float* ws_m, float* ws_l, cudaStream_t s)
{
    cudaError_t e;
    switch (c.D) {
    case 64: e = launch_decode_pv_d<64>(c, logits, ld_logits, Hq, ws_o, ws_m, ws_l, s); break;
    case 128: e = launch_decode_pv_d<128>(c, logits, ld_logits, Hq, ws_o, ws_m, ws_l, s); break;
    default: e = launch_decode_pv_d<256>(c, logits, ld_logits, Hq, ws_o, ws_m, ws_l, s); break;
    }
    if (e != cudaSuccess)
        return e;
    return combine(c, Hq, ws_o, ws_m, ws_l, out, s);
}

cudaError_t launch_decode_attention(const kivi_cache& c, const uint16_t* q, int Hq, float sm_scale,
                                    float* out, float* ws_o, float* ws_m, float* ws_l,
                                    cudaStream_t s)
{
    // the fused kernel needs bits_k == bits_v (checked by the caller)
    cudaError_t e;
    switch (c.D) {
    case 64: e = launch_decode_attention_d<64>(c, q, Hq, sm_scale, ws_o, ws_m, ws_l, s); break;
    case 128: e = launch_decode_attention_d<128>(c, q, Hq, sm_scale, ws_o, ws_m, ws_l, s); break;
    default: e = launch_decode_attention_d<256>(c, q, Hq, sm_scale, ws_o, ws_m, ws_l, s); break;
    }
    if (e != cudaSuccess)
        return e;
    return combine(c, Hq, ws_o, ws_m, ws_l, out, s);
}

}  // namespace kivi
