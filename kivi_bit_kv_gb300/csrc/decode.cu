// decode.cu -- host side of decode attention: the chunk plan, the dispatch
// to the kernels of the head dimension (decode_kernels.cuh, instantiated by
// decode_d64.cu / decode_d128.cu / decode_d256.cu), and the kernel that
// merges the per-chunk (o, m, l) partials.
#include <math.h>

#include "decode_mma.cuh"
#include "decode_stream.cuh"
#include "kivi_launch.h"

namespace kivi {

// The streamed decode is instantiated in decode_stream_d<D>_k<BK>.cu, not here.
#define KIVI_STREAM_EXTERN(DIM, BK)                                                                              \
    extern template cudaError_t launch_decode_stream<DIM, BK>(const kivi_cache&, const uint16_t*, int, float, \
                                                              float*, float*, cudaStream_t);
KIVI_STREAM_EXTERN(64, 2)
KIVI_STREAM_EXTERN(64, 4)
KIVI_STREAM_EXTERN(64, 8)
KIVI_STREAM_EXTERN(128, 2)
KIVI_STREAM_EXTERN(128, 4)
KIVI_STREAM_EXTERN(128, 8)
KIVI_STREAM_EXTERN(256, 2)
KIVI_STREAM_EXTERN(256, 4)
KIVI_STREAM_EXTERN(256, 8)
#undef KIVI_STREAM_EXTERN

// out[b][hq][d] = sum_c o_c[d] e^(m_c - M) / sum_c l_c e^(m_c - M), M = max m_c
// over the chunks c that hold tokens of sequence b.  CTA (b hq, y) writes
// channels [y C, y C + C), C = D / gridDim.y: one merge of the (m, l) pairs
// (each thread folds its chunks with the usual rescaling, then warps and
// warps' results in a fixed order) and the weighted sum with one 16-byte load
// per (chunk, column) and thread.  The first rows of o and their maxima are
// loaded together with the (m, l) pairs, so the merge costs one round trip to
// L2 after the chunk kernel's results become visible.
constexpr int kCombineThreads = 128;

__device__ __forceinline__ void merge_ml(float& m, float& l, float m2, float l2)
{
    if (m2 > m) {
        l = fmaf(l, expf(m - m2), l2);
        m = m2;
    } else if (m2 > -INFINITY) {
        l = fmaf(l2, expf(m2 - m), l);
    }
}

__global__ void __launch_bounds__(kCombineThreads)
decode_combine_kernel(const int32_t* __restrict__ len, int Hq, int D, int nchunks, int TC, int S,
                      const float* __restrict__ ws_o, const float* __restrict__ ws_m,
                      const float* __restrict__ ws_l, float* __restrict__ out)
{
    __shared__ __align__(16) float4 part[kCombineThreads];  // [rows][V] column sums
    __shared__ float red_m[kDecodeWarps], red_l[kDecodeWarps];
    constexpr int KP = 4;  // rows of o each thread loads before the merge
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t bhq = blockIdx.x;
    const int C = D / gridDim.y, c0 = blockIdx.y * C;
    const int V = C / 4, rows = kCombineThreads / V;
    const int v = threadIdx.x % V, r0 = threadIdx.x / V;
    const int n = ld_checked(len + bhq / Hq);  // not written by the chunk kernel: read before the wait
    const int nv = decode_chunks(n, TC, S);
    const float* mrow = ws_m + bhq * nchunks;
    const float* lrow = ws_l + bhq * nchunks;
    const float4* o4 = reinterpret_cast<const float4*>(ws_o + bhq * nchunks * D + c0);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float4 op[KP];
    float mp[KP];
#pragma unroll
    for (int i = 0; i < KP; ++i) {
        const int k = r0 + i * rows;
        if (k < nv) {
            op[i] = ld_checked(o4 + (size_t)k * (D / 4) + v);
            mp[i] = ld_checked(mrow + k);
        }
    }
    float m = -INFINITY, l = 0.0f;
    for (int k = threadIdx.x; k < nv; k += kCombineThreads)
        merge_ml(m, l, ld_checked(mrow + k), ld_checked(lrow + k));
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), l2 = __shfl_xor_sync(0xffffffffu, l, o);
        merge_ml(m, l, m2, l2);
    }
    if (lane == 0) {
        red_m[warp] = m;
        red_l[warp] = l;
    }
    __syncthreads();
    float M = red_m[0], L = red_l[0];
#pragma unroll
    for (int w = 1; w < kDecodeWarps; ++w)
        merge_ml(M, L, red_m[w], red_l[w]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < KP; ++i) {
        if (r0 + i * rows < nv) {
            const float e = expf(mp[i] - M);
            acc.x = fmaf(op[i].x, e, acc.x);
            acc.y = fmaf(op[i].y, e, acc.y);
            acc.z = fmaf(op[i].z, e, acc.z);
            acc.w = fmaf(op[i].w, e, acc.w);
        }
    }
#pragma unroll 4
    for (int k = r0 + KP * rows; k < nv; k += rows) {
        const float4 o = ld_checked(o4 + (size_t)k * (D / 4) + v);
        const float e = expf(ld_checked(mrow + k) - M);
        acc.x = fmaf(o.x, e, acc.x);
        acc.y = fmaf(o.y, e, acc.y);
        acc.z = fmaf(o.z, e, acc.z);
        acc.w = fmaf(o.w, e, acc.w);
    }
    part[r0 * V + v] = acc;
    __syncthreads();
    for (int d = threadIdx.x; d < C; d += kCombineThreads) {
        const float* pf = reinterpret_cast<const float*>(part);
        float o = 0.0f;
        for (int r = 0; r < rows; ++r)
            o += pf[r * C + d];
        st_checked(out + bhq * D + c0 + d, nv > 0 ? o / L : 0.0f);
    }
}

// ---------------------------------------------------------------- launch ---

int pv_chunks(const kivi_cache& c, int Hq)
{
    const ChunkPlan cp = chunk_plan(c, Hq);
    return decode_chunks(c.Tmax, cp.TC, cp.S);
}

static cudaError_t combine(const kivi_cache& c, int Hq, const float* ws_o, const float* ws_m,
                           const float* ws_l, float* out, cudaStream_t s)
{
    const int nch = pv_chunks(c, Hq);
    KIVI_SET_CHECK_RANGES(c, s, {{ws_o, (size_t)c.B * Hq * nch * c.D * 4}, {ws_m, (size_t)c.B * Hq * nch * 4},
                                 {ws_l, (size_t)c.B * Hq * nch * 4}, {out, (size_t)c.B * Hq * c.D * 4}});
    // channel slices per (b, hq): at least two CTAs per SM in all, 32 channels or more each
    const int rows = c.B * Hq;
    int ds = 1;
    while (ds < c.D / 32 && rows * ds < 2 * sm_count())
        ds *= 2;
    const ChunkPlan cp = chunk_plan(c, Hq);
    // programmatic dependent launch: the combine CTAs are scheduled while the
    // chunk kernel drains and wait in griddepcontrol.wait for its results
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows, ds);
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_combine_kernel, c.len, Hq, c.D, nch, cp.TC, cp.S,
                                       (const float*)ws_o, (const float*)ws_m, (const float*)ws_l, out);
    if (e != cudaSuccess) {  // attribute not supported: an ordinary launch
        (void)cudaGetLastError();
        decode_combine_kernel<<<dim3(rows, ds), kCombineThreads, 0, s>>>(c.len, Hq, c.D, nch, cp.TC, cp.S, ws_o,
                                                                        ws_m, ws_l, out);
    }
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
                                    float* out, float* ws, cudaStream_t s)
{
#define KIVI_STREAM_BK(DIM)                                                                  \
    switch (c.bits_k) {                                                                      \
    case 2: return launch_decode_stream<DIM, 2>(c, q, Hq, sm_scale, out, ws, s);            \
    case 4: return launch_decode_stream<DIM, 4>(c, q, Hq, sm_scale, out, ws, s);            \
    default: return launch_decode_stream<DIM, 8>(c, q, Hq, sm_scale, out, ws, s);           \
    }
    switch (c.D) {
    case 64: KIVI_STREAM_BK(64)
    case 128: KIVI_STREAM_BK(128)
    default: KIVI_STREAM_BK(256)
    }
#undef KIVI_STREAM_BK
}

size_t stream_ws_bytes(const kivi_cache& c, int Hq)
{
    const int NQ = Hq / c.H;
    return stream_ws_floats(c.D, heads_per_pass(NQ), kMaxStreamCTAs) * sizeof(float);
}

#ifdef KIVI_CHECKS
int32_t check_word_decode() { return take_check_word(); }
#endif

}  // namespace kivi
