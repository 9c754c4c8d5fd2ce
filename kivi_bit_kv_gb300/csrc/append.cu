// append.cu -- append one decoded token per sequence, flushing the oldest G
// residual tokens into the packed cache when the residual reaches R + G
// (CacheForge README, "How it works": recent tokens stay at higher precision;
// the quantization flow during decoding).
//
// Kernel 1, one CTA per (h, b): writes k, v into ring slot len mod (R+G) and,
// on a flush step, quantizes the G oldest ring tokens exactly like a prefix
// group (same lane quantizers as the encode kernels).  Kernel 2 advances
// len[b]; it runs after every CTA of kernel 1 has read the old length, so no
// CTA can observe a half-updated count.
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

template <int BV, int G>
__device__ __forceinline__ void flush_values(const kivi_cache& c, size_t bh, int Tq)
{
    const int D = c.D, NG = D / G, RG = c.R + c.G;
    for (int task = threadIdx.x; task < G * NG; task += blockDim.x) {
        const int gi = task % NG, r = task / NG;
        const int t = Tq + r;
        const uint16_t* src = c.vres + (bh * RG + t % RG) * D + gi * G;
        uint4 raw[G / 8];
#pragma unroll
        for (int v = 0; v < G / 8; ++v)
            raw[v] = ld_checked(reinterpret_cast<const uint4*>(src + v * 8));
        quant_store_value_group<BV, G>(c, bh, t, gi, raw);
    }
}

// Keys of a flushed group: one G-token group per channel, lanes (s, j) with s
// fastest (S = G/16 lanes per channel column).
template <int BK, int S>
__device__ __forceinline__ void flush_keys(const kivi_cache& c, size_t bh, int Tq)
{
    const int D = c.D, RG = c.R + c.G, NC = D / kLaneChans;
    const int lane = threadIdx.x & 31;
    const unsigned smask = (((1u << S) - 1u) << (lane & ~(S - 1)));
    for (int task = threadIdx.x; task < S * NC; task += blockDim.x) {
        const int s = task % S, j = task / S;
        const int t0 = Tq + s * kLaneTokens;
        uint4 raw[kLaneTokens];
#pragma unroll
        for (int i = 0; i < kLaneTokens; ++i)
            raw[i] = ld_checked(reinterpret_cast<const uint4*>(c.kres + (bh * RG + (t0 + i) % RG) * D +
                                                                (size_t)j * kLaneChans));
        // RG and t0 are multiples of 16: the lane's 16 ring rows never wrap
        quant_store_key_lane<BK, S>(c, bh, t0, Tq / c.G, j, s, smask, raw,
                                    c.kres + (bh * RG + t0 % RG) * D + (size_t)j * kLaneChans, D);
    }
}

template <int BK, int BV>
__global__ void __launch_bounds__(128)
append_kernel(kivi_cache c, const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
              int32_t* status)
{
    const size_t bh = blockIdx.x;
    const int b = (int)(bh / c.H), h = (int)(bh % c.H);
    const int L = ld_checked(c.len + b);
    if (L + 1 > c.Tmax) {
        if (h == 0 && threadIdx.x == 0)
            atomicExch(status, KIVI_ECAPACITY);
        return;
    }
    const int D = c.D, G = c.G, RG = c.R + c.G;
    const int slot = L % RG;
    for (int i = threadIdx.x; i < D / kLaneChans; i += blockDim.x) {
        const size_t o = (bh * RG + slot) * D + (size_t)i * kLaneChans;
        const size_t in = bh * D + (size_t)i * kLaneChans;
        st_checked(reinterpret_cast<uint4*>(c.kres + o), ld_checked(reinterpret_cast<const uint4*>(k + in)));
        st_checked(reinterpret_cast<uint4*>(c.vres + o), ld_checked(reinterpret_cast<const uint4*>(v + in)));
    }
    const int Tq = quantized_tokens(L, G, c.R);
    if (L + 1 - Tq != RG)
        return;  // uniform over the CTA
    __syncthreads();  // the new token is visible to every thread of the CTA

    // keys, then values: G token rows x D/G channel groups, one lane per group
    switch (G) {
    case 32:
        flush_keys<BK, 2>(c, bh, Tq);
        flush_values<BV, 32>(c, bh, Tq);
        break;
    case 64:
        flush_keys<BK, 4>(c, bh, Tq);
        flush_values<BV, 64>(c, bh, Tq);
        break;
    default:
        flush_keys<BK, 8>(c, bh, Tq);
        flush_values<BV, 128>(c, bh, Tq);
        break;
    }
}

__global__ void advance_len_kernel(int32_t* len, int B, int Tmax)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) {
        const int L = ld_checked(len + b);
        if (L + 1 <= Tmax)
            st_checked(len + b, L + 1);
    }
}

template <int BK>
static void launch_append_bk(const kivi_cache& c, const uint16_t* k, const uint16_t* v,
                             int32_t* status, cudaStream_t s)
{
    const dim3 grid(c.B * c.H);
    switch (c.bits_v) {
    case 2: append_kernel<BK, 2><<<grid, 128, 0, s>>>(c, k, v, status); break;
    case 4: append_kernel<BK, 4><<<grid, 128, 0, s>>>(c, k, v, status); break;
    default: append_kernel<BK, 8><<<grid, 128, 0, s>>>(c, k, v, status); break;
    }
}

cudaError_t launch_append(const kivi_cache& c, const uint16_t* k, const uint16_t* v,
                          int32_t* status, cudaStream_t s)
{
    KIVI_SET_CHECK_RANGES(c, s, {{k, (size_t)c.B * c.H * c.D * 2}, {v, (size_t)c.B * c.H * c.D * 2}, {status, 4}});
    switch (c.bits_k) {
    case 2: launch_append_bk<2>(c, k, v, status, s); break;
    case 4: launch_append_bk<4>(c, k, v, status, s); break;
    default: launch_append_bk<8>(c, k, v, status, s); break;
    }
    advance_len_kernel<<<(c.B + 127) / 128, 128, 0, s>>>(c.len, c.B, c.Tmax);
    return cudaGetLastError();
}

#ifdef KIVI_CHECKS
int32_t check_word_append() { return take_check_word(); }
#endif

}  // namespace kivi
