// quant.cu -- prefix encode of keys and values (one pass: min/max, scale and
// zero, codes, packing), plus the copy of the unquantized tail into the ring.
//
// Keys are quantized per channel over groups of G tokens and values per token
// over groups of G channels (CacheForge README, "How it works"); min and max
// come out of one combined reduction and the scales are built in place
// ("Contribution scope" of the same README).  Statistics are fp32 and codes
// are packed into int32 words (CacheSeek PR #4 change notes).
//
// HBM-bound: every fp16 element is read once with a 16-byte streaming load
// and written once as a b-bit code; statistics add 8 bytes per group column.
// Grids are 2-D -- x over token tiles, y over (b, h) slices -- so all index
// arithmetic is 32-bit shifts and masks.
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

constexpr int kEncodeThreads = 256;

__device__ __forceinline__ int log2_pow2(int x) { return __ffs(x) - 1; }

// Keys.  One lane = 16 tokens x 8 channels of a (b, h, G-token group) tile;
// the G/16 lanes of a tile column are adjacent.  A CTA covers 256 / (S*NC)
// groups of one slice.  Tiles past Tq copy their tokens into the ring.
template <int BITS>
__global__ void __launch_bounds__(kEncodeThreads)
quant_keys_kernel(kivi_cache c, const uint16_t* __restrict__ K, int T,
                  const int32_t* __restrict__ seq_lens)
{
    const int D = c.D;
    const int S = c.G / kLaneTokens, lgS = log2_pow2(S);
    const int NC = D / kLaneChans, lgNC = log2_pow2(NC);
    const int lane = threadIdx.x & 31;
    const unsigned smask = (((1u << S) - 1u) << (lane & ~(S - 1)));
    const int s = threadIdx.x & (S - 1);
    const int j = (threadIdx.x >> lgS) & (NC - 1);
    const int g = blockIdx.x * (kEncodeThreads >> (lgS + lgNC)) + (threadIdx.x >> (lgS + lgNC));
    const int t0 = g * c.G + s * kLaneTokens;
    const int RG = c.R + c.G;

    for (int bh = blockIdx.y; bh < c.B * c.H; bh += gridDim.y) {
        const int b = bh / c.H;
        const int n = seq_lens ? min(max(seq_lens[b], 0), T) : T;
        if (blockIdx.x == 0 && threadIdx.x == 0 && bh % c.H == 0)
            c.len[b] = n;
        if (g * c.G >= n)
            continue;  // uniform over the tile column
        const int Tq = quantized_tokens(n, c.G, c.R);
        const uint16_t* src = K + (size_t)bh * T * D + j * kLaneChans;
        if ((g + 1) * c.G <= Tq) {
            uint4 raw[kLaneTokens];
#pragma unroll
            for (int i = 0; i < kLaneTokens; ++i)
                raw[i] = ld_stream(src + (size_t)(t0 + i) * D);
            quant_store_key_lane<BITS>(c, bh, t0, g, j, s, S, smask, raw, src + (size_t)t0 * D, D);
        } else {
            for (int i = 0; i < kLaneTokens; ++i) {
                const int t = t0 + i;
                if (t >= Tq && t < n)
                    st_stream(c.kres + ((size_t)bh * RG + t % RG) * D + j * kLaneChans,
                              ld_stream(src + (size_t)t * D));
            }
        }
    }
}

// Values.  One lane = one channel group (G channels) of U token rows, so
// min/max, the division and the packing stay inside the lane.  A CTA covers
// 256 / (D/G) * U rows of one slice.
template <int BITS, int G>
__global__ void __launch_bounds__(kEncodeThreads)
quant_values_kernel(kivi_cache c, const uint16_t* __restrict__ V, int T,
                    const int32_t* __restrict__ seq_lens)
{
    constexpr int U = G == 32 ? 2 : 1;  // rows per lane: 8-16 loads in flight
    constexpr int NV = G / 8;           // 16-byte vectors per group
    const int D = c.D;
    const int NG = D / G, lgNG = log2_pow2(NG);
    const int gi = threadIdx.x & (NG - 1);
    const int rows_per_pass = kEncodeThreads >> lgNG;
    const int r0 = blockIdx.x * rows_per_pass * U + (threadIdx.x >> lgNG);
    const int RG = c.R + c.G;

    for (int bh = blockIdx.y; bh < c.B * c.H; bh += gridDim.y) {
        const int b = bh / c.H;
        const int n = seq_lens ? min(max(seq_lens[b], 0), T) : T;
        if (blockIdx.x == 0 && threadIdx.x == 0 && bh % c.H == 0)
            c.len[b] = n;
        const int Tq = quantized_tokens(n, c.G, c.R);
        const uint16_t* src = V + (size_t)bh * T * D + gi * G;
        uint4 raw[U][NV];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = r0 + u * rows_per_pass;
            if (t < n) {
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    raw[u][v] = ld_stream(src + (size_t)t * D + v * 8);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = r0 + u * rows_per_pass;
            if (t < Tq) {
                quant_store_value_group<BITS, G>(c, (size_t)bh, t, gi, raw[u]);
            } else if (t < n) {
                uint16_t* dst = c.vres + ((size_t)bh * RG + t % RG) * D + gi * G;
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    st_stream(dst + v * 8, raw[u][v]);
            }
        }
    }
}

__global__ void set_len_kernel(int32_t* len, int B, int T, const int32_t* __restrict__ seq_lens)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B)
        len[b] = seq_lens ? min(max(seq_lens[b], 0), T) : T;
}

static dim3 encode_grid(const kivi_cache& c, int tiles)
{
    const int bh = c.B * c.H;
    return dim3((unsigned)(tiles > 0 ? tiles : 1), (unsigned)(bh < 65535 ? bh : 65535));
}

cudaError_t launch_quant_keys(const kivi_cache& c, const uint16_t* K, int T,
                              const int32_t* seq_lens, cudaStream_t s)
{
    if (T > 0) {
        const int groups_per_cta = kEncodeThreads / ((c.G / kLaneTokens) * (c.D / kLaneChans));
        const int groups = (T + c.G - 1) / c.G;
        const dim3 grid = encode_grid(c, (groups + groups_per_cta - 1) / groups_per_cta);
        switch (c.bits_k) {
        case 2: quant_keys_kernel<2><<<grid, kEncodeThreads, 0, s>>>(c, K, T, seq_lens); break;
        case 4: quant_keys_kernel<4><<<grid, kEncodeThreads, 0, s>>>(c, K, T, seq_lens); break;
        default: quant_keys_kernel<8><<<grid, kEncodeThreads, 0, s>>>(c, K, T, seq_lens); break;
        }
    } else {
        set_len_kernel<<<(c.B + 127) / 128, 128, 0, s>>>(c.len, c.B, T, seq_lens);
    }
    return cudaGetLastError();
}

template <int BITS>
static void quant_values_bits(const kivi_cache& c, const uint16_t* V, int T,
                              const int32_t* seq_lens, cudaStream_t s)
{
    const int U = c.G == 32 ? 2 : 1;
    const int rows_per_cta = kEncodeThreads / (c.D / c.G) * U;
    const dim3 grid = encode_grid(c, (T + rows_per_cta - 1) / rows_per_cta);
    switch (c.G) {
    case 32: quant_values_kernel<BITS, 32><<<grid, kEncodeThreads, 0, s>>>(c, V, T, seq_lens); break;
    case 64: quant_values_kernel<BITS, 64><<<grid, kEncodeThreads, 0, s>>>(c, V, T, seq_lens); break;
    default: quant_values_kernel<BITS, 128><<<grid, kEncodeThreads, 0, s>>>(c, V, T, seq_lens); break;
    }
}

cudaError_t launch_quant_values(const kivi_cache& c, const uint16_t* V, int T,
                                const int32_t* seq_lens, cudaStream_t s)
{
    if (T > 0) {
        switch (c.bits_v) {
        case 2: quant_values_bits<2>(c, V, T, seq_lens, s); break;
        case 4: quant_values_bits<4>(c, V, T, seq_lens, s); break;
        default: quant_values_bits<8>(c, V, T, seq_lens, s); break;
        }
    } else {
        set_len_kernel<<<(c.B + 127) / 128, 128, 0, s>>>(c.len, c.B, T, seq_lens);
    }
    return cudaGetLastError();
}

}  // namespace kivi
