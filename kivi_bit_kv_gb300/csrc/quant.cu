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
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

// One lane = 16 tokens x 8 channels of one (b, h, G-token group) tile; the
// G/16 lanes of a tile column are adjacent, so the per-channel min/max over
// the group's tokens needs log2(G/16) shuffles.  Tiles past Tq copy their
// tokens into the residual ring instead.
template <int BITS>
__global__ void __launch_bounds__(256)
quant_keys_kernel(kivi_cache c, const uint16_t* __restrict__ K, int T,
                  const int32_t* __restrict__ seq_lens, int units_per_bh)
{
    using Cd = Codec<BITS>;
    const int D = c.D;
    const int S = c.G / kLaneTokens;
    const int NC = D / kLaneChans;
    const int lanes_per_unit = S * NC;
    const long long total = (long long)c.B * c.H * units_per_bh * lanes_per_unit;
    const int lane = threadIdx.x & 31;
    const unsigned smask = (((1u << S) - 1u) << (lane & ~(S - 1)));
    const long long stride = (long long)gridDim.x * blockDim.x;

    for (long long task = (long long)blockIdx.x * blockDim.x + threadIdx.x; task < total;
         task += stride) {
        // every condition below is uniform over the S lanes of one tile column
        const int s = (int)(task % S);
        const int j = (int)((task / S) % NC);
        const long long unit = task / lanes_per_unit;
        const int g = (int)(unit % units_per_bh);
        const long long bh = unit / units_per_bh;
        const int b = (int)(bh / c.H);
        const int n = seq_lens ? min(max(seq_lens[b], 0), T) : T;
        if (g == 0 && j == 0 && s == 0 && bh % c.H == 0)
            c.len[b] = n;
        if (g * c.G >= n)
            continue;
        const int Tq = quantized_tokens(n, c.G, c.R);
        const int t0 = g * c.G + s * kLaneTokens;
        const uint16_t* src = K + (size_t)bh * T * D + (size_t)j * kLaneChans;

        if ((g + 1) * c.G <= Tq) {
            uint4 raw[kLaneTokens];
#pragma unroll
            for (int i = 0; i < kLaneTokens; ++i)
                raw[i] = ld_stream(src + (size_t)(t0 + i) * D);
            quant_store_key_lane<BITS>(c, bh, t0, g, j, s, S, smask, raw);
        } else {
            const int RG = c.R + c.G;
            for (int i = 0; i < kLaneTokens; ++i) {
                const int t = t0 + i;
                if (t >= Tq && t < n)
                    st_stream(c.kres + ((size_t)bh * RG + t % RG) * D + (size_t)j * kLaneChans,
                              ld_stream(src + (size_t)t * D));
            }
        }
    }
}

// One lane = 8 channels of one token; the G/8 lanes of a channel group are
// adjacent.  Each thread keeps four rows in flight.
template <int BITS>
__global__ void __launch_bounds__(256)
quant_values_kernel(kivi_cache c, const uint16_t* __restrict__ V, int T,
                    const int32_t* __restrict__ seq_lens)
{
    constexpr int U = 4;
    const int D = c.D;
    const int NC = D / kLaneChans;
    const int LPG = c.G / kLaneChans;
    const long long total = (long long)c.B * c.H * T * NC;
    const int lane = threadIdx.x & 31;
    const unsigned gmask = (((1u << LPG) - 1u) << (lane & ~(LPG - 1)));
    const long long stride = (long long)gridDim.x * blockDim.x;
    const int RG = c.R + c.G;

    for (long long base = (long long)blockIdx.x * blockDim.x + threadIdx.x; base < total;
         base += U * stride) {
        uint4 raw[U];
        int tt[U], nn[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long task = base + u * stride;
            raw[u] = make_uint4(0u, 0u, 0u, 0u);
            tt[u] = -1;
            nn[u] = 0;
            if (task < total) {
                const int j = (int)(task % NC);
                const long long row = task / NC;
                const int t = (int)(row % T);
                const long long bh = row / T;
                const int b = (int)(bh / c.H);
                const int n = seq_lens ? min(max(seq_lens[b], 0), T) : T;
                tt[u] = t;
                nn[u] = n;
                if (t == 0 && j == 0 && bh % c.H == 0)
                    c.len[b] = n;
                if (t < n)
                    raw[u] = ld_stream(V + (size_t)row * D + (size_t)j * kLaneChans);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long task = base + u * stride;
            if (task >= total || tt[u] >= nn[u])
                continue;  // uniform over a channel group (same row)
            const int j = (int)(task % NC);
            const long long row = task / NC;
            const size_t bh = (size_t)(row / T);
            const int t = tt[u];
            const int Tq = quantized_tokens(nn[u], c.G, c.R);
            if (t < Tq)
                store_value_lane<BITS>(c, bh, t, j, raw[u], gmask);
            else
                st_stream(c.vres + (bh * RG + t % RG) * D + (size_t)j * kLaneChans, raw[u]);
        }
    }
}

__global__ void set_len_kernel(int32_t* len, int B, int T, const int32_t* __restrict__ seq_lens)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B)
        len[b] = seq_lens ? min(max(seq_lens[b], 0), T) : T;
}

static int grid_for(long long threads, int block, int per_sm)
{
    const long long want = (threads + block - 1) / block;
    const long long cap = (long long)sm_count() * per_sm;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

cudaError_t launch_quant_keys(const kivi_cache& c, const uint16_t* K, int T,
                              const int32_t* seq_lens, cudaStream_t s)
{
    if (T > 0) {
        const int units = (T + c.G - 1) / c.G;
        const long long threads = (long long)c.B * c.H * units * (c.G / kLaneTokens) *
                                  (c.D / kLaneChans);
        const int grid = grid_for(threads, 256, 16);
        switch (c.bits_k) {
        case 2: quant_keys_kernel<2><<<grid, 256, 0, s>>>(c, K, T, seq_lens, units); break;
        case 4: quant_keys_kernel<4><<<grid, 256, 0, s>>>(c, K, T, seq_lens, units); break;
        default: quant_keys_kernel<8><<<grid, 256, 0, s>>>(c, K, T, seq_lens, units); break;
        }
    } else {
        set_len_kernel<<<(c.B + 127) / 128, 128, 0, s>>>(c.len, c.B, T, seq_lens);
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_values(const kivi_cache& c, const uint16_t* V, int T,
                                const int32_t* seq_lens, cudaStream_t s)
{
    if (T > 0) {
        const long long threads = (long long)c.B * c.H * T * (c.D / kLaneChans);
        const int grid = grid_for((threads + 3) / 4, 256, 16);
        switch (c.bits_v) {
        case 2: quant_values_kernel<2><<<grid, 256, 0, s>>>(c, V, T, seq_lens); break;
        case 4: quant_values_kernel<4><<<grid, 256, 0, s>>>(c, V, T, seq_lens); break;
        default: quant_values_kernel<8><<<grid, 256, 0, s>>>(c, V, T, seq_lens); break;
        }
    } else {
        set_len_kernel<<<(c.B + 127) / 128, 128, 0, s>>>(c.len, c.B, T, seq_lens);
    }
    return cudaGetLastError();
}

}  // namespace kivi
