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
#include <algorithm>

#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

constexpr int kEncodeThreads = 256;

__device__ __forceinline__ int log2_pow2(int x) { return __ffs(x) - 1; }

// Keys.  One lane = 16 tokens x 8 channels of a (b, h, G-token group) tile;
// the G/16 lanes of a tile column are adjacent.  A CTA covers 256 / (S*NC)
// groups of one slice.  Tiles past Tq copy their tokens into the ring.
template <int BITS, int S>
__global__ void __launch_bounds__(kEncodeThreads)
quant_keys_kernel(kivi_cache c, const uint16_t* __restrict__ K, int T,
                  const int32_t* __restrict__ seq_lens)
{
    const int D = c.D;
    constexpr int lgS = S == 2 ? 1 : S == 4 ? 2 : 3;
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
        const int n = seq_lens ? min(max(ld_checked(seq_lens + b), 0), T) : T;
        if (blockIdx.x == 0 && threadIdx.x == 0 && bh % c.H == 0)
            st_checked(c.len + b, n);
        if (g * c.G >= n)
            continue;  // uniform over the tile column
        const int Tq = quantized_tokens(n, c.G, c.R);
        const uint16_t* src = K + (size_t)bh * T * D + j * kLaneChans;
        if ((g + 1) * c.G <= Tq) {
            uint4 raw[kLaneTokens];
#pragma unroll
            for (int i = 0; i < kLaneTokens; ++i)
                raw[i] = ld_stream(src + (size_t)(t0 + i) * D);
            quant_store_key_lane<BITS, S>(c, bh, t0, g, j, s, smask, raw, src + (size_t)t0 * D, D);
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

// Keys, staged.  A persistent CTA of 128 threads walks token tiles of
// 128 * 128 / D tokens (32 KB of fp16 K): while it encodes one tile from
// shared memory, the cp.async copies of its next tile fill the other buffer,
// so the loads stay in flight without holding registers.  Lane layout and
// arithmetic are those of quant_keys_kernel (16 tokens x 8 channels per
// lane, the G/16 lanes of a group column adjacent).  In shared memory the
// 16-byte chunk x of row r sits at x ^ (s * 8/S), s = (r mod G) / 16, so that
// the eight lanes of an LDS.128 phase read eight different bank groups.
constexpr int kKeyStageThreads = 128;
constexpr int kKeyStageBytes = 32 * 1024;

__device__ __forceinline__ int key_stage_swz(int r, int x, int lgS)
{
    return x ^ (((r >> 4) & ((1 << lgS) - 1)) << (3 - lgS));
}

// Encode one key lane (16 tokens x 8 channels) whose rows are staged in
// shared memory at lrow[i * stride], i = 0..15: statistics as in
// quant_key_lane, then the codes, fully unrolled over the P tokens of a word
// (constant shifts), each word-row stored (after its near-tie fix-up) as soon
// as it is complete.
template <int BITS, int S, int D>
__device__ __forceinline__ void quant_store_key_lane_smem(const kivi_cache& c, size_t bh, int t0, int g,
                                                          int j, int s, unsigned smask, const uint4* lrow)
{
    using Cd = Codec<BITS>;
    constexpr int stride = D / kLaneChans;  // 16-byte chunks per staged row
    __half2 mn[4], mx[4];
    {
        const uint4 r0 = lrow[0];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            mn[k] = mx[k] = as_h2(u4_word(r0, k));
    }
#pragma unroll
    for (int i = 1; i < kLaneTokens; ++i) {
        const uint4 r = lrow[i * stride];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __half2 v = as_h2(u4_word(r, k));
            mn[k] = __hmin2(mn[k], v);
            mx[k] = __hmax2(mx[k], v);
        }
    }
#pragma unroll
    for (int m = 1; m < S; m <<= 1)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            mn[k] = __hmin2(mn[k], as_h2(__shfl_xor_sync(smask, h2_bits(mn[k]), m)));
            mx[k] = __hmax2(mx[k], as_h2(__shfl_xor_sync(smask, h2_bits(mx[k]), m)));
        }
    float scale[8], zero[8], inv[8], nzero[8];
    key_lane_stats<BITS, S>(mn, mx, smask, scale, zero, inv);
    InvBracket ib[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        nzero[k] = -zero[k];
        ib[k] = inv_bracket(inv[k]);
    }
    if (s == 0) {
        const size_t so = (bh * (size_t)(c.Tmax / c.G) + g) * D + (size_t)j * kLaneChans;
        float4* sp = reinterpret_cast<float4*>(c.kscale + so);
        float4* zp = reinterpret_cast<float4*>(c.kzero + so);
        st_checked(sp, make_float4(scale[0], scale[1], scale[2], scale[3]));
        st_checked(sp + 1, make_float4(scale[4], scale[5], scale[6], scale[7]));
        st_checked(zp, make_float4(zero[0], zero[1], zero[2], zero[3]));
        st_checked(zp + 1, make_float4(zero[4], zero[5], zero[6], zero[7]));
    }
    // codes: word = sum_i t_bits_i 2^(b i) - bias * sum_i 2^(b i) (mod 2^32)
    constexpr uint32_t kWordBias = kCodeBias * (uint32_t)(((1ull << (Cd::P * BITS)) - 1) /
                                                          ((1ull << BITS) - 1));
    int32_t* dst = c.kq + (bh * (size_t)(c.Tmax / Cd::P) + t0 / Cd::P) * D + (size_t)j * kLaneChans;
#pragma unroll 1
    for (int w = 0; w < Cd::kWordRows; ++w) {
        uint32_t words[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            words[k] = 0u - kWordBias;
        unsigned flagged = 0u;
#pragma unroll
        for (int i = 0; i < Cd::P; ++i) {
            const uint4 r = lrow[(w * Cd::P + i) * stride];
            uint32_t diff = 0u;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float a = add_h_f(u4_half(r, k), nzero[k]);
                words[k] += bracket_code_bits_lop3(a, ib[k], diff) * (1u << (i * BITS));
            }
            flagged |= (diff != 0u ? 1u : 0u) << i;
        }
        if (__builtin_expect(flagged != 0u, 0)) {
#pragma unroll 1
            while (flagged) {
                const int i = __ffs(flagged) - 1;
                flagged &= flagged - 1;
                const uint4 r = lrow[(w * Cd::P + i) * stride];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float a = add_h_f(u4_half(r, k), nzero[k]);
                    uint32_t d1 = 0u;
                    const uint32_t fast = bracket_code_bits(a, ib[k], d1) - kCodeBias;
                    if (d1 != 0u)
                        words[k] += (exact_code(a, scale[k]) - fast) << (i * BITS);
                }
            }
        }
        st_stream(dst + (size_t)w * D, make_uint4(words[0], words[1], words[2], words[3]));
        st_stream(dst + (size_t)w * D + 4, make_uint4(words[4], words[5], words[6], words[7]));
    }
}

template <int BITS, int S, int D>
__global__ void __launch_bounds__(kKeyStageThreads, 3)
quant_keys_staged_kernel(kivi_cache c, const uint16_t* __restrict__ K, int T,
                         const int32_t* __restrict__ seq_lens, int tiles_per_seq)
{
    extern __shared__ __align__(16) uint4 kst[];  // two buffers of kKeyStageBytes
    constexpr int lgS = S == 2 ? 1 : S == 4 ? 2 : 3;
    constexpr int NC = D / kLaneChans, lgNC = NC == 8 ? 3 : NC == 16 ? 4 : 5;
    constexpr int TT = (kKeyStageBytes / 2) / D;   // tokens per tile
    const int lane = threadIdx.x & 31;
    const unsigned smask = (((1u << S) - 1u) << (lane & ~(S - 1)));
    const int s = threadIdx.x & (S - 1);
    const int j = (threadIdx.x >> lgS) & (NC - 1);
    const int gl = threadIdx.x >> (lgS + lgNC);   // group within the tile
    const int RG = c.R + c.G;
    const int ntiles = c.B * c.H * tiles_per_seq;
    constexpr int cpr = NC;                        // 16-byte chunks per row
    constexpr int rsweep = kKeyStageThreads / cpr; // rows per copy sweep
    const int cx = threadIdx.x & (cpr - 1), cr = threadIdx.x / cpr;

    auto tile_of = [&](int tile, int& bh, int& tt0, int& n) {
        bh = tile / tiles_per_seq;
        tt0 = (tile - bh * tiles_per_seq) * TT;
        const int b = bh / c.H;
        n = seq_lens ? min(max(ld_checked(seq_lens + b), 0), T) : T;
    };
    auto prefetch = [&](int tile, int buf) {
        if (tile < ntiles) {
            int bh, tt0, n;
            tile_of(tile, bh, tt0, n);
            const int rows = min(TT, n - tt0);
            if (rows > 0) {
                const uint16_t* src = K + ((size_t)bh * T + tt0) * D + cx * 8;
                uint4* dst = kst + (size_t)buf * (kKeyStageBytes / 16);
                if (rows == TT) {
                    // a full tile: TT / rsweep copies per thread; row r = cr + rsweep k with
                    // cr < rsweep <= 16, so the swizzle term (r / 16) mod S is a constant per k
                    static_assert(rsweep <= 16 && 16 % rsweep == 0, "row sweep");
#pragma unroll
                    for (int k = 0; k < TT / rsweep; ++k) {
                        constexpr int sh = 3 - lgS;
                        const int v = ((rsweep * k) >> 4) & (S - 1);
                        cp_async16(dst + (cr + rsweep * k) * cpr + (cx ^ (v << sh)),
                                   src + (size_t)(cr + rsweep * k) * D);
                    }
                } else {
                    for (int r = cr; r < rows; r += rsweep)
                        cp_async16(dst + r * cpr + key_stage_swz(r, cx, lgS), src + (size_t)r * D);
                }
            }
        }
        cp_async_commit();
    };

    int tile = blockIdx.x;
    prefetch(tile, 0);
    for (int k = 0; tile < ntiles; ++k, tile += gridDim.x) {
        prefetch(tile + gridDim.x, (k + 1) & 1);
        cp_async_wait_prior();
        __syncthreads();
        int bh, tt0, n;
        tile_of(tile, bh, tt0, n);
        if (tt0 == 0 && threadIdx.x == 0 && bh % c.H == 0)
            st_checked(c.len + bh / c.H, n);
        const int g = tt0 / c.G + gl;
        const int t0 = g * c.G + s * kLaneTokens;
        const int lr = gl * c.G + s * kLaneTokens;  // first tile row of this lane
        if (g * c.G < n) {
            const uint4* buf = kst + (size_t)(k & 1) * (kKeyStageBytes / 16);
            const int Tq = quantized_tokens(n, c.G, c.R);
            // the lane's 16 rows share one swizzled column (r / 16 is fixed)
            const uint4* lrow = buf + lr * cpr + key_stage_swz(lr, j, lgS);
            if ((g + 1) * c.G <= Tq) {
                quant_store_key_lane_smem<BITS, S, D>(c, bh, t0, g, j, s, smask, lrow);
            } else {
                for (int i = 0; i < kLaneTokens; ++i) {
                    const int t = t0 + i;
                    if (t >= Tq && t < n)
                        st_stream(c.kres + ((size_t)bh * RG + t % RG) * D + j * kLaneChans, lrow[i * cpr]);
                }
            }
        }
        __syncthreads();  // the buffer is refilled by the next iteration's prefetch
    }
    cp_async_wait_all();
}

// Values.  One lane = one channel group (G channels) of U token rows, so
// min/max, the division and the packing stay inside the lane.  A CTA covers
// 256 / (D/G) * U rows of one slice.
template <int BITS, int G>
__global__ void __launch_bounds__(kEncodeThreads, G == 128 ? 2 : 3)
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
        const int n = seq_lens ? min(max(ld_checked(seq_lens + b), 0), T) : T;
        if (blockIdx.x == 0 && threadIdx.x == 0 && bh % c.H == 0)
            st_checked(c.len + b, n);
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
        st_checked(len + b, seq_lens ? min(max(ld_checked(seq_lens + b), 0), T) : T);
}

static dim3 encode_grid(const kivi_cache& c, int tiles)
{
    const int bh = c.B * c.H;
    return dim3((unsigned)(tiles > 0 ? tiles : 1), (unsigned)(bh < 65535 ? bh : 65535));
}

template <int BITS, int S, int D>
static void staged_launch(const kivi_cache& c, const uint16_t* K, int T, const int32_t* seq_lens, cudaStream_t s)
{
    constexpr int TT = (kKeyStageBytes / 2) / D;
    const int tiles_per_seq = (T + TT - 1) / TT;
    const long ntiles = (long)c.B * c.H * tiles_per_seq;
    const int grid = (int)std::min<long>(ntiles, (long)sm_count() * 3);
    const size_t smem = 2 * kKeyStageBytes;
    cudaFuncSetAttribute(quant_keys_staged_kernel<BITS, S, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    quant_keys_staged_kernel<BITS, S, D><<<grid, kKeyStageThreads, smem, s>>>(c, K, T, seq_lens, tiles_per_seq);
}

template <int BITS, int S>
static void key_launch(const kivi_cache& c, const uint16_t* K, int T, const int32_t* seq_lens, cudaStream_t s)
{
    // staged when a group column takes at most 128 lanes: S * D / 8 <= 128
    if (c.D == 64) {
        staged_launch<BITS, S, 64>(c, K, T, seq_lens, s);
    } else if (c.D == 128 && S <= 8) {
        staged_launch<BITS, S, 128>(c, K, T, seq_lens, s);
    } else if constexpr (S <= 4) {
        staged_launch<BITS, S, 256>(c, K, T, seq_lens, s);
    } else {
        const int lanes_per_group = S * (c.D / kLaneChans);
        const int groups_per_cta = kEncodeThreads / lanes_per_group;
        const int groups = (T + c.G - 1) / c.G;
        const dim3 grid = encode_grid(c, (groups + groups_per_cta - 1) / groups_per_cta);
        quant_keys_kernel<BITS, S><<<grid, kEncodeThreads, 0, s>>>(c, K, T, seq_lens);
    }
}

template <int BITS>
static void key_launch_bits(const kivi_cache& c, const uint16_t* K, int T, const int32_t* seq_lens,
                            cudaStream_t s)
{
    switch (c.G / kLaneTokens) {  // S lanes per group column
    case 2: key_launch<BITS, 2>(c, K, T, seq_lens, s); break;
    case 4: key_launch<BITS, 4>(c, K, T, seq_lens, s); break;
    default: key_launch<BITS, 8>(c, K, T, seq_lens, s); break;
    }
}

cudaError_t launch_quant_keys(const kivi_cache& c, const uint16_t* K, int T,
                              const int32_t* seq_lens, cudaStream_t s)
{
    KIVI_SET_CHECK_RANGES(c, s, {{K, (size_t)c.B * c.H * T * c.D * 2}, {seq_lens, (size_t)c.B * 4}});
    if (T > 0) {
        switch (c.bits_k) {
        case 2: key_launch_bits<2>(c, K, T, seq_lens, s); break;
        case 4: key_launch_bits<4>(c, K, T, seq_lens, s); break;
        default: key_launch_bits<8>(c, K, T, seq_lens, s); break;
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
    KIVI_SET_CHECK_RANGES(c, s, {{V, (size_t)c.B * c.H * T * c.D * 2}, {seq_lens, (size_t)c.B * 4}});
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

#ifdef KIVI_CHECKS
int32_t check_word_quant() { return take_check_word(); }
#endif

}  // namespace kivi
