// kivi_device.cuh -- device-side building blocks shared by the libkivi kernels.
//
// Method: KIVI grouped asymmetric quantization (CacheForge README, "How it
// works"; CacheSeek PR #4 change notes: grouped statistics, int32 packing).
// Arithmetic contract (include/kivi.h):
//   scale = (max - min) / M, zero = min, code = clamp(rne((x - zero)/scale), 0, M)
// in fp32 with IEEE division; x_hat = fp16_rne(fmaf(code, scale, zero)).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "kivi.h"

namespace kivi {

// Tokens one lane covers in a key tile (one int2 word; two int4 / four int8).
constexpr int kLaneTokens = 16;
// Channels one lane covers in an encode / materialize tile (one 16-byte vector).
constexpr int kLaneChans = 8;

template <int BITS>
struct Codec {
    static constexpr int P = 32 / BITS;               // codes per int32 word
    static constexpr uint32_t M = (1u << BITS) - 1u;  // largest code
    static constexpr int kWordRows = kLaneTokens / P; // key word-rows per lane tile
};

__host__ __device__ __forceinline__ int quantized_tokens(int T, int G, int R)
{
    const int n = T - R;
    return n <= 0 ? 0 : (n / G) * G;
}

// ---------------------------------------------------------------- loads ---

__device__ __forceinline__ uint4 ld_stream(const void* p)   // read-once data
{
    return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint4 ld_nc(const void* p)       // read-only, may be shared
{
    return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ float4 ld_nc_f4(const float* p)
{
    return __ldg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void st_stream(void* p, uint4 v)
{
    __stcs(reinterpret_cast<uint4*>(p), v);
}

__device__ __forceinline__ uint16_t u4_half(const uint4& v, int k)   // k in [0, 8)
{
    const uint32_t w = k < 4 ? (k < 2 ? v.x : v.y) : (k < 6 ? v.z : v.w);
    return (uint16_t)((k & 1) ? (w >> 16) : (w & 0xffffu));
}
__device__ __forceinline__ uint32_t u4_word(const uint4& v, int i)   // i in [0, 4)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
__device__ __forceinline__ __half2 as_h2(uint32_t u)
{
    __half2 h;
    memcpy(&h, &u, 4);
    return h;
}
__device__ __forceinline__ uint32_t h2_bits(__half2 h)
{
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
}

// ------------------------------------------------------------ arithmetic ---

// (float)x_f16 + c with a single rounding: the fp32 subtraction x - zero when
// c = -zero (the conversion of x is exact).
__device__ __forceinline__ float add_h_f(uint16_t xh, float c)
{
    float r;
    asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(r) : "h"(xh), "f"(c));
    return r;
}

// Group statistics from canonical fp32 min / max.
template <int BITS>
__device__ __forceinline__ void group_stats(float mn, float mx, float& scale,
                                            float& zero, float& inv)
{
    zero = __fadd_rn(mn, 0.0f);  // -0 -> +0
    mx = __fadd_rn(mx, 0.0f);
    scale = __fdiv_rn(__fsub_rn(mx, zero), (float)Codec<BITS>::M);
    inv = scale != 0.0f ? __frcp_rn(scale) : 0.0f;
}

// code = clamp(rne(a / scale), 0, M) for a = x - zero >= 0, bit-identical to
// rounding the IEEE quotient.  Fast path: q0 = a * rn(1/scale).  For
// y = a/scale <= M(1 + 2^-23) < 256, |q0 - y| <= 2.0001 * 2^-24 * y and
// |rn(y) - y| <= 2^-24 * y, so |q0 - rn(y)| < 2^-14.  Unless q0 lies within
// 2^-12 of a half-integer, q0 and rn(y) sit strictly on the same side of
// every rounding boundary and round to the same integer; otherwise the IEEE
// quotient is formed and rounded.  scale == 0 gives inv == 0, q0 == 0, code 0.
template <int BITS>
__device__ __forceinline__ uint32_t quant_code(float a, float scale, float inv)
{
    const float q0 = __fmul_rn(a, inv);
    const float t = __fadd_rn(q0, 12582912.0f);  // 1.5 * 2^23: ulp 1, RNE
    const float r = __fsub_rn(t, 12582912.0f);
    const float d = __fsub_rn(q0, r);            // exact, in [-0.5, 0.5]
    uint32_t c = __float_as_uint(t) - 0x4B400000u;
    if (fabsf(d) >= 0.5f - 0x1p-12f)
        c = (uint32_t)__float2int_rn(__fdiv_rn(a, scale));
    return min(c, Codec<BITS>::M);
}

__device__ __forceinline__ uint16_t dequant_h(uint32_t code, float scale, float zero)
{
    return __half_as_ushort(__float2half_rn(__fmaf_rn((float)code, scale, zero)));
}

// ------------------------------------------------------ lane quantizers ---

// Key tile lane: 16 consecutive tokens x 8 channels (raw[i] = token i).
// The S = G/16 lanes holding the same group's channels are adjacent and
// aligned in the warp; `mask` names exactly them.  Produces the group's
// per-channel scale/zero (identical on all S lanes) and this lane's packed
// words: words[w][k] = word-row w (of Codec::kWordRows), channel k.
template <int BITS>
__device__ __forceinline__ void quant_key_lane(const uint4 (&raw)[kLaneTokens], int S,
                                               unsigned mask, float (&scale)[8],
                                               float (&zero)[8],
                                               uint32_t (&words)[Codec<BITS>::kWordRows][8])
{
    using Cd = Codec<BITS>;
    __half2 mn[4], mx[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        mn[c] = mx[c] = as_h2(u4_word(raw[0], c));
#pragma unroll
    for (int i = 1; i < kLaneTokens; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const __half2 v = as_h2(u4_word(raw[i], c));
            mn[c] = __hmin2(mn[c], v);
            mx[c] = __hmax2(mx[c], v);
        }
    for (int m = 1; m < S; m <<= 1)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            mn[c] = __hmin2(mn[c], as_h2(__shfl_xor_sync(mask, h2_bits(mn[c]), m)));
            mx[c] = __hmax2(mx[c], as_h2(__shfl_xor_sync(mask, h2_bits(mx[c]), m)));
        }
    // Every lane of the tile column now holds the same min / max.  The S lanes
    // split the eight divisions (lane s takes channels k with k % S == s) and
    // exchange the results.
    float inv[8], nzero[8];
    const int s_lane = (int)(threadIdx.x & 31) & (S - 1);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float lo = (k & 1) ? __high2float(mn[k >> 1]) : __low2float(mn[k >> 1]);
        const float hi = (k & 1) ? __high2float(mx[k >> 1]) : __low2float(mx[k >> 1]);
        zero[k] = __fadd_rn(lo, 0.0f);
        nzero[k] = -zero[k];
        scale[k] = 0.0f;
        inv[k] = 0.0f;
        if ((k & (S - 1)) == s_lane)  // S is a power of two <= 8
            group_stats<BITS>(lo, hi, scale[k], zero[k], inv[k]);
    }
    if (S > 1) {
        const int base = (int)(threadIdx.x & 31) & ~(S - 1);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int src = base + (k & (S - 1));
            scale[k] = __shfl_sync(mask, scale[k], src);
            inv[k] = __shfl_sync(mask, inv[k], src);
        }
    }
#pragma unroll
    for (int w = 0; w < Cd::kWordRows; ++w)
#pragma unroll
        for (int k = 0; k < 8; ++k)
            words[w][k] = 0u;
#pragma unroll
    for (int i = 0; i < kLaneTokens; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float a = add_h_f(u4_half(raw[i], k), nzero[k]);
            const uint32_t code = quant_code<BITS>(a, scale[k], inv[k]);
            words[i / Cd::P][k] |= code << ((i % Cd::P) * BITS);
        }
}

// Value group lane: one token's G consecutive channels (raw[i] = channels
// 8i..8i+7), reduced and coded by a single lane -- no shuffles.  words[w]
// holds channels w*P .. w*P+P-1 of the group.
template <int BITS, int G>
__device__ __forceinline__ void quant_value_group(const uint4 (&raw)[G / 8], float& scale,
                                                  float& zero,
                                                  uint32_t (&words)[G * BITS / 32])
{
    using Cd = Codec<BITS>;
    __half2 mn = as_h2(raw[0].x), mx = mn;
#pragma unroll
    for (int i = 0; i < G / 8; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (i == 0 && c == 0)
                continue;
            const __half2 v = as_h2(u4_word(raw[i], c));
            mn = __hmin2(mn, v);
            mx = __hmax2(mx, v);
        }
    const float lo = fminf(__low2float(mn), __high2float(mn));
    const float hi = fmaxf(__low2float(mx), __high2float(mx));
    float inv;
    group_stats<BITS>(lo, hi, scale, zero, inv);
    const float nz = -zero;
#pragma unroll
    for (int w = 0; w < G * BITS / 32; ++w)
        words[w] = 0u;
#pragma unroll
    for (int e = 0; e < G; ++e) {
        const uint32_t code = quant_code<BITS>(add_h_f(u4_half(raw[e / 8], e % 8), nz), scale, inv);
        words[e / Cd::P] |= code << ((e % Cd::P) * BITS);
    }
}

// --------------------------------------------------------- tile stores ---

// Quantize one key tile lane (16 tokens from t0, channels 8j..8j+7, raw rows
// loaded by the caller) of slice bh, group g, and store its words and -- on
// the first lane of the tile column (s == 0) -- the group statistics.  The S
// lanes of the tile column (`smask`) must call this together.
template <int BITS>
__device__ __forceinline__ void quant_store_key_lane(const kivi_cache& c, size_t bh, int t0,
                                                     int g, int j, int s, int S, unsigned smask,
                                                     const uint4 (&raw)[kLaneTokens])
{
    using Cd = Codec<BITS>;
    const int D = c.D;
    float scale[8], zero[8];
    uint32_t words[Cd::kWordRows][8];
    quant_key_lane<BITS>(raw, S, smask, scale, zero, words);
    int32_t* dst = c.kq + (bh * (size_t)(c.Tmax / Cd::P) + t0 / Cd::P) * D + (size_t)j * kLaneChans;
#pragma unroll
    for (int w = 0; w < Cd::kWordRows; ++w) {
        st_stream(dst + (size_t)w * D, make_uint4(words[w][0], words[w][1], words[w][2], words[w][3]));
        st_stream(dst + (size_t)w * D + 4, make_uint4(words[w][4], words[w][5], words[w][6], words[w][7]));
    }
    if (s == 0) {
        const size_t so = (bh * (size_t)(c.Tmax / c.G) + g) * D + (size_t)j * kLaneChans;
        float4* sp = reinterpret_cast<float4*>(c.kscale + so);
        float4* zp = reinterpret_cast<float4*>(c.kzero + so);
        sp[0] = make_float4(scale[0], scale[1], scale[2], scale[3]);
        sp[1] = make_float4(scale[4], scale[5], scale[6], scale[7]);
        zp[0] = make_float4(zero[0], zero[1], zero[2], zero[3]);
        zp[1] = make_float4(zero[4], zero[5], zero[6], zero[7]);
    }
}

// Quantize value group gi (channels gi*G .. gi*G+G-1) of token t in slice bh
// from `raw` and store its codes and statistics.
template <int BITS, int G>
__device__ __forceinline__ void quant_store_value_group(const kivi_cache& c, size_t bh, int t,
                                                        int gi, const uint4 (&raw)[G / 8])
{
    using Cd = Codec<BITS>;
    constexpr int NW = G * BITS / 32;  // 2, 4 or 8 words for G = 32
    float scale, zero;
    uint32_t words[NW];
    quant_value_group<BITS, G>(raw, scale, zero, words);
    const size_t row = bh * (size_t)c.Tmax + t;
    uint32_t* dst = reinterpret_cast<uint32_t*>(c.vq) + row * (c.D / Cd::P) + (size_t)gi * NW;
    if constexpr (NW == 2) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(words[0], words[1]);
    } else {
#pragma unroll
        for (int w = 0; w < NW; w += 4)
            *reinterpret_cast<uint4*>(dst + w) = make_uint4(words[w], words[w + 1], words[w + 2], words[w + 3]);
    }
    const size_t so = row * (c.D / G) + gi;
    c.vscale[so] = scale;
    c.vzero[so] = zero;
}

// ------------------------------------------------- fused-dequant windows ---
//
// The decode kernels never materialize x_hat.  A code c is turned into the
// fp32 value f = 1 + c * 2^(pos-23) by masking it into mantissa bits
// [pos, pos+b) of 1.0f (one LOP3 after a shared shift), and the multiplier
// carries 2^(23-pos): mult * f = mult + c.  The constant `mult` is removed
// once per group through the sum of the multipliers.  `pos` is chosen per
// code position so that one shift serves several codes ("windows").

template <int BITS>
struct Window;

// int2: code i of a word at bits [2i, 2i+2); windows at mantissa bits 17/19/21.
template <>
struct Window<2> {
    static constexpr int kCodes = 16;
    __device__ static __forceinline__ int pos(int i)
    {
        constexpr int t[16] = {19, 21, 17, 19, 21, 17, 19, 21, 17, 19, 21, 17, 19, 21, 17, 19};
        return t[i];
    }
    // shift applied to the word before masking code i (positive = left)
    __device__ static __forceinline__ int shift(int i)
    {
        constexpr int t[16] = {19, 19, 13, 13, 13, 7, 7, 7, 1, 1, 1, -5, -5, -5, -11, -11};
        return t[i];
    }
    static constexpr int kNumPos = 3;
    __device__ static __forceinline__ int pos_index(int i) { return (pos(i) - 17) / 2; }   // 0,1,2
    __device__ static __forceinline__ float mult_of_index(int k) { return k == 0 ? 64.0f : k == 1 ? 16.0f : 4.0f; }
};

// int4: code i at bits [4i, 4i+4); windows at mantissa bits 15/19.
template <>
struct Window<4> {
    static constexpr int kCodes = 8;
    __device__ static __forceinline__ int pos(int i)
    {
        constexpr int t[8] = {15, 19, 15, 19, 15, 19, 15, 19};
        return t[i];
    }
    __device__ static __forceinline__ int shift(int i)
    {
        constexpr int t[8] = {15, 15, 7, 7, -1, -1, -9, -9};
        return t[i];
    }
    static constexpr int kNumPos = 2;
    __device__ static __forceinline__ int pos_index(int i) { return i & 1; }   // 15 -> 0, 19 -> 1
    __device__ static __forceinline__ float mult_of_index(int k) { return k == 0 ? 256.0f : 16.0f; }
};

// int8: code i at bits [8i, 8i+8); one window at mantissa bits 15.
template <>
struct Window<8> {
    static constexpr int kCodes = 4;
    __device__ static __forceinline__ int pos(int) { return 15; }
    __device__ static __forceinline__ int shift(int i)
    {
        constexpr int t[4] = {15, 7, -1, -9};
        return t[i];
    }
    static constexpr int kNumPos = 1;
    __device__ static __forceinline__ int pos_index(int) { return 0; }
    __device__ static __forceinline__ float mult_of_index(int) { return 256.0f; }
};

// f(c) for code i of `word`: 1 + c * 2^(pos(i)-23).  All arguments but `word`
// are compile-time constants once the caller's loop over i is unrolled.
template <int BITS>
__device__ __forceinline__ float window_value(uint32_t word, int i)
{
    const int sh = Window<BITS>::shift(i);
    const uint32_t s = sh >= 0 ? (word << sh) : (word >> (-sh));
    const uint32_t m = ((1u << BITS) - 1u) << Window<BITS>::pos(i);
    return __uint_as_float((s & m) | 0x3F800000u);
}

}  // namespace kivi
