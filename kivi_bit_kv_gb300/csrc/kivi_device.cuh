// kivi_device.cuh -- device-side building blocks shared by the libkivi kernels.
//
// Method: KIVI grouped asymmetric quantization (CacheForge README, "How it
// works"; CacheSeek PR #4 change notes: grouped statistics, int32 packing).
// Arithmetic contract (include/kivi.h):
//   scale = (max - min) / M, zero = min, code = clamp(rne((x - zero)/scale), 0, M)
// in fp32 with IEEE division; x_hat = fp16_rne(fmaf(code, scale, zero)).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kivi.h"
#include "kivi_divm.h"

namespace kivi {

// ---------------------------------------------------------- checked build ---
// With KIVI_CHECKS defined, every global access of the encode, materialize,
// append, payload and split-decode kernels goes through KIVI_IN_RANGE: the
// bytes [p, p + n) must lie in one of the ranges the launcher wrote into this
// translation unit's table (the cache's arrays and the call's own buffers).
// A failed check records KIVI_ECHECK in this unit's check word (the first
// failure wins) and the access is skipped; kivi_check_status() reads and
// clears the words of every unit.  Without KIVI_CHECKS the checks compile
// away.
#ifdef KIVI_CHECKS
}  // namespace kivi
#include <initializer_list>
namespace kivi {
constexpr int kCheckRanges = 16;
struct CheckRange {
    uintptr_t lo, hi;
};
static __constant__ CheckRange g_check_ranges[kCheckRanges];
static __device__ int g_check_word;

__device__ __forceinline__ bool in_ranges(const void* p, size_t n)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
#pragma unroll 1
    for (int i = 0; i < kCheckRanges; ++i)
        if (a >= g_check_ranges[i].lo && a + n <= g_check_ranges[i].hi)
            return true;
    atomicCAS(&g_check_word, KIVI_OK, KIVI_ECHECK);
    return false;
}
#define KIVI_IN_RANGE(p, n) ::kivi::in_ranges((p), (n))

// Writes the table of this translation unit: the arrays of cache c (their
// sizes from kivi_buffer_bytes) and up to six buffers of the call.
struct CallBuf {
    const void* p;
    size_t bytes;
};
static inline cudaError_t set_check_ranges(const kivi_cache& c, cudaStream_t s,
                                           std::initializer_list<CallBuf> call = {})
{
    CheckRange r[kCheckRanges] = {};
    int n = 0;
    const void* arrays[9] = {c.kq, c.kscale, c.kzero, c.vq, c.vscale, c.vzero, c.kres, c.vres, c.len};
    for (int i = 0; i < 9; ++i) {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(arrays[i]);
        r[n++] = CheckRange{lo, lo + kivi_buffer_bytes(&c, i)};
    }
    for (const CallBuf& b : call)
        if (b.p && n < kCheckRanges) {
            const uintptr_t lo = reinterpret_cast<uintptr_t>(b.p);
            r[n++] = CheckRange{lo, lo + b.bytes};
        }
    return cudaMemcpyToSymbolAsync(g_check_ranges, r, sizeof r, 0, cudaMemcpyHostToDevice, s);
}
// Reads and clears this translation unit's check word (synchronizes).
static inline int32_t take_check_word()
{
    int32_t v = KIVI_OK;
    const int32_t zero = KIVI_OK;
    if (cudaMemcpyFromSymbol(&v, g_check_word, sizeof v) != cudaSuccess ||
        cudaMemcpyToSymbol(g_check_word, &zero, sizeof zero) != cudaSuccess)
        return KIVI_ECUDA;
    return v;
}
#define KIVI_SET_CHECK_RANGES(c, s, ...)                                      \
    do {                                                                      \
        const cudaError_t e_ = ::kivi::set_check_ranges((c), (s), __VA_ARGS__); \
        if (e_ != cudaSuccess)                                                \
            return e_;                                                        \
    } while (0)
#else
#define KIVI_IN_RANGE(p, n) true
#define KIVI_SET_CHECK_RANGES(c, s, ...) \
    do {                                 \
    } while (0)
#endif

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

// ------------------------------------------------------------- cp.async ---
// 16-byte asynchronous global -> shared copies (cached in L2 only).  A thread
// waits for its own groups with cp.async.wait_group -- a hardware wait, no
// spinning -- and a warp barrier then publishes them to the warp.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem)
{
    if (!KIVI_IN_RANGE(gmem, 16)) {
        *reinterpret_cast<uint4*>(smem) = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
// all but the most recent group
__device__ __forceinline__ void cp_async_wait_prior() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

// ---------------------------------------------------------------- loads ---

__device__ __forceinline__ uint4 ld_stream(const void* p)   // read-once data
{
    if (!KIVI_IN_RANGE(p, 16))
        return make_uint4(0u, 0u, 0u, 0u);
    return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint4 ld_nc(const void* p)       // read-only, may be shared
{
    if (!KIVI_IN_RANGE(p, 16))
        return make_uint4(0u, 0u, 0u, 0u);
    return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ float4 ld_nc_f4(const float* p)
{
    if (!KIVI_IN_RANGE(p, 16))
        return make_float4(0.f, 0.f, 0.f, 0.f);
    return __ldg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void st_stream(void* p, uint4 v)
{
    if (KIVI_IN_RANGE(p, 16))
        __stcs(reinterpret_cast<uint4*>(p), v);
}
// A global store of one value, bounds-checked in the checked build.
template <class T>
__device__ __forceinline__ void st_checked(T* p, T v)
{
    if (KIVI_IN_RANGE(p, sizeof(T)))
        *p = v;
}
// A global load of one value (zero where a check fails).
template <class T>
__device__ __forceinline__ T ld_checked(const T* p)
{
    return KIVI_IN_RANGE(p, sizeof(T)) ? *p : T{};
}
// The same through the read-only path (data no kernel of the call writes).
template <class T>
__device__ __forceinline__ T ldg_checked(const T* p)
{
    return KIVI_IN_RANGE(p, sizeof(T)) ? __ldg(p) : T{};
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

// RN(x / M) for a group range x (kivi_divm.h): one FMUL and one FFMA.  An
// infinite range (non-finite input) keeps the IEEE quotient, infinity.
template <int BITS>
__device__ __forceinline__ float div_code_range(float x)
{
    const float q = __fmaf_rn(x, DivM<BITS>::hi, __fmul_rn(x, DivM<BITS>::lo));
    return isinf(x) ? x : q;
}

// Group statistics from canonical fp32 min / max.
template <int BITS>
__device__ __forceinline__ void group_stats(float mn, float mx, float& scale,
                                            float& zero, float& inv)
{
    zero = __fadd_rn(mn, 0.0f);  // -0 -> +0
    mx = __fadd_rn(mx, 0.0f);
    scale = div_code_range<BITS>(__fsub_rn(mx, zero));
    inv = scale != 0.0f ? __frcp_rn(scale) : 0.0f;
}

// Scales, zeros and reciprocals of the eight channels of a key lane from the
// min / max its tile column shares (mn, mx: channel pairs).  Lane s of the
// column's S lanes computes channels k = S kk + s, 8/S of them with the same
// instructions on every lane, and the lanes exchange the results.
template <int BITS, int S>
__device__ __forceinline__ void key_lane_stats(const __half2 (&mn)[4], const __half2 (&mx)[4], unsigned mask,
                                               float (&scale)[8], float (&zero)[8], float (&inv)[8])
{
    const int lane = (int)(threadIdx.x & 31), s = lane & (S - 1), base = lane & ~(S - 1);
#pragma unroll
    for (int k = 0; k < 8; ++k)
        zero[k] = __fadd_rn((k & 1) ? __high2float(mn[k >> 1]) : __low2float(mn[k >> 1]), 0.0f);
    constexpr int NK = 8 / S;
    float sc[NK], iv[NK];
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
        // channel k = S kk + s: pair (S kk) / 2 + s / 2, half s & 1 (S is even)
        const int w = (S * kk) / 2 + (s >> 1);
        __half2 a = mn[0], b = mx[0];
#pragma unroll
        for (int w2 = 1; w2 < 4; ++w2)
            if (w == w2) {
                a = mn[w2];
                b = mx[w2];
            }
        const float lo = (s & 1) ? __high2float(a) : __low2float(a);
        const float hi = (s & 1) ? __high2float(b) : __low2float(b);
        float z;
        group_stats<BITS>(lo, hi, sc[kk], z, iv[kk]);
    }
#pragma unroll
    for (int kk = 0; kk < NK; ++kk)
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) {
            scale[S * kk + s2] = __shfl_sync(mask, sc[kk], base + s2);
            inv[S * kk + s2] = __shfl_sync(mask, iv[kk], base + s2);
        }
}

// Exact code: round-half-even of the IEEE quotient a / scale (scale > 0).
// Kept out of line: it runs only for quotients near a rounding boundary.
static __device__ __noinline__ uint32_t exact_code(float a, float scale)
{
    return (uint32_t)__float2int_rn(__fdiv_rn(a, scale));
}

// Code of a = x - zero >= 0 with its own exactness test, without a division.
// With inv = rn(1/scale), the bracket inv_lo = rn(inv (1 - 2^-21)) and
// inv_hi = rn(inv (1 + 2^-21)) satisfies
//   inv_lo <= (1/scale)(1 - 2^-24),   inv_hi >= (1/scale)(1 + 2^-24)
// (inv is within 2^-24 of 1/scale, each product rounding within 2^-24 more),
// and the IEEE quotient q = rn(a / scale) is within 2^-24 of a / scale, so,
// as a >= 0,
//   a inv_lo <= q <= a inv_hi.
// t_lo = rn(a inv_lo + C) and t_hi = rn(a inv_hi + C), C = 1.5 * 2^23 (ulp 1,
// even): each FFMA rounds the exact product to the nearest integer, ties to
// even, and that rounding is monotone, so t_lo == t_hi means every value in
// [a inv_lo, a inv_hi] -- q included -- rounds to the same integer: the code
// is t_lo - C.  Otherwise (a half-integer inside the bracket: about 2^(b-20)
// of the codes) the caller takes exact_code().  No code exceeds M:
// a inv_lo <= q <= M (1 + 2^-23).  scale == 0 gives inv == 0, both brackets 0
// and code 0.  Returns the bits of t_lo; `diff` collects t_lo ^ t_hi.
struct InvBracket {
    float lo, hi;
};
__device__ __forceinline__ InvBracket inv_bracket(float inv)
{
    return {__fmul_rn(inv, 1.0f - 0x1p-21f), __fmul_rn(inv, 1.0f + 0x1p-21f)};
}
// bracket_code_bits with the collection pinned to one 3-input LOP3 (the
// compiler otherwise turns the OR of XORs into compare-and-select chains).
__device__ __forceinline__ uint32_t bracket_code_bits_lop3(float a, InvBracket ib, uint32_t& diff)
{
    const uint32_t tl = __float_as_uint(__fmaf_rn(a, ib.lo, 12582912.0f));
    const uint32_t th = __float_as_uint(__fmaf_rn(a, ib.hi, 12582912.0f));
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xBE;" : "=r"(d) : "r"(tl), "r"(th), "r"(diff));  // (tl ^ th) | diff
    diff = d;
    return tl;
}
__device__ __forceinline__ uint32_t bracket_code_bits(float a, InvBracket ib, uint32_t& diff)
{
    const uint32_t tl = __float_as_uint(__fmaf_rn(a, ib.lo, 12582912.0f));
    const uint32_t th = __float_as_uint(__fmaf_rn(a, ib.hi, 12582912.0f));
    diff |= tl ^ th;
    return tl;
}
constexpr uint32_t kCodeBias = 0x4B400000u;

// 2^23 as an opaque register value: keeps the operand of the per-code LOP3 in
// a register instead of being rematerialized per use.
__device__ __forceinline__ uint32_t two23_bits()
{
    uint32_t v = 0x4B000000u;
    asm volatile("" : "+r"(v));
    return v;
}

// (float)((word >> sh) & M) without a conversion instruction: one LOP3 places
// the code in the mantissa of 2^23, one exact subtraction removes 2^23.
__device__ __forceinline__ float code_float(uint32_t shifted, uint32_t mask, uint32_t two23)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(shifted), "r"(mask), "r"(two23));
    return __fsub_rn(__uint_as_float(r), 8388608.0f);
}

// Two dequantized values fp16_rne(fmaf(code, scale, zero)) packed as half2
// bits (first in the low half); f0, f1 are the codes as floats.
__device__ __forceinline__ uint32_t dequant_h2(float f0, float f1, float s0, float z0, float s1,
                                               float z1)
{
    const __half2 h = __floats2half2_rn(__fmaf_rn(f0, s0, z0), __fmaf_rn(f1, s1, z1));
    return h2_bits(h);
}

// ------------------------------------------------------ lane quantizers ---

// Key tile lane: 16 consecutive tokens x 8 channels (raw[i] = token i).
// The S = G/16 lanes holding the same group's channels are adjacent and
// aligned in the warp; `mask` names exactly them.  Produces the group's
// per-channel scale/zero (identical on all S lanes) and this lane's packed
// words: words[w][k] = word-row w (of Codec::kWordRows), channel k.
template <int BITS, int S>
__device__ __forceinline__ void quant_key_lane(const uint4 (&raw)[kLaneTokens],
                                               unsigned mask, float (&scale)[8],
                                               float (&zero)[8], float (&inv)[8],
                                               uint32_t (&words)[Codec<BITS>::kWordRows][8],
                                               unsigned& flagged)
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
#pragma unroll
    for (int m = 1; m < S; m <<= 1)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            mn[c] = __hmin2(mn[c], as_h2(__shfl_xor_sync(mask, h2_bits(mn[c]), m)));
            mx[c] = __hmax2(mx[c], as_h2(__shfl_xor_sync(mask, h2_bits(mx[c]), m)));
        }
    // every lane of the tile column now holds the same min / max
    key_lane_stats<BITS, S>(mn, mx, mask, scale, zero, inv);
    float nzero[8];
    InvBracket ib[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        nzero[k] = -zero[k];
        ib[k] = inv_bracket(inv[k]);
    }
    // Pack t_bits * 2^sh (IMAD) and remove the constant bias once per word:
    // sum_i (bias + c_i) 2^(b i) - bias * sum_i 2^(b i) = sum_i c_i 2^(b i) (mod 2^32).
    constexpr uint32_t kWordBias = kCodeBias * (uint32_t)(((1ull << (Cd::P * BITS)) - 1) /
                                                          ((1ull << BITS) - 1));
#pragma unroll
    for (int w = 0; w < Cd::kWordRows; ++w)
#pragma unroll
        for (int k = 0; k < 8; ++k)
            words[w][k] = 0u - kWordBias;
    flagged = 0u;
#pragma unroll
    for (int i = 0; i < kLaneTokens; ++i) {
        uint32_t diff = 0u;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float a = add_h_f(u4_half(raw[i], k), nzero[k]);
            words[i / Cd::P][k] += bracket_code_bits(a, ib[k], diff) * (1u << ((i % Cd::P) * BITS));
        }
        flagged |= (diff != 0u ? 1u : 0u) << i;
    }
}

// Rows of a key lane whose fast codes need the exact quotient (bit i of
// `flagged`), re-read from `row0 + i * stride`: one small loop, kept out of
// the unrolled main body.
template <int BITS>
__device__ __forceinline__ void key_lane_fixup(unsigned flagged, const uint16_t* row0, size_t stride,
                                               const float (&scale)[8], const float (&inv)[8],
                                               const float (&zero)[8],
                                               uint32_t (&words)[Codec<BITS>::kWordRows][8])
{
    using Cd = Codec<BITS>;
#pragma unroll 1
    while (flagged) {
        const int i = __ffs(flagged) - 1;
        flagged &= flagged - 1;
        const uint4 r = *reinterpret_cast<const uint4*>(row0 + (size_t)i * stride);
        const int sh = (i % Cd::P) * BITS;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float a = add_h_f(u4_half(r, k), -zero[k]);
            uint32_t diff = 0u;
            const uint32_t fast = bracket_code_bits(a, inv_bracket(inv[k]), diff) - kCodeBias;
            if (diff != 0u) {
                const uint32_t fix = (exact_code(a, scale[k]) - fast) << sh;
#pragma unroll
                for (int w = 0; w < Cd::kWordRows; ++w)
                    if (w == i / Cd::P)
                        words[w][k] += fix;
            }
        }
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
    const InvBracket ib = inv_bracket(inv);
    constexpr uint32_t kWordBias = kCodeBias * (uint32_t)(((1ull << (Cd::P * BITS)) - 1) /
                                                          ((1ull << BITS) - 1));
#pragma unroll
    for (int w = 0; w < G * BITS / 32; ++w)
        words[w] = 0u - kWordBias;
#pragma unroll
    for (int e0 = 0; e0 < G; e0 += 8) {
        uint32_t diff = 0u;
#pragma unroll
        for (int e = e0; e < e0 + 8; ++e) {
            const uint32_t tb = bracket_code_bits(add_h_f(u4_half(raw[e / 8], e % 8), nz), ib, diff);
            words[e / Cd::P] += tb * (1u << ((e % Cd::P) * BITS));
        }
        if (__builtin_expect(diff != 0u, 0)) {
#pragma unroll
            for (int e = e0; e < e0 + 8; ++e) {
                const float a = add_h_f(u4_half(raw[e / 8], e % 8), nz);
                uint32_t d1 = 0u;
                const uint32_t fast = bracket_code_bits(a, ib, d1) - kCodeBias;
                if (d1 != 0u)
                    words[e / Cd::P] += (exact_code(a, scale) - fast) << ((e % Cd::P) * BITS);
            }
        }
    }
}

// --------------------------------------------------------- tile stores ---

// Quantize one key tile lane (16 tokens from t0, channels 8j..8j+7, raw rows
// loaded by the caller) of slice bh, group g, and store its words and -- on
// the first lane of the tile column (s == 0) -- the group statistics.  The S
// lanes of the tile column (`smask`) must call this together.
template <int BITS, int S>
__device__ __forceinline__ void quant_store_key_lane(const kivi_cache& c, size_t bh, int t0,
                                                     int g, int j, int s, unsigned smask,
                                                     const uint4 (&raw)[kLaneTokens],
                                                     const uint16_t* row0, size_t row_stride)
{
    using Cd = Codec<BITS>;
    const int D = c.D;
    float scale[8], zero[8], inv[8];
    uint32_t words[Cd::kWordRows][8];
    unsigned flagged;
    quant_key_lane<BITS, S>(raw, smask, scale, zero, inv, words, flagged);
    if (__builtin_expect(flagged != 0u, 0))
        key_lane_fixup<BITS>(flagged, row0, row_stride, scale, inv, zero, words);
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
        st_checked(sp, make_float4(scale[0], scale[1], scale[2], scale[3]));
        st_checked(sp + 1, make_float4(scale[4], scale[5], scale[6], scale[7]));
        st_checked(zp, make_float4(zero[0], zero[1], zero[2], zero[3]));
        st_checked(zp + 1, make_float4(zero[4], zero[5], zero[6], zero[7]));
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
        st_checked(reinterpret_cast<uint2*>(dst), make_uint2(words[0], words[1]));
    } else {
#pragma unroll
        for (int w = 0; w < NW; w += 4)
            st_checked(reinterpret_cast<uint4*>(dst + w), make_uint4(words[w], words[w + 1], words[w + 2], words[w + 3]));
    }
    const size_t so = row * (c.D / G) + gi;
    st_checked(c.vscale + so, scale);
    st_checked(c.vzero + so, zero);
}

}  // namespace kivi
