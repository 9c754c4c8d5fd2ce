// decode_mma.cuh -- building blocks of the decode-attention kernels: q . K_hat^T
// and p . V_hat over the packed KIVI cache on the warp-level tensor cores, with
// dequantization fused into the operand build.
//
// Both products factor the group statistics out of the contraction
// (CacheForge README, "How it works": keys per channel, values per token):
//   keys   s_t = sum_d (q_d s_gd) c_td + sum_d q_d z_gd     (g = group of t)
//   values o_d = sum_t (p_t s_tg) c_td + sum_t p_t z_tg     (g = group of d)
// The first sum is an m16n8k16 MMA whose A operand holds the integer codes
// and whose B operand holds the weights w = q s or p s; the second is a plain
// fp32 dot product per group.
//
// A operand.  Packed words run along the output axis (keys: 32/b tokens of one
// channel; values: 32/b channels of one token), while an A register pairs two
// values along the contraction axis.  One PRMT moves byte y of two words (two
// channels of a key word-row, or two tokens of a value word-column) into bytes
// 0 and 2 of a register; one AND then keeps the code at position m of that
// byte in both halves.  Each half is the fp16 subnormal c * 2^(b m) * 2^-24,
// exact for every code (c 2^(b m) <= 255 < 2^10); the factor 2^(24 - b m) is
// applied to the fp32 accumulator at the end.  No conversion instruction runs
// per code.
//
// B operand.  w is split into two fp16 terms, hi = w with its low 13
// mantissa bits cleared (exact in fp16) and lo = fp16(w - hi), and both MMAs
// accumulate into the same fp32 registers, so the weights carry about 22
// significant bits.  Ranges: p <= 1 and s <= 131008 / 3 keep |p s| < 65504;
// for keys q is pre-scaled per head by a power of two so that max |q| < 1
// (the factor returns exactly in the epilogue).
//
// Warp tile.  The 8 lane groups g of a warp (lanes 4g .. 4g+3) own the 16
// rows of an MMA tile, two rows each; rows g and g+8 of tile j are the code
// positions 2 pi and 2 pi + 1 (pi = v NT + j) of the word-row (keys) or
// word-column (values) the lane group loads.  A tile's N = 8 columns are
// (group, query head) pairs, so one B fragment serves tokens (channels) from
// several statistic groups and several heads of a grouped-query set; each
// output reads the column of its own group.
#pragma once

#include <math.h>

#include "kivi_device.cuh"

namespace kivi {

constexpr int kDecodeThreads = 128;
constexpr int kDecodeWarps = kDecodeThreads / 32;
constexpr int kChunkTokens = 1024;  // tokens per decode CTA (one split-T chunk)

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

// Query heads processed together per KV head: 8, 4, 2 or 1.
__host__ __device__ constexpr int heads_per_pass(int NQ)
{
    return NQ % 8 == 0 ? 8 : NQ % 4 == 0 ? 4 : NQ % 2 == 0 ? 2 : 1;
}

// fp32 q row in shared memory: channel d at qpad(d) (4 floats of padding per
// 16 channels spread the LDS.128 of the four lanes of a lane group over banks).
__host__ __device__ constexpr int qstride_of(int D) { return D + D / 4; }
__device__ __forceinline__ int qpad(int d) { return d + ((d >> 4) << 2); }

// D += A * B, m16n8k16, fp16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// PRMT selector: byte y of the first word to byte 0, byte y of the second to
// byte 2 (bytes 1 and 3 are don't-care; the AND clears them).
__host__ __device__ constexpr uint32_t pair_sel(int y) { return (uint32_t)y | ((uint32_t)(4 + y) << 8); }

template <int BITS>
__device__ __forceinline__ uint32_t code_pair(uint32_t w0, uint32_t w1, uint32_t sel, int m)
{
    const uint32_t hm = ((1u << BITS) - 1u) << (BITS * m);
    return __byte_perm(w0, w1, sel) & (hm | (hm << 16));
}

// fp32 factor that undoes the 2^(b m - 24) of a code at byte position m.
template <int BITS>
__host__ __device__ constexpr float code_unscale(int m) { return (float)(1u << (24 - BITS * m)); }

// w = hi + lo as two fp16 pairs (see the B operand note above).
__device__ __forceinline__ void split_hi_lo(float a, float b, uint32_t& hi, uint32_t& lo)
{
    const float ah = __uint_as_float(__float_as_uint(a) & 0xFFFFE000u);
    const float bh = __uint_as_float(__float_as_uint(b) & 0xFFFFE000u);
    hi = h2_bits(__floats2half2_rn(ah, bh));
    lo = h2_bits(__floats2half2_rn(__fsub_rn(a, ah), __fsub_rn(b, bh)));
}

// Positions of the rows of tile j for sub-lane v (see the warp-tile note).
template <int BITS, int NT>
struct TileRows {
    static constexpr int CPB = 8 / BITS;  // codes per byte
    // byte and in-byte position of rows g (a) and g + 8 (b) of tile j, v = 0
    __host__ __device__ static constexpr int ya(int j) { return (2 * j) / CPB; }
    __host__ __device__ static constexpr int yb(int j) { return (2 * j + 1) / CPB; }
    __host__ __device__ static constexpr int ma(int j) { return (2 * j) % CPB; }
    __host__ __device__ static constexpr int mb(int j) { return (2 * j + 1) % CPB; }
    // selector offset of sub-lane v: its positions start at 2 v NT, a whole
    // number of bytes (2 NT is a multiple of CPB for every shape used)
    __device__ static uint32_t sel_offset(int v) { return (uint32_t)(2 * v * NT / CPB) * 0x101u; }
    static_assert((2 * NT) % CPB == 0, "sub-lane positions must start on a byte");
};

// ------------------------------------------------------------------ keys ---

template <int BITS, int NQB>
struct KeyTile {
    static constexpr int P = 32 / BITS;
    static constexpr int WR = cmin(8, (8 / NQB) * 32 / P);  // word-rows per warp tile
    static constexpr int LPW = 8 / WR;                      // lane groups per word-row
    static constexpr int TOK = WR * P;                      // tokens per warp tile
    static constexpr int NT = TOK / 16;                     // MMA tiles per warp tile
};

// Stages query heads hq0 .. hq0+NQB-1 of sequence b: qs[h][qpad(d)] = q 2^-e_h
// with 2^-e_h the power of two that brings max_d |q| into [1/2, 1), and
// fac[h] = sm_scale 2^e_h.  Called by the whole CTA between barriers.
template <int NQB>
__device__ __forceinline__ void stage_q(const uint16_t* __restrict__ q, int D, float sm_scale,
                                        float* qs, float* fac)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int qstride = qstride_of(D);
    for (int h = warp; h < NQB; h += kDecodeWarps) {
        const uint16_t* row = q + (size_t)h * D;
        float mx = 0.0f;
        for (int d = lane; d < D; d += 32)
            mx = fmaxf(mx, fabsf(__half2float(__ushort_as_half(row[d]))));
        for (int m = 16; m > 0; m >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
        float inv = 1.0f, f = 1.0f;
        if (mx > 0.0f && mx <= 65504.0f) {
            const uint32_t E = __float_as_uint(mx) >> 23;  // mx in [2^(E-127), 2^(E-126))
            inv = __uint_as_float((253u - E) << 23);        // 2^(126 - E)
            f = __uint_as_float((E + 1u) << 23);            // 2^(E - 126)
        }
        for (int d = lane; d < D; d += 32)
            qs[h * qstride + qpad(d)] = __half2float(__ushort_as_half(row[d])) * inv;
        if (lane == 0)
            fac[h] = sm_scale * f;
    }
}

// Logits of the quantized tokens [t_begin, tq_end) of KV head bh for NQB
// query heads; sink(h, t, s) receives each one.  t_begin and tq_end are
// multiples of G (tq_end may also be a chunk end, a multiple of 1024).
template <int BITS, int NQB, class Sink>
__device__ __forceinline__ void qk_quantized(const kivi_cache& c, size_t bh, int t_begin, int tq_end,
                                             const float* qs, const float* fac, Sink sink)
{
    using T = KeyTile<BITS, NQB>;
    using Rows = TileRows<BITS, T::NT>;
    const int D = c.D, G = c.G;
    const int qstride = qstride_of(D);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, tg = lane & 3;
    const int wr = g % T::WR, v = g / T::WR;
    const uint32_t soff = Rows::sel_offset(v);
    const int NGW = T::TOK / G > 1 ? T::TOK / G : 1;  // statistic groups per warp tile
    const int gi = g / NQB, hq = g % NQB;              // B column of this lane group
    const float* qrow = qs + hq * qstride;
    const int gi_row = (wr * T::P) / G;                // group of this lane group's rows

    for (int tok0 = t_begin + warp * T::TOK; tok0 < tq_end; tok0 += kDecodeWarps * T::TOK) {
        float acc[T::NT][4];
#pragma unroll
        for (int j = 0; j < T::NT; ++j)
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
        float zacc = 0.0f;
        const int grp = tok0 / G + gi;
        const bool col_ok = gi < NGW && grp * G < tq_end;
        const bool row_ok = tok0 + wr * T::P < tq_end;
        const int32_t* kw = c.kq + (bh * (size_t)(c.Tmax / T::P) + tok0 / T::P + wr) * D + tg * 16;
        const size_t so = (bh * (size_t)(c.Tmax / G) + grp) * D + tg * 16;

#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 64) {
            uint4 W[4];
            float4 S[4], Z[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                W[i] = row_ok ? ld_nc(kw + c0 + 4 * i) : make_uint4(0u, 0u, 0u, 0u);
                S[i] = col_ok ? ld_nc_f4(c.kscale + so + c0 + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
                Z[i] = col_ok ? ld_nc_f4(c.kzero + so + c0 + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const float4 qv = *reinterpret_cast<const float4*>(qrow + qpad(c0 + tg * 16 + 4 * s));
                zacc = fmaf(qv.x, Z[s].x, zacc);
                zacc = fmaf(qv.y, Z[s].y, zacc);
                zacc = fmaf(qv.z, Z[s].z, zacc);
                zacc = fmaf(qv.w, Z[s].w, zacc);
                uint32_t bh0, bl0, bh1, bl1;
                split_hi_lo(qv.x * S[s].x, qv.y * S[s].y, bh0, bl0);
                split_hi_lo(qv.z * S[s].z, qv.w * S[s].w, bh1, bl1);
#pragma unroll
                for (int j = 0; j < T::NT; ++j) {
                    const uint32_t sa = pair_sel(Rows::ya(j)) + soff;
                    const uint32_t sb = pair_sel(Rows::yb(j)) + soff;
                    const uint32_t a0 = code_pair<BITS>(W[s].x, W[s].y, sa, Rows::ma(j));
                    const uint32_t a1 = code_pair<BITS>(W[s].x, W[s].y, sb, Rows::mb(j));
                    const uint32_t a2 = code_pair<BITS>(W[s].z, W[s].w, sa, Rows::ma(j));
                    const uint32_t a3 = code_pair<BITS>(W[s].z, W[s].w, sb, Rows::mb(j));
                    mma_f16(acc[j], a0, a1, a2, a3, bh0, bh1);
                    mma_f16(acc[j], a0, a1, a2, a3, bl0, bl1);
                }
            }
        }
        // zero terms: column sums over the four lanes, then the lane's two columns
        zacc += __shfl_xor_sync(0xffffffffu, zacc, 1);
        zacc += __shfl_xor_sync(0xffffffffu, zacc, 2);
        const float zc[2] = {__shfl_sync(0xffffffffu, zacc, 8 * tg),
                             __shfl_sync(0xffffffffu, zacc, 8 * tg + 4)};
        if (!row_ok)
            continue;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int u = 2 * tg + cc;
            if (u / NQB != gi_row)
                continue;
            const int h = u % NQB;
            const float f = fac[h];
            const int tbase = tok0 + wr * T::P + 2 * v * T::NT;
#pragma unroll
            for (int j = 0; j < T::NT; ++j) {
                sink(h, tbase + 2 * j, f * fmaf(code_unscale<BITS>(Rows::ma(j)), acc[j][cc], zc[cc]));
                sink(h, tbase + 2 * j + 1, f * fmaf(code_unscale<BITS>(Rows::mb(j)), acc[j][2 + cc], zc[cc]));
            }
        }
    }
}

// Logits of the fp16 residual tokens [t0, t_end): D/32 lanes per token, each
// a 32-channel segment, fp32 FMA.
template <int NQB, class Sink>
__device__ __forceinline__ void qk_residual(const kivi_cache& c, size_t bh, int t0, int t_end,
                                            const float* qs, const float* fac, Sink sink)
{
    const int D = c.D, RG = c.R + c.G;
    const int qstride = qstride_of(D);
    const int LPR = D / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = lane % LPR;
    const int rows = 32 / LPR;
    for (int base = t0 + warp * rows; base < t_end; base += kDecodeWarps * rows) {
        const int t = base + lane / LPR;
        float acc[NQB];
#pragma unroll
        for (int h = 0; h < NQB; ++h)
            acc[h] = 0.0f;
        if (t < t_end) {
            const uint16_t* kr = c.kres + (bh * RG + t % RG) * D + seg * 32;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint4 kv = ld_nc(kr + u * 8);
#pragma unroll
                for (int e4 = 0; e4 < 2; ++e4)
#pragma unroll
                    for (int h = 0; h < NQB; ++h) {
                        const float4 qv =
                            *reinterpret_cast<const float4*>(qs + h * qstride + qpad(seg * 32 + u * 8 + e4 * 4));
                        const float qq[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            acc[h] = fmaf(qq[e], __half2float(__ushort_as_half(u4_half(kv, e4 * 4 + e))), acc[h]);
                    }
            }
        }
        for (int m = 1; m < LPR; m <<= 1)
#pragma unroll
            for (int h = 0; h < NQB; ++h)
                acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], m);
        if (t < t_end && seg == 0)
#pragma unroll
            for (int h = 0; h < NQB; ++h)
                sink(h, t, fac[h] * acc[h]);
    }
}

// ---------------------------------------------------------------- values ---

template <int BITS, int NQB>
struct ValTile {
    static constexpr int P = 32 / BITS;
    static constexpr int WC = cmin(BITS == 2 ? 4 : 8, (8 / NQB) * 32 / P);  // word-columns per block
    static constexpr int LPW = 8 / WC;   // lane groups per word-column
    static constexpr int CH = WC * P;    // channels per block
    static constexpr int NT = CH / 16;   // MMA tiles per block
};

// Shared-memory floats the p . V phase needs beyond p: per split, NQB x D
// partial outputs and NQB x (D / G) zero terms.
__host__ __device__ constexpr int pv_part_floats(int NQB, int D, int G)
{
    return kDecodeWarps * NQB * (D + D / G);
}

// Splits of the token range across the warps for a block count NCB.
__device__ __forceinline__ int pv_splits(int NCB) { return NCB >= kDecodeWarps ? 1 : kDecodeWarps / NCB; }

// p . V_hat over tokens [t_begin, t_end) of KV head bh for NQB query heads:
// p_sm[h][t - t_begin] holds the unnormalized probabilities.  Quantized
// tokens [t_begin, tq_end) go through the code MMA, residual tokens
// [tq_end, t_end) (from the fp16 ring) through the same tiles with the raw
// values as A and p as B.  Writes o_part[split][h][d] (without zero terms)
// and z_part[split][h][g]; each entry is written by exactly one lane, so the
// CTA's sum over splits is deterministic.
template <int BITS, int NQB>
__device__ __forceinline__ void pv_chunk(const kivi_cache& c, size_t bh, int t_begin, int tq_end,
                                         int t_end, const float* p_sm, float* o_part, float* z_part)
{
    using T = ValTile<BITS, NQB>;
    using Rows = TileRows<BITS, T::NT>;
    const int D = c.D, G = c.G, NGv = D / G, RG = c.R + c.G;
    const int DW = D / T::P;       // words per token row
    const int NCB = DW / T::WC;    // channel blocks
    const int NSPLIT = pv_splits(NCB);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, tg = lane & 3;
    const int wcl = g % T::WC, v = g / T::WC;
    const uint32_t soff = Rows::sel_offset(v);
    const int NGW = T::CH / G > 1 ? T::CH / G : 1;
    const int gi = g / NQB, hq = g % NQB;
    const bool col_ok = gi < NGW;
    const float* prow = p_sm + hq * kChunkTokens;  // p of token t at prow[t - t_begin]
    const int nq_slices = (tq_end - t_begin) / 16;          // quantized part: whole slices
    const int nr_slices = (t_end - tq_end + 15) / 16;       // residual part: last one ragged

    for (int unit = warp; unit < NCB * NSPLIT; unit += kDecodeWarps) {
        const int cb = unit % NCB, split = unit / NCB;
        const int grp0 = (cb * T::CH) / G;
        const int grp = grp0 + gi;
        float acc[T::NT][4];
#pragma unroll
        for (int j = 0; j < T::NT; ++j)
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
        float zacc = 0.0f;
        const int32_t* vw = c.vq + bh * (size_t)c.Tmax * DW + cb * T::WC + wcl;
        const float* vs = c.vscale + bh * (size_t)c.Tmax * NGv + grp;
        const float* vz = c.vzero + bh * (size_t)c.Tmax * NGv + grp;

        constexpr int UNR = 4;
#pragma unroll 1
        for (int k0 = split; k0 < nq_slices; k0 += NSPLIT * UNR) {
            uint32_t W[UNR][4];
            float S[UNR][4], Z[UNR][4];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const bool ok = k0 + u * NSPLIT < nq_slices;
                const size_t t = (size_t)t_begin + (k0 + u * NSPLIT) * 16 + 4 * tg;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    W[u][i] = ok ? (uint32_t)__ldg(vw + (t + i) * DW) : 0u;
                    S[u][i] = ok && col_ok ? __ldg(vs + (t + i) * NGv) : 0.0f;
                    Z[u][i] = ok && col_ok ? __ldg(vz + (t + i) * NGv) : 0.0f;
                }
            }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int k = k0 + u * NSPLIT;
                if (k >= nq_slices)
                    break;
                const float4 pv = *reinterpret_cast<const float4*>(prow + k * 16 + 4 * tg);
                zacc = fmaf(pv.x, Z[u][0], zacc);
                zacc = fmaf(pv.y, Z[u][1], zacc);
                zacc = fmaf(pv.z, Z[u][2], zacc);
                zacc = fmaf(pv.w, Z[u][3], zacc);
                uint32_t bh0, bl0, bh1, bl1;
                split_hi_lo(pv.x * S[u][0], pv.y * S[u][1], bh0, bl0);
                split_hi_lo(pv.z * S[u][2], pv.w * S[u][3], bh1, bl1);
#pragma unroll
                for (int j = 0; j < T::NT; ++j) {
                    const uint32_t sa = pair_sel(Rows::ya(j)) + soff;
                    const uint32_t sb = pair_sel(Rows::yb(j)) + soff;
                    const uint32_t a0 = code_pair<BITS>(W[u][0], W[u][1], sa, Rows::ma(j));
                    const uint32_t a1 = code_pair<BITS>(W[u][0], W[u][1], sb, Rows::mb(j));
                    const uint32_t a2 = code_pair<BITS>(W[u][2], W[u][3], sa, Rows::ma(j));
                    const uint32_t a3 = code_pair<BITS>(W[u][2], W[u][3], sb, Rows::mb(j));
                    mma_f16(acc[j], a0, a1, a2, a3, bh0, bh1);
                    mma_f16(acc[j], a0, a1, a2, a3, bl0, bl1);
                }
            }
        }
        // undo the code scaling before the residual tokens join the sums
#pragma unroll
        for (int j = 0; j < T::NT; ++j) {
            acc[j][0] *= code_unscale<BITS>(Rows::ma(j));
            acc[j][1] *= code_unscale<BITS>(Rows::ma(j));
            acc[j][2] *= code_unscale<BITS>(Rows::mb(j));
            acc[j][3] *= code_unscale<BITS>(Rows::mb(j));
        }
        // residual tokens: A = (v[t][d], v[t+1][d]) pairs, B = p (hi / lo)
        // the lane's 2 NT channels ch0 .. ch0 + 2 NT - 1 are contiguous: one
        // 16-byte (NT = 4) or 8-byte (NT = 2) load per residual token
        static_assert(T::NT == 2 || T::NT == 4, "value tiles per block");
        const int ch0 = (cb * T::WC + wcl) * T::P + 2 * v * T::NT;
#pragma unroll 1
        for (int k = split; k < nr_slices; k += NSPLIT) {
            const int tb = tq_end + k * 16 + 4 * tg;
            uint32_t X[4][T::NT];
            float pr[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = tb + i;
                const bool ok = t < t_end;
                pr[i] = ok && col_ok ? prow[t - t_begin] : 0.0f;
                const uint16_t* vr = c.vres + (bh * RG + (ok ? t : 0) % RG) * D + ch0;
                if constexpr (T::NT == 4) {
                    const uint4 x = ok ? ld_nc(vr) : make_uint4(0u, 0u, 0u, 0u);
                    X[i][0] = x.x;
                    X[i][1] = x.y;
                    X[i][2] = x.z;
                    X[i][3] = x.w;
                } else {
                    const uint2 x = ok ? __ldg(reinterpret_cast<const uint2*>(vr)) : make_uint2(0u, 0u);
                    X[i][0] = x.x;
                    X[i][1] = x.y;
                }
            }
            uint32_t bh0, bl0, bh1, bl1;
            split_hi_lo(pr[0], pr[1], bh0, bl0);
            split_hi_lo(pr[2], pr[3], bh1, bl1);
#pragma unroll
            for (int j = 0; j < T::NT; ++j) {
                const uint32_t a0 = __byte_perm(X[0][j], X[1][j], 0x5410);
                const uint32_t a1 = __byte_perm(X[0][j], X[1][j], 0x7632);
                const uint32_t a2 = __byte_perm(X[2][j], X[3][j], 0x5410);
                const uint32_t a3 = __byte_perm(X[2][j], X[3][j], 0x7632);
                mma_f16(acc[j], a0, a1, a2, a3, bh0, bh1);
                mma_f16(acc[j], a0, a1, a2, a3, bl0, bl1);
            }
        }

        zacc += __shfl_xor_sync(0xffffffffu, zacc, 1);
        zacc += __shfl_xor_sync(0xffffffffu, zacc, 2);
        float* op = o_part + (size_t)split * NQB * D;
        float* zp = z_part + (size_t)split * NQB * NGv;
        if (tg == 0 && col_ok)
            zp[hq * NGv + grp] = zacc;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int u = 2 * tg + cc;
            const int ugi = u / NQB, uh = u % NQB;
            if (ugi >= NGW)
                continue;
#pragma unroll
            for (int j = 0; j < T::NT; ++j) {
                const int cha = ch0 + 2 * j;
                if (grp0 + ugi != cha / G)
                    continue;
                op[uh * D + cha] = acc[j][cc];
                op[uh * D + cha + 1] = acc[j][2 + cc];
            }
        }
    }
}

// Chunk softmax statistics over p_sm[h][0 .. n) (holding logits on entry):
// m_h = max, p = exp(s - m_h) in place, l_h = sum p.  Whole CTA.
template <int NQB>
__device__ __forceinline__ void chunk_softmax(float* p_sm, int n, float (&m)[NQB], float (&l)[NQB],
                                              float* red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int h = 0; h < NQB; ++h) {
        float mx = -INFINITY;
        for (int t = threadIdx.x; t < n; t += kDecodeThreads)
            mx = fmaxf(mx, p_sm[h * kChunkTokens + t]);
        m[h] = mx;
    }
#pragma unroll
    for (int h = 0; h < NQB; ++h)
        for (int k = 16; k > 0; k >>= 1)
            m[h] = fmaxf(m[h], __shfl_xor_sync(0xffffffffu, m[h], k));
    if (lane == 0)
#pragma unroll
        for (int h = 0; h < NQB; ++h)
            red[warp * NQB + h] = m[h];
    __syncthreads();
#pragma unroll
    for (int h = 0; h < NQB; ++h) {
        float r = red[h];
#pragma unroll
        for (int w = 1; w < kDecodeWarps; ++w)
            r = fmaxf(r, red[w * NQB + h]);
        m[h] = r;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < NQB; ++h) {
        float s = 0.0f;
        for (int t = threadIdx.x; t < n; t += kDecodeThreads) {
            const float e = expf(p_sm[h * kChunkTokens + t] - m[h]);
            p_sm[h * kChunkTokens + t] = e;
            s += e;
        }
        l[h] = s;
    }
#pragma unroll
    for (int h = 0; h < NQB; ++h)
        for (int k = 16; k > 0; k >>= 1)
            l[h] += __shfl_xor_sync(0xffffffffu, l[h], k);
    if (lane == 0)
#pragma unroll
        for (int h = 0; h < NQB; ++h)
            red[warp * NQB + h] = l[h];
    __syncthreads();  // also publishes p_sm
#pragma unroll
    for (int h = 0; h < NQB; ++h) {
        float r = red[h];
#pragma unroll
        for (int w = 1; w < kDecodeWarps; ++w)
            r += red[w * NQB + h];
        l[h] = r;
    }
}

// Writes the chunk's partial (o, m, l) for query heads hq0 .. hq0+NQB-1:
// o[h][d] = sum over splits of o_part + z_part of d's group.  Whole CTA,
// after a barrier that follows pv_chunk.
template <int NQB>
__device__ __forceinline__ void write_partials(int D, int G, int nsplit, const float* o_part,
                                               const float* z_part, const float (&m)[NQB],
                                               const float (&l)[NQB], size_t row0, int nchunks,
                                               float* ws_o, float* ws_m, float* ws_l)
{
    const int NGv = D / G;
    for (int idx = threadIdx.x; idx < NQB * D; idx += kDecodeThreads) {
        const int h = idx / D, d = idx % D;
        float s = 0.0f;
        for (int sp = 0; sp < nsplit; ++sp)
            s += o_part[((size_t)sp * NQB + h) * D + d] + z_part[((size_t)sp * NQB + h) * NGv + d / G];
        ws_o[(row0 + (size_t)h * nchunks) * D + d] = s;
    }
#pragma unroll
    for (int h = 0; h < NQB; ++h)
        if (threadIdx.x == h) {
            ws_m[row0 + (size_t)h * nchunks] = m[h];
            ws_l[row0 + (size_t)h * nchunks] = l[h];
        }
}

}  // namespace kivi
