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
// Staging.  A CTA owns one KV head and one chunk of TC tokens.  The chunk's
// packed keys (word-rows and per-channel statistics) and packed values (token
// rows and per-token statistics) are contiguous in HBM; at launch every thread
// issues its share of 16-byte cp.async copies of both into shared memory (two
// commit groups, keys first), so the whole chunk is in flight at once and the
// tiles read shared memory only.  The 16-byte chunks are placed with an XOR
// swizzle so that the tile reads are free of bank conflicts.
//
// A operand, codes as fp16 subnormals.  A code c at bit position p of a
// 16-bit half (p + b <= 10) is the fp16 subnormal c 2^(p - 24) once the other
// bits are cleared: one AND yields two A values, exact for every code, and the
// factor 2^(24 - p) is applied to the fp32 accumulator afterwards.  No
// conversion instruction runs per code.
//   keys: a key word holds 32/b tokens of one channel, while an A register
//   pairs two channels of one token; one PRMT moves byte y of two channel
//   words into bytes 0 and 2 of a register, then ANDs pick the positions.
//   values: a value word holds 32/b channels of one token, an A register pairs
//   two tokens of one channel; ldmatrix.trans delivers exactly that pairing at
//   16-bit granularity (half h of tokens 2 tg and 2 tg + 1), so ANDs alone (and
//   one shift for the top positions) build the operand.
//
// B operand.  w is split into two fp16 terms, hi = w with its low 13
// mantissa bits cleared (exact in fp16) and lo = fp16(w - hi), and both MMAs
// accumulate into the same fp32 registers, so the weights carry about 22
// significant bits.  Ranges: p <= 1 and s <= 131008 / 3 keep |p s| < 65504;
// for keys q is pre-scaled per head by a power of two so that max |q| < 1
// (the factor returns exactly in the epilogue).
//
// Columns.  A tile's N = 8 columns are (statistic group, query head) pairs,
// so one B fragment serves rows from several groups and several heads of a
// grouped-query set; each output reads the column of its own group.
#pragma once

#include <math.h>

#include "kivi_device.cuh"

namespace kivi {

constexpr int kDecodeThreads = 128;
constexpr int kDecodeWarps = kDecodeThreads / 32;

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }
__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x >> 1); }

// Query heads processed together per KV head: 4, 2 or 1.
__host__ __device__ constexpr int heads_per_pass(int NQ) { return NQ % 4 == 0 ? 4 : NQ % 2 == 0 ? 2 : 1; }

// D += A * B, m16n8k16, fp16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Four 8x8 b16 matrices, transposed: lanes 8i .. 8i+7 give the row addresses
// of matrix i; r[i] of lane (g, tg) holds rows 2 tg and 2 tg + 1 of column g.
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(addr));
}

// Two-bit ... eight-bit code field at position p of both 16-bit halves.
template <int BITS>
__host__ __device__ constexpr uint32_t half_pair_mask(int p)
{
    return (((1u << BITS) - 1u) << p) | ((((1u << BITS) - 1u) << p) << 16);
}

// fp32 factor that undoes the 2^(p - 24) of a code at bit position p of a half.
__host__ __device__ constexpr float code_unscale_bits(int p) { return (float)(1u << (24 - p)); }

// w = hi + lo as two fp16 pairs (see the B operand note above).
__device__ __forceinline__ void split_hi_lo(float a, float b, uint32_t& hi, uint32_t& lo)
{
    const float ah = __uint_as_float(__float_as_uint(a) & 0xFFFFE000u);
    const float bh = __uint_as_float(__float_as_uint(b) & 0xFFFFE000u);
    hi = h2_bits(__floats2half2_rn(ah, bh));
    lo = h2_bits(__floats2half2_rn(__fsub_rn(a, ah), __fsub_rn(b, bh)));
}

// One fp16 pair of the split: hi (part 0) or lo (part 1).
__device__ __forceinline__ uint32_t split_part(float a, float b, int part)
{
    const float ah = __uint_as_float(__float_as_uint(a) & 0xFFFFE000u);
    const float bh = __uint_as_float(__float_as_uint(b) & 0xFFFFE000u);
    return h2_bits(__floats2half2_rn(part ? __fsub_rn(a, ah) : ah, part ? __fsub_rn(b, bh) : bh));
}

// Power of two f with mx f in [2^13, 2^14) for the largest statistic mx >= 0
// of a chunk (1 when mx == 0): the decode weights q s f (|q| < 1) and p s f
// (p <= 1) then lie below 2^14, and every weight within 2^-27 of the largest
// keeps its hi part a normal fp16 number, so the hi / lo split holds its 22
// bits relative to the chunk's largest weight however small the statistics
// are.  f and 1 / f are exact.
__device__ __forceinline__ float weight_scale_pow2(float mx)
{
    if (!(mx > 0.0f))
        return 1.0f;
    const int E = min(max((int)(__float_as_uint(mx) >> 23), 127 - 40), 254);
    return __uint_as_float((uint32_t)(267 - E) << 23);  // 2^(140 - E)
}

// Largest of n non-negative staged statistics, over the whole CTA; every
// thread receives it.  red: kDecodeWarps floats of shared memory.  Contains
// barriers: call from every thread, after the statistics are visible.
__device__ __forceinline__ float cta_max_stat(const float* s, int n, float* red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float mx = 0.0f;
    for (int i = threadIdx.x; i < n; i += kDecodeThreads)
        mx = fmaxf(mx, s[i]);
    for (int k = 16; k > 0; k >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
    __syncthreads();  // red may still be read by a previous reduction
    if (lane == 0)
        red[warp] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < kDecodeWarps; ++w)
        mx = fmaxf(mx, red[w]);
    return mx;
}

// -------------------------------------------------------------- shapes ---

// Keys: the 8 lane groups g of a warp take WR word-rows (LPW = 8 / WR lane
// groups per word-row, sub-lane v = g / WR); rows g and g + 8 of MMA tile j
// are code positions 2 pi and 2 pi + 1, pi = v NT + j, of the lane group's
// word-row; TOK tokens per warp tile.
template <int BITS, int NQB>
struct KeyTile {
    static constexpr int P = 32 / BITS;
    static constexpr int CPB = 8 / BITS;                    // codes per byte
    static constexpr int WR = cmin(8, (8 / NQB) * 32 / P);  // word-rows per warp tile
    static constexpr int TOK = WR * P;                      // tokens per warp tile
    static constexpr int NT = TOK / 16;                     // MMA tiles per warp tile
    // byte / bit position of rows g (a) and g + 8 (b) of tile j for v = 0
    __host__ __device__ static constexpr int ya(int j) { return (2 * j) / CPB; }
    __host__ __device__ static constexpr int yb(int j) { return (2 * j + 1) / CPB; }
    __host__ __device__ static constexpr int pa(int j) { return BITS * ((2 * j) % CPB); }
    __host__ __device__ static constexpr int pb(int j) { return BITS * ((2 * j + 1) % CPB); }
    static_assert((2 * NT) % CPB == 0, "sub-lane positions must start on a byte");
    // hi and lo weights as separate B columns (one MMA per tile) when the
    // (group, head) units of a warp tile take at most four columns
    static constexpr bool HL = NQB == 1 || (NQB == 2 && BITS >= 4);
};

// Values: a 16-byte segment of a token row holds 8 halves of HC codes; the
// lane group g owns half g, and tile j its positions 2j (row g) and 2j + 1
// (row g + 8).  Positions whose field would reach the fp16 exponent are read
// after one right shift by SHIFT bits.
template <int BITS>
struct ValTile {
    static constexpr int P = 32 / BITS;
    static constexpr int HC = 16 / BITS;                    // codes per 16-bit half
    static constexpr int CS = 8 * HC;                       // channels per segment
    static constexpr int NT = HC / 2;                       // MMA tiles per segment
    static constexpr int NDIRECT = BITS == 2 ? 5 : HC / 2;  // positions read unshifted
    static constexpr int SHIFT = NDIRECT * BITS;
    __host__ __device__ static constexpr bool shifted(int m) { return m >= NDIRECT; }
    __host__ __device__ static constexpr int bitpos(int m) { return BITS * (shifted(m) ? m - NDIRECT : m); }
};

// ------------------------------------------------------- shared memory ---

// Staged keys: word-rows [TC/P][D] then scales and zeros [TC/G][D] (words).
__host__ __device__ constexpr size_t key_stage_words(int TC, int D, int bits_k, int G)
{
    return (size_t)(TC / (32 / bits_k)) * D + 2 * (size_t)(TC / G) * D;
}
// Probability rows [NQB][TX + 8] for chunks of up to TX tokens (the pad
// spreads heads over banks).
__host__ __device__ constexpr int prob_stride(int TX) { return TX + 8; }
// B fragments of p . V: [(D/G) NQB rows][TX/2] uint2 (hi pair, lo pair of
// tokens 2i, 2i+1), pair i of row r stored at i ^ bb_swz(r).
__host__ __device__ constexpr int bb_stride(int TX) { return TX / 2; }
__host__ __device__ constexpr int bb_swz(int r) { return (r & 3) << 2; }
__host__ __device__ constexpr size_t bb_words(int TX, int D, int G, int NQB)
{
    return 2 * (size_t)(D / G) * NQB * bb_stride(TX);
}
// Split partials [4][NQB][D]; per-warp zero terms and exponential sums
// [4][NQB][D/G + 1] (entry D/G of a row is the sum).
__host__ __device__ constexpr size_t part_words(int D, int NQB) { return (size_t)kDecodeWarps * NQB * D; }
__host__ __device__ constexpr size_t zs_words(int D, int G, int NQB) { return (size_t)kDecodeWarps * NQB * (D / G + 1); }

// Largest slack S (tokens the last chunk of a sequence may hold beyond TC,
// so that a short tail does not cost a CTA of its own).  A sequence keeps at
// least R tokens in its fp16 residual (read from the ring, never staged), so
// with S <= R the quantized tokens of any chunk still fit the TC staged ones:
// the last chunk starts at c TC > n - TC - S and its quantized tokens end at
// or before n - R.  A multiple of 16 (whole p . V slices).
__host__ __device__ constexpr int max_chunk_slack(int TC, int R) { return cmin(R, TC / 4) & ~15; }
// Chunks of a sequence of n tokens: all but the last hold TC tokens, the
// last one at most TC + S.
__host__ __device__ constexpr int decode_chunks(int n, int TC, int S)
{
    return n <= 0 ? 0 : cmax(1, (n - S + TC - 1) / TC);
}

// Word offsets into a decode kernel's dynamic shared memory: the staged keys
// and / or values of TC tokens, then the probabilities (logits) and B
// fragments of up to TX = TC + slack tokens, the split partials when they do
// not overlay a dead region, and the zero terms (or these on the logits).
struct DecodeLayout {
    size_t kw, ks, kz, vw, vs, vz;
    size_t p, bb, part, zs, total;
    bool bb_on_keys, part_on_vstats, zs_on_p;
};

// keys / values: whether the kernel stages them.  The B fragments overlay the
// staged keys (dead once the logits exist), the split partials the value
// statistics (dead once the B fragments exist) when one pass covers all query
// heads of the staged chunk.
__host__ __device__ inline DecodeLayout decode_layout(int TC, int TX, int D, int bits_k, int bits_v, int G,
                                                      int NQB, bool multipass, bool keys, bool values,
                                                      bool zs_on_p = false)
{
    DecodeLayout L{};
    size_t o = 0;
    if (keys) {
        const size_t kwn = (size_t)(TC / (32 / bits_k)) * D, ksn = (size_t)(TC / G) * D;
        L.kw = o;
        L.ks = o + kwn;
        L.kz = L.ks + ksn;
        o = L.kz + ksn;
    }
    size_t vsn = 0;
    if (values) {
        const size_t vwn = (size_t)TC * (D / (32 / bits_v));
        vsn = (size_t)TC * (D / G);
        L.vw = o;
        L.vs = o + vwn;
        L.vz = L.vs + vsn;
        o = L.vz + vsn;
        L.p = o;
        o += (size_t)NQB * prob_stride(TX);
        const size_t bbn = bb_words(TX, D, G, NQB);
        L.bb_on_keys = keys && bbn <= key_stage_words(TC, D, bits_k, G);
        if (L.bb_on_keys) {
            L.bb = L.kw;
        } else {
            L.bb = o;
            o += bbn;
        }
        L.part_on_vstats = !multipass && part_words(D, NQB) <= 2 * vsn;
        if (L.part_on_vstats) {
            L.part = L.vs;
        } else {
            L.part = o;
            o += part_words(D, NQB);
        }
        // the zero terms get their own words, or (zs_on_p, when shared memory
        // is tight) overlay the logits, dead once the B fragments exist:
        // pv_weights then writes them after a barrier
        L.zs_on_p = zs_on_p;
        if (zs_on_p) {
            L.zs = L.p;
        } else {
            L.zs = o;
            o += zs_words(D, G, NQB);
        }
    }
    L.total = o;
    return L;
}

// Chunking of the decode kernels: TC tokens per chunk, the largest of 1024
// ... 64 that is a multiple of G and of the key warp tile and whose
// fused-kernel layout (staged keys and values, probabilities, B fragments,
// partials) fits three CTAs per SM (else two, else one); then the slack S of
// the last chunk, max_chunk_slack(TC, R) if the layout with it still fits the
// same budget, else 0.
struct ChunkPlan {
    int TC, S, ctas_per_sm;
    bool zs_on_p;
};

// fp32 q row in shared memory: channel d at qpad(d) (4 floats of padding per
// 16 channels spread the LDS.128 of the four lanes of a lane group over banks)
// and rows D + D/4 (+16) floats apart, 16 (mod 32), so that two heads read by
// one quarter-warp use the other half of the banks.
__host__ __device__ constexpr int qstride_of(int D) { return D + D / 4 + ((D + D / 4) % 32 == 0 ? 16 : 0); }

// Shared memory per SM, and what each resident CTA also takes besides the
// dynamic layout: the runtime's reserve and the static q rows / reductions.
constexpr size_t kSmemPerSM = 228 * 1024;
constexpr size_t kSmemReservedPerCTA = 1024;
__host__ __device__ constexpr size_t decode_static_smem(int D, int NQB)
{
    return 4 * ((size_t)NQB * qstride_of(D) + NQB + (size_t)kDecodeWarps * NQB);
}

__host__ __device__ inline ChunkPlan decode_chunk_plan(int D, int bits_k, int bits_v, int G, int R, int NQ)
{
    const int NQB = heads_per_pass(NQ);
    const int P = 32 / bits_k;
    const int tok = cmin(8, (8 / NQB) * 32 / P) * P;
    const int tc_min = cmax(cmax(tok, G), 64);
    auto bytes = [&](int TC, int S, bool zp) {
        return 4 * decode_layout(TC, TC + S, D, bits_k, bits_v, G, NQB, NQ > NQB, true, true, zp).total;
    };
    for (int ctas = 3; ctas >= 1; --ctas) {
        const size_t budget = kSmemPerSM / ctas - kSmemReservedPerCTA - decode_static_smem(D, NQB);
        for (int TC = 1024; TC >= tc_min; TC >>= 1)
            for (int zp = 0; zp < 2; ++zp)  // the zero terms on the logits only if that makes it fit
                if (bytes(TC, 0, zp) <= budget) {
                    const int S = max_chunk_slack(TC, R);
                    return {TC, bytes(TC, S, zp) <= budget ? S : 0, ctas, zp != 0};
                }
    }
    return {tc_min, 0, 1, true};
}

inline ChunkPlan chunk_plan(const kivi_cache& c, int Hq)
{
    return decode_chunk_plan(c.D, c.bits_k, c.bits_v, c.G, c.R, Hq / c.H);
}

// ------------------------------------------------------------- staging ---

// Physical 16-byte chunk of logical chunk x in key row r (word-row or
// statistics group row).  qk_quantized's lanes 0-7 read chunks 4 tg + i
// (tg = 0..3) of two consecutive rows; the XOR spreads those eight chunks
// over the eight 16-byte bank groups.  It changes bits 0-1 only, so a chunk
// stays in its row.
__device__ __forceinline__ int key_swz(int r, int x) { return x ^ (((x >> 3) & 1) | ((r & 1) << 1)); }

// Physical segment of segment s in value row t, for NSEG segments per row:
// ldmatrix reads one segment of 8 consecutive rows per phase; the XOR puts
// those 8 x 16 bytes into distinct bank groups.
__device__ __forceinline__ int val_swz(int t, int s, int NSEG)
{
    const int sh = NSEG >= 8 ? 0 : ilog2(8 / NSEG);
    const int msk = (NSEG >= 8 ? 8 : NSEG) - 1;
    return s ^ ((t >> sh) & msk);
}

// cp.async copies of the chunk's quantized keys [t_begin, tq_end) into kw /
// ks / kz (key_swz layout); rows from tq_end up to the next multiple of TOK
// tokens are zero-filled so that whole warp tiles can be read unguarded.  A
// thread's 16-byte chunks are kDecodeThreads apart, i.e. a fixed column of
// every (kDecodeThreads / chunks-per-row)-th row, so its swizzled column is
// fixed (the row step is even) and the loops only advance pointers.
template <int BITS, int TOK, int D>
__device__ __forceinline__ void stage_keys(const kivi_cache& c, size_t bh, int t_begin, int tq_end,
                                           uint32_t* kw, float* ks, float* kz)
{
    constexpr int P = 32 / BITS;
    const int lgG = ilog2(c.G);
    constexpr int lg = ilog2(D / 4);                // 16-byte chunks per row: D / 4
    constexpr int step = kDecodeThreads >> lg;      // rows per sweep (even)
    const int x = threadIdx.x & (D / 4 - 1), r0 = threadIdx.x >> lg;
    const int xs = key_swz(r0, x);
    const int n = tq_end - t_begin, npad = (n + TOK - 1) / TOK * TOK;
    constexpr size_t adv = (size_t)step * D;        // words per sweep
    {
        const int nw = n / P, nwp = npad / P;
        const int32_t* src = c.kq + (bh * (size_t)(c.Tmax / P) + t_begin / P) * D + (size_t)r0 * D + 4 * x;
        uint32_t* dst = kw + (size_t)r0 * D + 4 * xs;
        int r = r0;
        for (; r < nw; r += step, src += adv, dst += adv)
            cp_async16(dst, src);
        for (; r < nwp; r += step, dst += adv)
            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    {
        const int ng = n >> lgG, ngp = (npad + c.G - 1) >> lgG;
        const size_t so = (bh * (size_t)(c.Tmax >> lgG) + (t_begin >> lgG)) * D + (size_t)r0 * D + 4 * x;
        const float* s1 = c.kscale + so;
        const float* s2 = c.kzero + so;
        const size_t d0 = (size_t)r0 * D + 4 * xs;
        float* d1 = ks + d0;
        float* d2 = kz + d0;
        int r = r0;
        for (; r < ng; r += step, s1 += adv, s2 += adv, d1 += adv, d2 += adv) {
            cp_async16(d1, s1);
            cp_async16(d2, s2);
        }
        for (; r < ngp; r += step, d1 += adv, d2 += adv) {
            *reinterpret_cast<float4*>(d1) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(d2) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// cp.async copies of the chunk's quantized values [t_begin, tq_end): token
// rows into vw (val_swz layout), statistics into vs / vz [t - t_begin][D/G].
// As for the keys, a thread's segment (and its swizzled place) is fixed.
template <int BITS, int D>
__device__ __forceinline__ void stage_values(const kivi_cache& c, size_t bh, int t_begin, int tq_end,
                                             uint32_t* vw, float* vs, float* vz)
{
    constexpr int P = 32 / BITS, DW = D / P, NSEG = DW / 4;
    const int NGv = D >> ilog2(c.G);
    constexpr int lg = ilog2(NSEG);
    const int n = tq_end - t_begin;
    const int seg = threadIdx.x & (NSEG - 1), t0 = threadIdx.x >> lg;
    constexpr int step = kDecodeThreads >> lg;      // tokens per sweep (a multiple of 8)
    constexpr size_t adv = (size_t)kDecodeThreads * 4;  // words per sweep
    {
        const int32_t* src = c.vq + (bh * (size_t)c.Tmax + t_begin) * DW + (size_t)threadIdx.x * 4;
        uint32_t* dst = vw + (size_t)t0 * DW + val_swz(t0, seg, NSEG) * 4;
        for (int t = t0; t < n; t += step, src += adv, dst += adv)
            cp_async16(dst, src);
    }
    {
        const int nf = (n * NGv) / 4;  // n is a multiple of 32
        const size_t so = (bh * (size_t)c.Tmax + t_begin) * NGv + (size_t)threadIdx.x * 4;
        const float* s1 = c.vscale + so;
        const float* s2 = c.vzero + so;
        float* d1 = vs + threadIdx.x * 4;
        float* d2 = vz + threadIdx.x * 4;
        for (int i = threadIdx.x; i < nf; i += kDecodeThreads, s1 += adv, s2 += adv, d1 += adv, d2 += adv) {
            cp_async16(d1, s1);
            cp_async16(d2, s2);
        }
    }
}

// ------------------------------------------------------------------ keys ---

__device__ __forceinline__ int qpad(int d) { return d + ((d >> 4) << 2); }

// Stages query heads hq0 .. hq0+NQB-1 of sequence b: qs[h][qpad(d)] = q 2^-e_h fk
// with 2^-e_h the power of two that brings max_d |q| into [1/2, 1) and fk the
// chunk's key weight scale (weight_scale_pow2 of its largest key scale), and
// fac[h] = sm_scale 2^e_h / fk.  Called by the whole CTA between barriers.
template <int NQB, int D>
__device__ __forceinline__ void stage_q(const uint16_t* __restrict__ q, float sm_scale, float fk, float* qs,
                                        float* fac)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int qstride = qstride_of(D);
    for (int h = warp; h < NQB; h += kDecodeWarps) {
        const uint16_t* row = q + (size_t)h * D;
        float mx = 0.0f;
        for (int d = lane; d < D; d += 32)
            mx = fmaxf(mx, fabsf(__half2float(__ushort_as_half(ld_checked(row + d)))));
        for (int m = 16; m > 0; m >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
        float inv = 1.0f, f = 1.0f;
        if (mx > 0.0f && mx <= 65504.0f) {
            const uint32_t E = __float_as_uint(mx) >> 23;  // mx in [2^(E-127), 2^(E-126))
            inv = __uint_as_float((253u - E) << 23);        // 2^(126 - E)
            f = __uint_as_float((E + 1u) << 23);            // 2^(E - 126)
        }
        inv *= fk;
        f *= __frcp_rn(fk);  // exact: fk is a power of two
        for (int d = lane; d < D; d += 32)
            qs[h * qstride + qpad(d)] = __half2float(__ushort_as_half(ld_checked(row + d))) * inv;
        if (lane == 0)
            fac[h] = sm_scale * f;
    }
}

// Query head whose logits land in running-maximum slot `slot` of the calling
// lane in qk_quantized (-1: none).
template <int BITS, int NQB>
__device__ __forceinline__ int qk_slot_head(int slot)
{
    const int tg = threadIdx.x & 3;
    if (KeyTile<BITS, NQB>::HL)
        return slot == 0 ? tg % NQB : -1;
    return (2 * tg + slot) % NQB;
}

// Logits of quantized tokens for NQB query heads from the staged keys of the
// chunk starting at t_begin (zero-filled up to a whole warp tile); the calling
// warp takes the warp tiles that start at tok_first, tok_first + tok_step, ...
// below tok_end (<= tq_end, the end of the quantized tokens); sink(h, t, s)
// receives each logit.  lmax[slot] keeps the running maximum of the logits
// the lane emits for head qk_slot_head<BITS, NQB>(slot) (two slots; the
// caller initializes them).
template <int BITS, int NQB, int D, class Sink>
__device__ __forceinline__ void qk_quantized(int G, int t_begin, int tq_end, int tok_first,
                                             int tok_end, int tok_step, const uint32_t* kw,
                                             const float* ks, const float* kz, const float* qs,
                                             const float* fac, Sink sink, float (&lmax)[2])
{
    using T = KeyTile<BITS, NQB>;
    constexpr int qstride = qstride_of(D);
    constexpr int cpr = D / 4;  // 16-byte chunks per staged row
    const int lgG = ilog2(G);
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tg = lane & 3;
    const int wr = g % T::WR, v = g / T::WR;
    const uint32_t soff = (uint32_t)(2 * v * T::NT / T::CPB) * 0x101u;  // byte offset of sub-lane v
    const int NGW = cmax(1, T::TOK >> lgG);         // statistic groups per warp tile
    // B column g: unit (group gi, head hq) = g / 2 and weight part g & 1 with
    // hi / lo columns, else unit g with hi and lo in two MMAs
    const int unit = T::HL ? g >> 1 : g, part = g & 1;
    const int gi = cmin(unit / NQB, NGW - 1);       // clamped; extra columns unused
    const int hq = unit % NQB;
    const float* qrow = qs + hq * qstride + qpad(tg * 16);
    const int gi_row = (wr * T::P) >> lgG;          // group of this lane group's rows

    for (int tok0 = tok_first; tok0 < tok_end; tok0 += tok_step) {
        float acc[T::NT][4];
#pragma unroll
        for (int j = 0; j < T::NT; ++j)
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
        float zacc = 0.0f;
        const int lr = (tok0 - t_begin) / T::P + wr;    // staged word-row
        const int lgp = ((tok0 - t_begin) >> lgG) + gi; // staged group row of the B column
        const int xr = (tg >> 1) | ((lr & 1) << 1);     // key_swz of this lane's chunks
        const int xg = (tg >> 1) | ((lgp & 1) << 1);
        const uint4* wrow = reinterpret_cast<const uint4*>(kw) + lr * cpr + 4 * tg;
        const float4* srow = reinterpret_cast<const float4*>(ks) + lgp * cpr + 4 * tg;
        const float4* zrow = reinterpret_cast<const float4*>(kz) + lgp * cpr + 4 * tg;

#pragma unroll 1
        for (int c0 = 0; c0 < cpr; c0 += 16) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint4 W = wrow[c0 + (s ^ xr)];
                const float4 S = srow[c0 + (s ^ xg)];
                const float4 Z = zrow[c0 + (s ^ xg)];
                const float4 qv = *reinterpret_cast<const float4*>(qrow + 5 * c0 + 4 * s);
                zacc = fmaf(qv.x, Z.x, zacc);
                zacc = fmaf(qv.y, Z.y, zacc);
                zacc = fmaf(qv.z, Z.z, zacc);
                zacc = fmaf(qv.w, Z.w, zacc);
                uint32_t bh0, bl0, bh1, bl1;
                if constexpr (T::HL) {
                    bh0 = split_part(qv.x * S.x, qv.y * S.y, part);
                    bh1 = split_part(qv.z * S.z, qv.w * S.w, part);
                } else {
                    split_hi_lo(qv.x * S.x, qv.y * S.y, bh0, bl0);
                    split_hi_lo(qv.z * S.z, qv.w * S.w, bh1, bl1);
                }
#pragma unroll
                for (int j = 0; j < T::NT; ++j) {
                    const uint32_t sa = ((uint32_t)T::ya(j) | ((uint32_t)(4 + T::ya(j)) << 8)) + soff;
                    const uint32_t sb = ((uint32_t)T::yb(j) | ((uint32_t)(4 + T::yb(j)) << 8)) + soff;
                    const uint32_t ma = half_pair_mask<BITS>(T::pa(j)), mb = half_pair_mask<BITS>(T::pb(j));
                    const uint32_t a0 = __byte_perm(W.x, W.y, sa) & ma;
                    const uint32_t a1 = __byte_perm(W.x, W.y, sb) & mb;
                    const uint32_t a2 = __byte_perm(W.z, W.w, sa) & ma;
                    const uint32_t a3 = __byte_perm(W.z, W.w, sb) & mb;
                    mma_f16(acc[j], a0, a1, a2, a3, bh0, bh1);
                    if constexpr (!T::HL)
                        mma_f16(acc[j], a0, a1, a2, a3, bl0, bl1);
                }
            }
        }
        // zero terms: column sums over the four lanes, then the lane's columns
        // (every lane shuffles, before any lane leaves the iteration).  With
        // hi / lo columns, columns 2 tg and 2 tg + 1 both belong to unit tg.
        zacc += __shfl_xor_sync(0xffffffffu, zacc, 1);
        zacc += __shfl_xor_sync(0xffffffffu, zacc, 2);
        const float zc[2] = {__shfl_sync(0xffffffffu, zacc, 8 * tg),
                             __shfl_sync(0xffffffffu, zacc, 8 * tg + 4)};
        if (tok0 + wr * T::P >= tq_end)
            continue;
        const int tbase = tok0 + wr * T::P + 2 * v * T::NT;
        if constexpr (T::HL) {
            const int h = tg % NQB;
            if (tg / NQB == gi_row) {
                const float f = fac[h];
#pragma unroll
                for (int j = 0; j < T::NT; ++j) {
                    const float s0 = f * fmaf(code_unscale_bits(T::pa(j)), acc[j][0] + acc[j][1], zc[0]);
                    const float s1 = f * fmaf(code_unscale_bits(T::pb(j)), acc[j][2] + acc[j][3], zc[0]);
                    sink(h, tbase + 2 * j, s0);
                    sink(h, tbase + 2 * j + 1, s1);
                    lmax[0] = fmaxf(lmax[0], fmaxf(s0, s1));
                }
            }
        } else {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int u = 2 * tg + cc;
                if (u / NQB != gi_row)
                    continue;
                const int h = u % NQB;
                const float f = fac[h];
#pragma unroll
                for (int j = 0; j < T::NT; ++j) {
                    const float s0 = f * fmaf(code_unscale_bits(T::pa(j)), acc[j][cc], zc[cc]);
                    const float s1 = f * fmaf(code_unscale_bits(T::pb(j)), acc[j][2 + cc], zc[cc]);
                    sink(h, tbase + 2 * j, s0);
                    sink(h, tbase + 2 * j + 1, s1);
                    lmax[cc] = fmaxf(lmax[cc], fmaxf(s0, s1));
                }
            }
        }
    }
}

// Logits of fp16 residual tokens (read from the ring in global memory): D/32
// lanes per token, each a 32-channel segment, fp32 FMA; the calling warp
// takes 32 / (D/32) tokens from base0, then every `step` tokens, below t_end.
template <int NQB, int D, class Sink>
__device__ __forceinline__ void qk_residual(const kivi_cache& c, size_t bh, int base0, int step, int t_end,
                                            const float* qs, const float* fac, Sink sink, float (&rmax)[NQB])
{
    const int RG = c.R + c.G;
    constexpr int qstride = qstride_of(D);
    constexpr int LPR = D / 32;
    const int lane = threadIdx.x & 31;
    const int seg = lane % LPR;
    for (int base = base0; base < t_end; base += step) {
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
            for (int h = 0; h < NQB; ++h) {
                const float sv = fac[h] * acc[h];
                sink(h, t, sv);
                rmax[h] = fmaxf(rmax[h], sv);
            }
    }
}

// ---------------------------------------------------------------- values ---

// Per-head maximum over the CTA of the per-thread maxima m[h] (logits of
// the chunk); every thread receives the result.  Whole CTA; its barrier also
// publishes what the threads wrote to shared memory before the call.
template <int NQB>
__device__ __forceinline__ void chunk_max(float (&m)[NQB], float* red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int h = 0; h < NQB; ++h) {
        float mx = m[h];
        for (int k = 16; k > 0; k >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
        if (lane == 0)
            red[warp * NQB + h] = mx;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < NQB; ++h) {
        float r = red[h];
#pragma unroll
        for (int w = 1; w < kDecodeWarps; ++w)
            r = fmaxf(r, red[w * NQB + h]);
        m[h] = r;
    }
}

// B fragments of p . V for the chunk, from the logits in p_sm and the chunk
// maxima mx: p_ht = exp(s_ht - mx_h); bb row r = g NQB + h, pair i (stored
// at i ^ bb_swz(r)) holds the (hi, lo) fp16 pairs of tokens 2i, 2i+1 of
// w = p_ht s_tg for quantized tokens (t < nq) and of w = p_ht for residual
// tokens (nq <= t < n), zero up to the end of the last 16-token slice.
// zw[warp][h][g] = the warp's share of sum over quantized t of p_ht z_tg,
// zw[warp][h][NGV] its share of sum over t of p_ht (when zw_on_p, zw
// overlays p_sm and is written after a barrier).  One thread per token pair; whole CTA, the
// caller's barrier publishes both.
template <int NQB, int NGV>
__device__ __forceinline__ void pv_weights_g(int n, int nq, int i_first, int i_end, int i_step,
                                             const float* p_sm, int ps, const float (&mx)[NQB],
                                             const float* vs, const float* vz, float fv, uint2* bb, int bbs,
                                             float* zw, bool zw_on_p)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float z[NQB][NGV], l[NQB];
#pragma unroll
    for (int h = 0; h < NQB; ++h) {
        l[h] = 0.0f;
#pragma unroll
        for (int gg = 0; gg < NGV; ++gg)
            z[h][gg] = 0.0f;
    }
    for (int i = i_first; i < i_end; i += i_step) {
        const int t = 2 * i;
        float e0[NQB], e1[NQB];
#pragma unroll
        for (int h = 0; h < NQB; ++h) {
            // p_sm rows are even-strided and t is even; entries past n are not read as weights
            const float2 sv = *reinterpret_cast<const float2*>(p_sm + h * ps + t);
            e0[h] = t < n ? expf(sv.x - mx[h]) : 0.0f;
            e1[h] = t + 1 < n ? expf(sv.y - mx[h]) : 0.0f;
            l[h] += e0[h] + e1[h];
        }
        float s0[NGV], s1[NGV];
        if (t < nq) {  // nq is even: t + 1 is quantized too
#pragma unroll
            for (int gg = 0; gg < NGV; ++gg) {
                s0[gg] = vs[t * NGV + gg] * fv;
                s1[gg] = vs[(t + 1) * NGV + gg] * fv;
                const float z0 = vz[t * NGV + gg], z1 = vz[(t + 1) * NGV + gg];
#pragma unroll
                for (int h = 0; h < NQB; ++h)
                    z[h][gg] = fmaf(e0[h], z0, fmaf(e1[h], z1, z[h][gg]));
            }
        } else {
#pragma unroll
            for (int gg = 0; gg < NGV; ++gg)
                s0[gg] = s1[gg] = 1.0f;
        }
#pragma unroll
        for (int h = 0; h < NQB; ++h)
#pragma unroll
            for (int gg = 0; gg < NGV; ++gg) {
                const int r = gg * NQB + h;
                uint2 hl;
                split_hi_lo(e0[h] * s0[gg], e1[h] * s1[gg], hl.x, hl.y);
                bb[r * bbs + (i ^ bb_swz(r))] = hl;
            }
    }
#pragma unroll
    for (int h = 0; h < NQB; ++h) {
#pragma unroll
        for (int gg = 0; gg < NGV; ++gg)
            for (int k = 16; k > 0; k >>= 1)
                z[h][gg] += __shfl_xor_sync(0xffffffffu, z[h][gg], k);
        for (int k = 16; k > 0; k >>= 1)
            l[h] += __shfl_xor_sync(0xffffffffu, l[h], k);
    }
    if (zw_on_p)
        __syncthreads();  // zw overlays p_sm: every thread has read its logits
    if (lane == 0)
#pragma unroll
        for (int h = 0; h < NQB; ++h) {
#pragma unroll
            for (int gg = 0; gg < NGV; ++gg)
                zw[(warp * NQB + h) * (NGV + 1) + gg] = z[h][gg];
            zw[(warp * NQB + h) * (NGV + 1) + NGV] = l[h];
        }
}

// Pairs i_first, i_first + i_step, ... below i_end of the chunk.  Pairs past
// the last token (up to the end of the last 16-token slice) get zero weights.
// Quantized tokens' weights carry the chunk's value weight scale fv
// (weight_scale_pow2 of its largest value scale); pv_unit takes it out again.
template <int NQB>
__device__ __forceinline__ void pv_weights(int n, int nq, int NGv, int i_first, int i_end, int i_step,
                                           const float* p_sm, int ps, const float (&mx)[NQB],
                                           const float* vs, const float* vz, float fv, uint2* bb, int bbs,
                                           float* zw, bool zw_on_p)
{
    switch (NGv) {
    case 1: pv_weights_g<NQB, 1>(n, nq, i_first, i_end, i_step, p_sm, ps, mx, vs, vz, fv, bb, bbs, zw, zw_on_p); break;
    case 2: pv_weights_g<NQB, 2>(n, nq, i_first, i_end, i_step, p_sm, ps, mx, vs, vz, fv, bb, bbs, zw, zw_on_p); break;
    case 4: pv_weights_g<NQB, 4>(n, nq, i_first, i_end, i_step, p_sm, ps, mx, vs, vz, fv, bb, bbs, zw, zw_on_p); break;
    default: pv_weights_g<NQB, 8>(n, nq, i_first, i_end, i_step, p_sm, ps, mx, vs, vz, fv, bb, bbs, zw, zw_on_p); break;
    }
}
// Pairs a chunk of n tokens (nq quantized) needs: through the last residual slice.
__host__ __device__ constexpr int pv_pairs(int n, int nq) { return (nq + ((n - nq + 15) & ~15)) / 2; }

// Splits of the token range across the warps for NSP segment groups.
__host__ __device__ constexpr int pv_splits(int NSP) { return NSP >= kDecodeWarps ? 1 : kDecodeWarps / NSP; }
template <int BITS>
__host__ __device__ constexpr int pv_segs_per_load(int D) { return D / (32 / BITS) / 4 >= 2 ? 2 : 1; }
template <int BITS>
__host__ __device__ constexpr int pv_seg_groups(int D) { return D / (32 / BITS) / 4 / pv_segs_per_load<BITS>(D); }

// p . V_hat for NQB query heads and the channels of segment group sp (SPL
// segments of 8 halves each) with the staged values of the chunk at t_begin
// (vw, val_swz layout) and B fragments of pv_weights (pair i of the chunk at
// bb pair i).  Quantized 16-token slices k = kq, kq + kstep, ...
// below kq_end through ldmatrix.trans; residual slices kr, kr + kstep, ...
// below kr_end (tokens tq_end + 16 kr ...) from the fp16 ring with the raw
// values as A.  Writes o_out[h][d] (no zero terms) for the segment group's
// channels, each entry by exactly one lane.
template <int BITS, int NQB, int D>
__device__ __forceinline__ void pv_unit(const kivi_cache& c, size_t bh, int t_begin, int tq_end,
                                        int t_end, const uint32_t* vw, const uint2* bb, int bbs,
                                        int sp, int kq, int kq_end, int kr, int kr_end,
                                        int kstep, float inv_fv, float* o_out)
{
    using T = ValTile<BITS>;
    const int G = c.G, lgG = ilog2(G), RG = c.R + c.G;
    constexpr int DW = D / T::P, NSEG = DW / 4;
    constexpr int SPL = pv_segs_per_load<BITS>(D);  // segments per ldmatrix (x4: 2, x2: 1)
    const int NGS = cmax(1, T::CS >> lgG);      // groups per segment (1 or 2)
    // hi and lo weights as separate B columns when the (group, head) units
    // take at most four: B column g is unit g / 2, part g & 1
    constexpr bool HL = NQB <= 2;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tg = lane & 3;
    const int unit = HL ? g >> 1 : g, part = g & 1;
    const int gl = cmin(unit / NQB, NGS - 1), hq = unit % NQB;  // clamped; extra columns unused
    // ldmatrix row of this lane: matrix mi = lane / 8 = 2 s + (token half)
    const int mi = lane >> 3, lrow = (lane & 7) + 8 * (mi & 1), lseg = SPL == 2 ? mi >> 1 : 0;
    const int seg0 = sp * SPL;
    float acc[2][T::NT][4];
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int j = 0; j < T::NT; ++j)
            acc[s][j][0] = acc[s][j][1] = acc[s][j][2] = acc[s][j][3] = 0.0f;
    const uint2* bp[2];
    int bx[2];  // bb_swz of the lane's row
    int grp_first[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        grp_first[s] = ((seg0 + s) * T::CS) >> lgG;
        const int r = (grp_first[s] + gl) * NQB + hq;
        bp[s] = bb + (size_t)r * bbs;
        bx[s] = bb_swz(r);
    }
    // swizzled address of this lane's ldmatrix row (val_swz depends on the
    // row within its 8-token group only)
    const uint32_t a0 = smem_addr(vw + (size_t)lrow * DW + val_swz(lrow, seg0 + lseg, NSEG) * 4);
    const uint32_t astep = 16u * DW * 4u;  // one 16-token slice

#pragma unroll 1
    for (int k = kq; k < kq_end; k += kstep) {
        uint32_t R[4];
        if (SPL == 2)
            ldsm_x4_t(R, a0 + k * astep);
        else
            ldsm_x2_t(R, a0 + k * astep);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (s >= SPL)
                break;
            uint2 b01, b23;
            if constexpr (HL) {
                const uint32_t* b32 = reinterpret_cast<const uint32_t*>(bp[s]) + part;
                b01.x = b32[2 * ((k * 8 + tg) ^ bx[s])];
                b23.x = b32[2 * ((k * 8 + 4 + tg) ^ bx[s])];
            } else {
                b01 = bp[s][(k * 8 + tg) ^ bx[s]];
                b23 = bp[s][(k * 8 + 4 + tg) ^ bx[s]];
            }
            const uint32_t Rl = R[2 * s], Rh = R[2 * s + 1];
            const uint32_t Rls = Rl >> T::SHIFT, Rhs = Rh >> T::SHIFT;
#pragma unroll
            for (int j = 0; j < T::NT; ++j) {
                const int m0 = 2 * j, m1 = 2 * j + 1;
                const uint32_t mk0 = half_pair_mask<BITS>(T::bitpos(m0));
                const uint32_t mk1 = half_pair_mask<BITS>(T::bitpos(m1));
                const uint32_t x0 = (T::shifted(m0) ? Rls : Rl) & mk0;
                const uint32_t x1 = (T::shifted(m1) ? Rls : Rl) & mk1;
                const uint32_t x2 = (T::shifted(m0) ? Rhs : Rh) & mk0;
                const uint32_t x3 = (T::shifted(m1) ? Rhs : Rh) & mk1;
                mma_f16(acc[s][j], x0, x1, x2, x3, b01.x, b23.x);
                if constexpr (!HL)
                    mma_f16(acc[s][j], x0, x1, x2, x3, b01.y, b23.y);
            }
        }
    }
    // undo the code scaling and the weight scale before the residual tokens
    // join the sums
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int j = 0; j < T::NT; ++j) {
            const float f0 = code_unscale_bits(T::bitpos(2 * j)) * inv_fv;
            const float f1 = code_unscale_bits(T::bitpos(2 * j + 1)) * inv_fv;
            acc[s][j][0] *= f0;
            acc[s][j][1] *= f0;
            acc[s][j][2] *= f1;
            acc[s][j][3] *= f1;
        }
    // residual tokens: A = (v[t][d], v[t+1][d]) pairs, B = p (hi / lo).
    // The lane's HC channels of a segment are contiguous: one 16 / 8 /
    // 4-byte load per token and segment.
    const int nq2 = (tq_end - t_begin) / 2;  // pair index of the first residual token
#pragma unroll 1
    for (int k = kr; k < kr_end; k += kstep) {
        const int tb = tq_end + k * 16 + 2 * tg;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (s >= SPL)
                break;
            const int ch0 = (seg0 + s) * T::CS + g * T::HC;
            uint32_t X[4][T::NT];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = tb + (i & 1) + 8 * (i >> 1);
                const bool ok = t < t_end;
                const uint16_t* vr = c.vres + (bh * RG + (ok ? t : 0) % RG) * D + ch0;
                if constexpr (T::NT == 4) {
                    const uint4 x = ok ? ld_nc(vr) : make_uint4(0u, 0u, 0u, 0u);
                    X[i][0] = x.x;
                    X[i][1] = x.y;
                    X[i][2] = x.z;
                    X[i][3] = x.w;
                } else if constexpr (T::NT == 2) {
                    const uint2 x = ok ? ldg_checked(reinterpret_cast<const uint2*>(vr)) : make_uint2(0u, 0u);
                    X[i][0] = x.x;
                    X[i][1] = x.y;
                } else {
                    X[i][0] = ok ? ldg_checked(reinterpret_cast<const uint32_t*>(vr)) : 0u;
                }
            }
            uint2 b01, b23;
            if constexpr (HL) {
                const uint32_t* b32 = reinterpret_cast<const uint32_t*>(bp[s]) + part;
                b01.x = b32[2 * ((nq2 + k * 8 + tg) ^ bx[s])];
                b23.x = b32[2 * ((nq2 + k * 8 + 4 + tg) ^ bx[s])];
            } else {
                b01 = bp[s][(nq2 + k * 8 + tg) ^ bx[s]];
                b23 = bp[s][(nq2 + k * 8 + 4 + tg) ^ bx[s]];
            }
#pragma unroll
            for (int j = 0; j < T::NT; ++j) {
                const uint32_t x0 = __byte_perm(X[0][j], X[1][j], 0x5410);
                const uint32_t x1 = __byte_perm(X[0][j], X[1][j], 0x7632);
                const uint32_t x2 = __byte_perm(X[2][j], X[3][j], 0x5410);
                const uint32_t x3 = __byte_perm(X[2][j], X[3][j], 0x7632);
                mma_f16(acc[s][j], x0, x1, x2, x3, b01.x, b23.x);
                if constexpr (!HL)
                    mma_f16(acc[s][j], x0, x1, x2, x3, b01.y, b23.y);
            }
        }
    }

#pragma unroll
    for (int s = 0; s < 2; ++s) {
        if (s >= SPL)
            break;
        const int ch0 = (seg0 + s) * T::CS + g * T::HC;
        if constexpr (HL) {
            // columns 2 tg (hi) and 2 tg + 1 (lo) both belong to unit tg
            const int ugl = tg / NQB, uh = tg % NQB;
            if (ugl < NGS && grp_first[s] + ugl == (ch0 >> lgG)) {
#pragma unroll
                for (int j = 0; j < T::NT; ++j) {
                    o_out[uh * D + ch0 + 2 * j] = acc[s][j][0] + acc[s][j][1];
                    o_out[uh * D + ch0 + 2 * j + 1] = acc[s][j][2] + acc[s][j][3];
                }
            }
        } else {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int u = 2 * tg + cc;
                const int ugl = u / NQB, uh = u % NQB;
                if (ugl >= NGS || grp_first[s] + ugl != (ch0 >> lgG))
                    continue;
#pragma unroll
                for (int j = 0; j < T::NT; ++j) {
                    o_out[uh * D + ch0 + 2 * j] = acc[s][j][cc];
                    o_out[uh * D + ch0 + 2 * j + 1] = acc[s][j][2 + cc];
                }
            }
        }
    }
}

// p . V_hat of the whole chunk by the CTA: each warp takes units (segment
// group, token split) and writes o_part[split] (splits of one segment group
// are different warps).
template <int BITS, int NQB, int D>
__device__ __forceinline__ void pv_chunk(const kivi_cache& c, size_t bh, int TX, int t_begin,
                                         int tq_end, int t_end, const uint32_t* vw, const uint2* bb,
                                         float inv_fv, float* o_part)
{
    constexpr int NSP = pv_seg_groups<BITS>(D);
    constexpr int NSPLIT = pv_splits(NSP);
    const int nq_slices = (tq_end - t_begin) / 16;
    const int nr_slices = (t_end - tq_end + 15) / 16;
    for (int unit = threadIdx.x >> 5; unit < NSP * NSPLIT; unit += kDecodeWarps) {
        const int sp = unit % NSP, split = unit / NSP;
        pv_unit<BITS, NQB, D>(c, bh, t_begin, tq_end, t_end, vw, bb, bb_stride(TX), sp, split, nq_slices,
                              split, nr_slices, NSPLIT, inv_fv, o_part + (size_t)split * NQB * D);
    }
}

// Writes the chunk's partial (o, m, l) for query heads hq0 .. hq0+NQB-1:
// o[h][d] = sum over warps of zs[w][h][group of d] + sum over splits of
// o_part, l[h] = sum over warps of zs[w][h][D/G] (fixed orders: the result
// is deterministic).  Whole CTA, after a barrier that follows pv_chunk.
template <int NQB, int D>
__device__ __forceinline__ void write_partials(int G, int nsplit, const float* o_part,
                                               const float* zs, const float (&m)[NQB], size_t row0,
                                               int nchunks, float* ws_o, float* ws_m, float* ws_l)
{
    constexpr int lgD = ilog2(D);
    const int lgG = ilog2(G), NGv = D >> lgG, zr = NQB * (NGv + 1);
    for (int idx = threadIdx.x; idx < NQB * D; idx += kDecodeThreads) {
        const int h = idx >> lgD, d = idx & (D - 1);
        const int zi = h * (NGv + 1) + (d >> lgG);
        float s = zs[zi];
#pragma unroll
        for (int w = 1; w < kDecodeWarps; ++w)
            s += zs[w * zr + zi];
        for (int sp = 0; sp < nsplit; ++sp)
            s += o_part[(size_t)sp * NQB * D + idx];
        st_checked(ws_o + (row0 + (size_t)h * nchunks) * D + d, s);
    }
#pragma unroll
    for (int h = 0; h < NQB; ++h)
        if (threadIdx.x == h) {
            float l = zs[h * (NGv + 1) + NGv];
#pragma unroll
            for (int w = 1; w < kDecodeWarps; ++w)
                l += zs[w * zr + h * (NGv + 1) + NGv];
            st_checked(ws_m + row0 + (size_t)h * nchunks, m[h]);
            st_checked(ws_l + row0 + (size_t)h * nchunks, l);
        }
}

}  // namespace kivi
