// decode_stream.cuh -- kivi_decode_attention as one persistent, pipelined
// kernel: the decode-time consumer of the KIVI cache (q . K_hat^T, softmax,
// p . V_hat over the packed cache plus the fp16 residual, dequantization
// fused into the operand build; CacheForge README, "How it works").
//
// Work.  The rows of the problem are (sequence b, KV head h, pass) -- one pass
// covers NQB query heads of h's grouped-query set -- and a row of n tokens is
// cut into tiles: ceil(Tq/TS) quantized tiles of TS tokens (the last one
// shorter), then ceil((n - Tq)/RT) residual tiles of RT fp16 tokens.  Both
// kinds move about the same number of bytes.  One CTA runs per SM; CTA i takes
// a contiguous range of the tiles of all rows in order, cut where the running
// weight of the tiles (each tile one unit, each row a fixed extra for its
// start and finish) crosses i/N of the total, so the load is balanced
// whatever the (device-side, ragged) lengths and however many rows a range
// touches.
// A row that lies wholly inside one CTA's range is finished there and its
// output written; a row cut by a range boundary leaves one partial (o, m, l)
// per CTA, merged by decode_stream_combine_kernel.
//
// Pipeline.  A CTA is three warpgroups (setmaxnreg: the two consumer
// warpgroups at 224 registers a thread, the third at 56).  In the third,
// lane 0 of warp 8 issues the key copies of every tile of the range and lane
// 0 of warp 9 the value copies: each waits for a free stage of the ring,
// announces its bytes on the stage's full mbarrier and issues 1-D bulk copies
// (cp.async.bulk, the TMA engine), global to shared -- three per quantized
// tile (packed word-rows, scales, zeros of its side; each a contiguous range
// of its buffer) and one or two per residual tile (the ring slots, which
// wrap at most once).  Warps 0 .. NC-1 are consumers: they take the range's
// tiles in order from a shared counter (each reserves its next tile while it
// computes the current one), wait for the tile's stage, compute the whole
// tile and release the stage.  The query heads of a row are loaded from
// global memory into the warp's scratch when the warp starts a row.  Each
// consumer keeps its own online-softmax state (running maximum m, sums l,
// the weighted value sums) per row segment (the range's tiles of one row);
// when it moves on, it publishes the state to one of two merge buffers, and
// the warp that completes the segment's tile count merges the states and
// writes the row's output (or the CTA's partial for a cut row).
//
// A quantized tile, per consumer warp:
//   1. q . K_hat on the warp-level tensor cores (decode_mma.cuh: codes as
//      fp16 subnormals in the A operand, weights q s as hi / lo fp16 pairs in
//      B, one MMA per 16 x 16 codes), zero terms sum_d q_d z_gd in fp32;
//      the logits go to a per-warp row in shared memory.  The weights carry a
//      power of two f (weight_scale_pow2 of max|q| times the tile's largest
//      key scale) that keeps them normal fp16 numbers, and the logits divide
//      it out.
//   2. the online softmax over the tile's logits: new maximum, rescaling of
//      the state, p = exp(s - m).
//   3. the value weights u = p s f_v (f_v from the tile's largest value
//      scale) as hi / lo fp16 pairs in B-fragment order, and the zero terms
//      sum_t p_t z_tg, then p . V_hat with the codes from ldmatrix.trans.
// A residual tile: q . K on the tensor cores with the fp16 keys as A and the
// fp16 query as B (both exact, fp32 accumulation), the softmax as above, and
// p . V in fp32 FMA over the fp16 values.
//
// Every wait on an mbarrier gives up after two seconds (which only a fault
// elsewhere could cause): it records KIVI_ETIMEOUT in the workspace's status
// word, the outputs of the affected rows are then meaningless, and the CTA
// leaves once the copies it issued have landed (a bounded wait as well).
#pragma once

#include <math.h>

#include "decode_mma.cuh"
#include "kivi_launch.h"

namespace kivi {

// ------------------------------------------------------------------ PTX ---

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return done != 0;
}
// 1-D bulk copy global -> shared, completing `bytes` on the mbarrier.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(b))
                 : "memory");
}
// The same with shared-memory addresses already converted.
__device__ __forceinline__ void bulk_g2s_a(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx_a(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
constexpr uint64_t kStreamWaitNs = 2000000000ull;  // a wait on a stage gives up after 2 s

// Bounds checks of a library built with KIVI_CHECKS defined: a failed check
// records KIVI_ECHECK in the workspace status word (the first failure wins;
// the host clears the word before the launch) and the access it guards is
// skipped.  Without KIVI_CHECKS every check is true and compiles away.
#ifdef KIVI_CHECKS
__device__ __forceinline__ bool kivi_check(bool ok, int* status)
{
    if (!ok)
        atomicCAS(status, KIVI_OK, KIVI_ECHECK);
    return ok;
}
#else
__device__ __forceinline__ bool kivi_check(bool, int*) { return true; }
#endif

// Nanoseconds of the global timer.
__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase of parity `parity` of mbarrier b; false if it has not
// completed within kStreamWaitNs or *abort became set.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* b, uint32_t parity, const volatile int* abort);
// 2^x (ex2.approx: relative error below 2^-22; 2^-inf = 0).  The streamed
// decode keeps its logits in log2 units (the softmax scale times log2 e), so
// every exponential of the softmax is one ex2.
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void named_bar(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* b, uint32_t parity, const volatile int* abort)
{
    if (mbar_try_wait(b, parity))
        return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(b, parity))
            return true;
        if ((it & 63u) == 0 && (*abort || global_ns() - t0 > kStreamWaitNs))
            return false;
    }
}

// ---------------------------------------------------------------- shape ---

__host__ __device__ constexpr int pow2floor(int x) { return x <= 1 ? 1 : 2 * pow2floor(x / 2); }
__host__ __device__ constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }

constexpr int kMaxStreamCTAs = 1024;          // workspace sizing bound on the grid
constexpr int kStreamStaticSmem = 512;        // room left for the kernel's static shared arrays
constexpr int kStreamHeaderFloats = 4;        // workspace header (status word)
constexpr int kStreamMaxStages = 32;          // stages of the ring (the consumed counters are static)

// Compile-time shape of the streamed decode for key / value widths BK / BV,
// NQB query heads per pass, head dimension D and NC consumer warps.  Sizes
// that depend on the group size G (32, 64 or 128) are taken at G = 32, the
// largest.
// Warp roles of the streamed decode: three warpgroups.  Warps 0..7 are the
// consumers (NC of them take tiles, NC <= 8), warp 8 issues the key copies and
// warp 9 the value copies of every stage, warps 10 and 11 only hand their
// registers back.  The block is launched with 168 registers per thread
// (384 threads); the consumer warpgroups then raise theirs to 224 and the
// third lowers its to 56 (setmaxnreg): 2 x 128 x 224 + 128 x 56 = 384 x 168,
// and each SM sub-partition holds two consumer warps and one other
// (2 x 224 + 56 registers a lane, within its 16K).
constexpr int kStreamWarps = 12;
constexpr int kStreamConsumerWarps = 8;
constexpr int kStreamLaunchRegs = 168;
constexpr int kStreamConsumerRegs = 224;
constexpr int kStreamOtherRegs = 56;
static_assert(2 * 128 * kStreamConsumerRegs + 128 * kStreamOtherRegs == 32 * kStreamWarps * kStreamLaunchRegs,
              "the register split uses exactly the registers the block is launched with");
static_assert((2 * kStreamConsumerRegs + kStreamOtherRegs) * 32 <= 16384, "registers of one SM sub-partition");

template <int BK, int BV, int NQB, int D, int NC>
struct StreamCfg {
    using KT = KeyTile<BK, NQB>;
    using VT = ValTile<BV>;
    static constexpr int PK = 32 / BK, PV = 32 / BV;
    static constexpr int TOK = KT::TOK;                // tokens per key warp tile
    static constexpr int DW = D / PV;                  // value words per token
    static constexpr int NSEG = DW / 4;                // 16-byte value segments per token
    static constexpr int SPL = NSEG >= 2 ? 2 : 1;      // segments per ldmatrix
    static constexpr int NTV = VT::NT;                 // value MMA tiles per segment
    static constexpr int NGM = D / 32;                 // statistic groups per row (G = 32)
    static constexpr int CPL = D / 32;                 // residual channels per lane
    // bytes per quantized token (codes and fp32 statistics at G = 32); a
    // quantized stage holds about 16 KB, a residual stage as much
    static constexpr int BPT = D * (BK + BV) / 8 + D / 2;
    static constexpr int TS = cmax(cmax(TOK, 32), pow2floor(16384 / BPT));
    static constexpr int RT = cmax(16, cmin(64, pow2floor(TS * BPT / (4 * D))));
    // stage slot (bytes from the slot start, each region 16-byte aligned)
    static constexpr int KROW = D * 4;                 // key word-row
    static constexpr int KSR = cmax(1, TS / 32);       // key statistic rows
    static constexpr int O_KW = 0;
    static constexpr int O_KS = O_KW + (TS / PK) * KROW;
    static constexpr int O_KZ = O_KS + KSR * D * 4;
    static constexpr int O_VW = O_KZ + KSR * D * 4;
    static constexpr int O_VS = O_VW + TS * DW * 4;
    static constexpr int O_VZ = O_VS + TS * NGM * 4;
    static constexpr int Q_END = O_VZ + TS * NGM * 4;
    static constexpr int RROW = D * 2;                 // residual row
    static constexpr int O_KR = O_KW;
    static constexpr int O_VR = O_KR + RT * RROW;
    static constexpr int R_END = O_VR + RT * RROW;
    static constexpr int SLOT = round_up(cmax(Q_END, R_END), 128);
    // per-consumer scratch (floats): logits / probabilities [NQB][LS]
    // (two floats of padding per 16 tokens), the scaled query [NQB][QWS]
    // and, over it once q . K is done, the value weights [2 parts][UNITS][UTS]
    // fp16 for UB tokens at a time, then the row's query heads [NQB][D] fp16
    static constexpr int LS = TS + TS / 8;
    static constexpr int QWS = D + 4;
    static constexpr int UNITS = NGM * NQB;            // value weight units (group, head)
    static constexpr bool HLV = NQB <= 2;              // value hi / lo in separate B columns
    static constexpr int UF = HLV ? 4 : 8;             // units per B fragment
    static constexpr int UB = UNITS <= 8 ? TS : cmin(TS, 64);
    static constexpr int UTS = UB + 8;                 // halves per weight row
    static constexpr int W_LG = 0;
    static constexpr int W_QW = W_LG + NQB * LS;
    static constexpr int W_UB = W_QW;
    static constexpr int W_Q = round_up(W_UB + cmax(NQB * QWS, UNITS * UTS), 4);
    static constexpr int QPIECES = NQB * D / 8;                  // 16-byte pieces of them
    static constexpr int WARP_FLOATS = W_Q + NQB * D / 2;
    // merge buffer (floats): o [NC][NQB][D], m, l [NC][NQB], z [NC][NQB][NGM];
    // NMB of them, used by row segments in turn: two where a pass holds one
    // or two query heads (rows end often; two still leave a twelfth stage at
    // int2, D = 128), one for four heads, whose buffer is four times larger
    // and whose rows are long enough that segments rarely end close together
    // (the space buys the eighth consumer warp: 69.6 against 75.3 us on
    // K, V [4, 8, 32768, 128] with 32 query heads)
    static constexpr int M_O = 0;
    static constexpr int M_M = M_O + NC * NQB * D;
    static constexpr int M_L = M_M + NC * NQB;
    static constexpr int M_Z = M_L + NC * NQB;
    static constexpr int M_END = round_up(M_Z + NC * NQB * NGM, 4);
    static constexpr int NMB = NQB == 4 ? 1 : 2;
    static constexpr int FIXED_BYTES = 4 * (NC * WARP_FLOATS + NMB * M_END) + kStreamStaticSmem;
    static constexpr int THREADS = 32 * kStreamWarps;
    static_assert(TS % TOK == 0 && TS % 16 == 0 && RT % 16 == 0 && RT <= TS, "tile shape");
    static_assert(UB % 16 == 0 && TS % UB == 0, "weight batches");
    static_assert(UF % NQB == 0, "a fragment holds whole groups");
};

// Stages that fit the shared memory of one SM next to the fixed areas.
constexpr int kStreamSmemBytes = 227 * 1024;  // dynamic + static shared memory of one CTA
template <class C>
__host__ __device__ constexpr int stream_stages()
{
    return cmin((kStreamSmemBytes - C::FIXED_BYTES) / (C::SLOT + 16), kStreamMaxStages);
}

// Consumer warps of the streamed decode for a shape: up to eight, fewer when
// the shared memory would otherwise hold no more stages than consumers --
// every consumer then has a stage and at least one more is in flight.
constexpr int kStreamMaxConsumers = kStreamConsumerWarps;
template <int BK, int BV, int NQB, int D, int NC = kStreamMaxConsumers>
__host__ __device__ constexpr int stream_consumers()
{
    if constexpr (NC <= 1)
        return 1;
    else
        return stream_stages<StreamCfg<BK, BV, NQB, D, NC>>() >= NC + 1 ? NC
                                                                          : stream_consumers<BK, BV, NQB, D, NC - 1>();
}

// Workspace of the streamed decode: header (status word), two partial
// (o, m, l) slots per CTA, and per CTA a descriptor of the row its range
// ends in (kStreamDescInts ints) for the combine kernel.
constexpr int kStreamDescInts = 8;
__host__ __device__ inline size_t stream_partial_floats(int D, int NQB, int ctas)
{
    return (size_t)ctas * 2 * NQB * (D + 2);
}
inline size_t stream_ws_floats(int D, int NQB, int ctas)
{
    return (size_t)kStreamHeaderFloats + stream_partial_floats(D, NQB, ctas) + (size_t)ctas * kStreamDescInts;
}

// ---------------------------------------------------------- tile walker ---

// Position in the row-major sequence of tiles: sequence b, row rr = h NP +
// pass of b, tile j of the row; the rest describes sequence b.
struct Walk {
    int b, rr, j;
    int len, Tq, nq, nt;
};

__device__ __forceinline__ void walk_load(Walk& w, const kivi_cache& c, int TS, int RT)
{
    w.len = c.len[w.b];
    w.Tq = quantized_tokens(w.len, c.G, c.R);
    w.nq = (w.Tq + TS - 1) / TS;
    w.nt = w.nq + (w.len - w.Tq + RT - 1) / RT;
}

__device__ __forceinline__ void walk_next(Walk& w, const kivi_cache& c, int RB, int TS, int RT)
{
    if (++w.j < w.nt)
        return;
    w.j = 0;
    if (++w.rr < RB)
        return;
    w.rr = 0;
    for (++w.b; w.b < c.B; ++w.b) {
        walk_load(w, c, TS, RT);
        if (w.nt > 0)
            return;
    }
}

// Advances the walker by n tiles; returns the number of rows it left (each
// starts a new row segment).  Stops at the end of the sequences.
__device__ __forceinline__ int walk_skip(Walk& w, const kivi_cache& c, int RB, int TS, int RT, int n)
{
    int crossed = 0;
    w.j += n;
    while (w.j >= w.nt && w.b < c.B) {
        w.j -= w.nt;
        ++crossed;
        if (++w.rr < RB)
            continue;
        w.rr = 0;
        for (++w.b; w.b < c.B; ++w.b) {
            walk_load(w, c, TS, RT);
            if (w.nt > 0)
                break;
        }
    }
    return crossed;
}

// Tokens of the current tile: [t0, t0 + n), quantized or residual.
__device__ __forceinline__ bool walk_quant(const Walk& w) { return w.j < w.nq; }
__device__ __forceinline__ int walk_t0(const Walk& w, int TS, int RT)
{
    return w.j < w.nq ? w.j * TS : w.Tq + (w.j - w.nq) * RT;
}
__device__ __forceinline__ int walk_n(const Walk& w, int TS, int RT)
{
    const int t0 = walk_t0(w, TS, RT);
    return w.j < w.nq ? min(TS, w.Tq - t0) : min(RT, w.len - t0);
}


// Exclusive prefix sums of the pairs (v.x, v.y) over the CTA (THREADS
// threads) and their totals; red holds 2 x THREADS / 32 values.
template <int THREADS>
__device__ __forceinline__ longlong2 cta_exscan2(longlong2 v, longlong2& total, long long* red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long x = v.x, y = v.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long ux = __shfl_up_sync(0xffffffffu, x, o);
        const long long uy = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) {
            x += ux;
            y += uy;
        }
    }
    if (lane == 31) {
        red[2 * warp] = x;
        red[2 * warp + 1] = y;
    }
    __syncthreads();
    long long ox = 0, oy = 0, tx = 0, ty = 0;
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) {
        const long long rx = red[2 * w], ry = red[2 * w + 1];
        ox += w < warp ? rx : 0;
        oy += w < warp ? ry : 0;
        tx += rx;
        ty += ry;
    }
    __syncthreads();
    total = make_longlong2(tx, ty);
    return make_longlong2(ox + x - v.x, oy + y - v.y);
}

// CTA range record: first tile (global index) and its position; wend: the
// split weight at the end of that tile's row.
struct RangeStart {
    long long g, wend;
    int b, rr, j;
};

// The split of the tiles among the CTAs weighs each quantized tile
// kStreamTileWeight, each residual tile kStreamResWeight, and each row
// row_extra(NQB) more, put on the row's first tile: starting and finishing a
// row segment (the query load, the state merge over NQB heads, the partial
// tiles) costs a CTA about as much as two tiles per head, so ranges of equal
// tile counts end at different times when their numbers of rows differ (on
// B = 64 ragged rows of 1024-8192 tokens, CTA end times spread from 262 to
// 291 us with equal tile counts).  Measured: a residual tile weighs as much
// as a quantized one (heavier or lighter residual weights were slower).
constexpr int kStreamTileWeight = 8;
constexpr int kStreamResWeight = 8;
__host__ __device__ constexpr int row_extra(int NQB) { return 16 * NQB; }

// A row's tiles for the split: nq quantized, nr residual.
struct RowTiles {
    int nq, nr;
};
__device__ __forceinline__ RowTiles row_tile_counts(int len, const kivi_cache& c, int TS, int RT)
{
    const int Tq = quantized_tokens(len, c.G, c.R);
    return RowTiles{(Tq + TS - 1) / TS, (len - Tq + RT - 1) / RT};
}
template <int NQB>
__device__ __forceinline__ long long row_weight(RowTiles t)
{
    return t.nq + t.nr > 0
               ? (long long)t.nq * kStreamTileWeight + (long long)t.nr * kStreamResWeight + row_extra(NQB)
               : 0;
}
// The tile of a row whose weight interval holds offset off (< the row's
// weight): tile 0 covers the row's extra and its own weight.
template <int NQB>
__device__ __forceinline__ int tile_at(RowTiles t, long long off)
{
    const long long x = off - row_extra(NQB);
    const long long q = (long long)t.nq * kStreamTileWeight;
    const int j = x < q ? (int)(x / kStreamTileWeight) : t.nq + (int)((x - q) / kStreamResWeight);
    return x < 0 ? 0 : j;
}

// Start of CTA k's range and of CTA k+1's (the end), from the device-side
// lengths: two passes over the sequences (totals, then location).  With Wtot
// the weight of all tiles, range k starts at the tile whose weight interval
// holds Wtot k / N (tile 0 of a row covers the row's extra weight and its
// own), so a range may be empty; *total receives Wtot.
template <int THREADS, int NQB>
__device__ __forceinline__ void locate_range(const kivi_cache& c, int RB, int TS, int RT, int k, int N,
                                             RangeStart& r0, RangeStart& r1, long long* red, RangeStart* sh,
                                             long long* total = nullptr)
{
    long long W = 0, NT = 0;
    for (int base = 0; base < c.B; base += THREADS) {
        const int b = base + (int)threadIdx.x;
        const RowTiles t = b < c.B ? row_tile_counts(c.len[b], c, TS, RT) : RowTiles{0, 0};
        longlong2 tot;
        cta_exscan2<THREADS>(make_longlong2(RB * row_weight<NQB>(t), (long long)RB * (t.nq + t.nr)), tot, red);
        W += tot.x;
        NT += tot.y;
    }
    const long long X[2] = {W * k / N, W * (k + 1) / N};
    if (threadIdx.x < 2)
        sh[threadIdx.x] = RangeStart{NT, W, c.B, 0, 0};
    __syncthreads();
    long long ew = 0, et = 0;
    for (int base = 0; base < c.B; base += THREADS) {
        const int b = base + (int)threadIdx.x;
        const RowTiles t = b < c.B ? row_tile_counts(c.len[b], c, TS, RT) : RowTiles{0, 0};
        const int nt = t.nq + t.nr;
        const long long wr = row_weight<NQB>(t);
        longlong2 tot;
        const longlong2 ex = cta_exscan2<THREADS>(make_longlong2(RB * wr, (long long)RB * nt), tot, red);
        const long long xw = ew + ex.x, xt = et + ex.y;
#pragma unroll
        for (int i = 0; i < 2; ++i)
            if (nt > 0 && xw <= X[i] && X[i] < xw + RB * wr) {
                const long long o = X[i] - xw;
                const int rr = (int)(o / wr);
                const int j = tile_at<NQB>(t, o - rr * wr);
                sh[i] = RangeStart{xt + (long long)rr * nt + j, xw + (rr + 1) * wr, b, rr, j};
            }
        ew += tot.x;
        et += tot.y;
    }
    __syncthreads();
    r0 = sh[0];
    r1 = sh[1];
    if (total)
        *total = W;
}

// ------------------------------------------------------- consumer state ---

template <class C, int NQB>
struct ConsumerState {
    float m[NQB];                    // running maxima (of the logits)
    float l[NQB];                    // lane partial sums of exp(s - m)
    float z[NQB][C::NGM];            // lane partial zero terms sum_t p_t z_tg
    float o[C::NSEG][C::NTV][4];     // weighted value sums, MMA layout, in units 1 / fv
    float r[NQB][C::CPL];            // residual weighted sums, channels lane*CPL + i
    float qmax[NQB];                 // max |q| of the row's heads (< 0: not yet known)
    float fv;                        // current value weight scale of o
};

template <class C, int NQB>
__device__ __forceinline__ void state_reset(ConsumerState<C, NQB>& s)
{
#pragma unroll
    for (int h = 0; h < NQB; ++h) {
        s.m[h] = -INFINITY;
        s.l[h] = 0.0f;
        s.qmax[h] = -1.0f;
#pragma unroll
        for (int g = 0; g < C::NGM; ++g)
            s.z[h][g] = 0.0f;
#pragma unroll
        for (int i = 0; i < C::CPL; ++i)
            s.r[h][i] = 0.0f;
    }
#pragma unroll
    for (int sg = 0; sg < C::NSEG; ++sg)
#pragma unroll
        for (int j = 0; j < C::NTV; ++j)
            s.o[sg][j][0] = s.o[sg][j][1] = s.o[sg][j][2] = s.o[sg][j][3] = 0.0f;
    s.fv = 1.0f;
}

__device__ __forceinline__ int lg_phys(int t) { return t + 2 * (t >> 4); }

__device__ __forceinline__ float sel4(const float (&a)[4], int i)
{
    return i == 0 ? a[0] : i == 1 ? a[1] : i == 2 ? a[2] : a[3];
}
template <int N>
__device__ __forceinline__ float seln(const float (&a)[N], int i)
{
    float r = a[0];
#pragma unroll
    for (int k = 1; k < N; ++k)
        r = i == k ? a[k] : r;
    return r;
}

// Value head of the lane's MMA output column pair cc (0, 1) for fragment-
// local units (2 tg + cc without hi / lo columns, tg with them).
template <class C, int NQB>
__device__ __forceinline__ int pv_col_head(int tg, int cc)
{
    return C::HLV ? tg % NQB : (2 * tg + cc) % NQB;
}

// ----------------------------------------------------------- quantized ---

// Warp maximum of non-negative floats: their bit patterns order like
// unsigned integers, so one integer reduction gives it.
__device__ __forceinline__ float warp_max_nonneg(float x)
{
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(x)));
}
// Warp maximum of any floats (NaN excluded): a monotone map to signed
// integers, one integer reduction, and the map back.
__device__ __forceinline__ float warp_max(float x)
{
    const int b = __float_as_int(x);
    const int key = b >= 0 ? b : b ^ 0x7fffffff;
    const int m = __reduce_max_sync(0xffffffffu, key);
    return __int_as_float(m >= 0 ? m : m ^ 0x7fffffff);
}

// Largest statistic of the first n floats at p (a multiple of 4), per warp.
__device__ __forceinline__ float warp_max_stat(const float* p, int n)
{
    const int lane = threadIdx.x & 31;
    float mx = 0.0f;
    for (int i = 4 * lane; i < n; i += 128) {
        const float4 v = *reinterpret_cast<const float4*>(p + i);
        mx = fmaxf(fmaxf(mx, v.x), fmaxf(fmaxf(v.y, v.z), v.w));
    }
    return warp_max_nonneg(mx);
}

// The largest key statistic (first nk floats at pk) and the largest value
// statistic (first nv at pv) of a tile, per warp, each at most MAXK / MAXV
// floats: all loads issued first, tree maxima, one integer reduction each
// (the two chains are independent, so their latencies overlap).
template <int MAXK, int MAXV>
__device__ __forceinline__ void warp_max_stats2(const float* pk, int nk, const float* pv, int nv, float& mk,
                                                float& mv)
{
    constexpr int LK = (MAXK + 127) / 128, LV = (MAXV + 127) / 128;
    const int lane = threadIdx.x & 31;
    float4 k4[LK], v4[LV];
#pragma unroll
    for (int u = 0; u < LK; ++u) {
        const int i = 4 * lane + 128 * u;
        k4[u] = i < nk ? *reinterpret_cast<const float4*>(pk + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < LV; ++u) {
        const int i = 4 * lane + 128 * u;
        v4[u] = i < nv ? *reinterpret_cast<const float4*>(pv + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float a[LK], b[LV];
#pragma unroll
    for (int u = 0; u < LK; ++u)
        a[u] = fmaxf(fmaxf(k4[u].x, k4[u].y), fmaxf(k4[u].z, k4[u].w));
#pragma unroll
    for (int u = 0; u < LV; ++u)
        b[u] = fmaxf(fmaxf(v4[u].x, v4[u].y), fmaxf(v4[u].z, v4[u].w));
#pragma unroll
    for (int w = 1; w < LK; w *= 2)
#pragma unroll
        for (int u = 0; u + w < LK; u += 2 * w)
            a[u] = fmaxf(a[u], a[u + w]);
#pragma unroll
    for (int w = 1; w < LV; w *= 2)
#pragma unroll
        for (int u = 0; u + w < LV; u += 2 * w)
            b[u] = fmaxf(b[u], b[u + w]);
    mk = warp_max_nonneg(a[0]);
    mv = warp_max_nonneg(b[0]);
}

// q . K_hat of one key warp tile (tokens tok0 .. tok0 + TOK of the stage,
// valid below n) into the logit rows lg[h][lg_phys(t)] for valid tokens.
// kst0: the stage's first key statistic row is group kst0; t0: first token
// of the stage in its sequence; fac[h] = sm_scale log2(e) / f_h.
template <int BK, int NQB, int D, class C>
__device__ __forceinline__ void qk_warp_tile(int lgG, int t0, int tok0, int n, const uint8_t* slot,
                                             const float* qw, const float (&fac)[NQB], float* lg)
{
    using T = KeyTile<BK, NQB>;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tg = lane & 3;
    const int wr = g % T::WR, v = g / T::WR;
    const uint32_t soff = (uint32_t)(2 * v * T::NT / T::CPB) * 0x101u;
    const int NGW = cmax(1, T::TOK >> lgG);
    const int unit = T::HL ? g >> 1 : g, part = g & 1;
    const int gi = cmin(unit / NQB, NGW - 1);
    const int hq = unit % NQB;
    const int gi_row = (wr * T::P) >> lgG;
    const int krow = ((t0 + tok0) >> lgG) + gi - (t0 >> lgG);  // stage statistics row of the B column
    const uint4* wrow = reinterpret_cast<const uint4*>(slot + C::O_KW + (tok0 / T::P + wr) * C::KROW);
    const float4* srow = reinterpret_cast<const float4*>(slot + C::O_KS) + krow * (D / 4);
    const float4* zrow = reinterpret_cast<const float4*>(slot + C::O_KZ) + krow * (D / 4);
    const float4* qrow = reinterpret_cast<const float4*>(qw + hq * C::QWS);

    float acc[T::NT][4];
#pragma unroll
    for (int j = 0; j < T::NT; ++j)
        acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
    float zacc = 0.0f;
    // two channel blocks per iteration: a fully unrolled loop overflows the
    // instruction cache next to the other phases
#pragma unroll 2
    for (int s = 0; s < D / 16; ++s) {
        const int cidx = 2 * tg + (s & 1) + 8 * (s >> 1);  // 16-byte chunk: channels 4 cidx .. 4 cidx + 3
        const uint4 W = wrow[cidx];
        const float4 S = srow[cidx];
        const float4 Z = zrow[cidx];
        const float4 Q = qrow[cidx];
        zacc = fmaf(Q.x, Z.x, zacc);
        zacc = fmaf(Q.y, Z.y, zacc);
        zacc = fmaf(Q.z, Z.z, zacc);
        zacc = fmaf(Q.w, Z.w, zacc);
        uint32_t bh0, bl0, bh1, bl1;
        if constexpr (T::HL) {
            bh0 = split_part(Q.x * S.x, Q.y * S.y, part);
            bh1 = split_part(Q.z * S.z, Q.w * S.w, part);
        } else {
            split_hi_lo(Q.x * S.x, Q.y * S.y, bh0, bl0);
            split_hi_lo(Q.z * S.z, Q.w * S.w, bh1, bl1);
        }
#pragma unroll
        for (int j = 0; j < T::NT; ++j) {
            const uint32_t sa = ((uint32_t)T::ya(j) | ((uint32_t)(4 + T::ya(j)) << 8)) + soff;
            const uint32_t sb = ((uint32_t)T::yb(j) | ((uint32_t)(4 + T::yb(j)) << 8)) + soff;
            const uint32_t ma = half_pair_mask<BK>(T::pa(j)), mb = half_pair_mask<BK>(T::pb(j));
            const uint32_t a0 = __byte_perm(W.x, W.y, sa) & ma;
            const uint32_t a1 = __byte_perm(W.x, W.y, sb) & mb;
            const uint32_t a2 = __byte_perm(W.z, W.w, sa) & ma;
            const uint32_t a3 = __byte_perm(W.z, W.w, sb) & mb;
            mma_f16(acc[j], a0, a1, a2, a3, bh0, bh1);
            if constexpr (!T::HL)
                mma_f16(acc[j], a0, a1, a2, a3, bl0, bl1);
        }
    }
    zacc += __shfl_xor_sync(0xffffffffu, zacc, 1);
    zacc += __shfl_xor_sync(0xffffffffu, zacc, 2);
    const float zc0 = __shfl_sync(0xffffffffu, zacc, 8 * tg);
    const float zc1 = __shfl_sync(0xffffffffu, zacc, 8 * tg + 4);
    if (tok0 + wr * T::P >= n)
        return;
    const int tbase = tok0 + wr * T::P + 2 * v * T::NT;
    if constexpr (T::HL) {
        const int h = tg % NQB;
        if (tg / NQB == gi_row) {
            const float f = seln<NQB>(fac, h);
            float* row = lg + h * C::LS;
#pragma unroll
            for (int j = 0; j < T::NT; ++j) {
                const float s0 = f * fmaf(code_unscale_bits(T::pa(j)), acc[j][0] + acc[j][1], zc0);
                const float s1 = f * fmaf(code_unscale_bits(T::pb(j)), acc[j][2] + acc[j][3], zc0);
                *reinterpret_cast<float2*>(row + lg_phys(tbase + 2 * j)) = make_float2(s0, s1);
            }
        }
    } else {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int u = 2 * tg + cc;
            if (u / NQB != gi_row)
                continue;
            const int h = u % NQB;
            const float f = seln<NQB>(fac, h);
            const float zc = cc ? zc1 : zc0;
            float* row = lg + h * C::LS;
#pragma unroll
            for (int j = 0; j < T::NT; ++j) {
                const float s0 = f * fmaf(code_unscale_bits(T::pa(j)), acc[j][cc], zc);
                const float s1 = f * fmaf(code_unscale_bits(T::pb(j)), acc[j][2 + cc], zc);
                *reinterpret_cast<float2*>(row + lg_phys(tbase + 2 * j)) = make_float2(s0, s1);
            }
        }
    }
}

// Online softmax over the n logits of the stage in lg: new maxima, the
// state's rescaling (alpha for the sums, alpha * fv_new / fv for o), and
// p = exp(s - m) written over the logits.  Whole warp; lg is published by the
// caller's __syncwarp and published again here.
template <class C, int NQB>
__device__ __forceinline__ void softmax_stage(ConsumerState<C, NQB>& st, float* lg, int n, float fv_new)
{
    const int lane = threadIdx.x & 31;
    float mt[NQB];
#pragma unroll
    for (int h = 0; h < NQB; ++h)
        mt[h] = -INFINITY;
#pragma unroll
    for (int u = 0; u < (C::TS + 63) / 64; ++u) {
        const int t = 2 * (lane + 32 * u);
        if (t < n) {
#pragma unroll
            for (int h = 0; h < NQB; ++h) {
                const float2 x = *reinterpret_cast<const float2*>(lg + h * C::LS + lg_phys(t));
                mt[h] = fmaxf(mt[h], t + 1 < n ? fmaxf(x.x, x.y) : x.x);
            }
        }
    }
    float alpha[NQB];
    bool same = fv_new == st.fv;  // no rescaling at all: common once the maxima settle
#pragma unroll
    for (int h = 0; h < NQB; ++h) {
        mt[h] = warp_max(mt[h]);
        const float mn = fmaxf(st.m[h], mt[h]);
        alpha[h] = ex2(st.m[h] - mn);  // 0 while the state is empty; 1 if the maximum stays
        same = same && alpha[h] == 1.0f;
        st.m[h] = mn;
    }
    if (!same) {  // warp-uniform: every lane holds the same maxima and scales
#pragma unroll
        for (int h = 0; h < NQB; ++h) {
            st.l[h] *= alpha[h];
#pragma unroll
            for (int g = 0; g < C::NGM; ++g)
                st.z[h][g] *= alpha[h];
#pragma unroll
            for (int i = 0; i < C::CPL; ++i)
                st.r[h][i] *= alpha[h];
        }
        // o is kept in units of 1 / fv: rescale to the new value weight scale
        const float ratio = fv_new * __frcp_rn(st.fv);  // exact: powers of two
        st.fv = fv_new;
        const int tg = lane & 3;
        const float ro0 = seln<NQB>(alpha, pv_col_head<C, NQB>(tg, 0)) * ratio;
        const float ro1 = seln<NQB>(alpha, pv_col_head<C, NQB>(tg, 1)) * ratio;
#pragma unroll
        for (int sg = 0; sg < C::NSEG; ++sg)
#pragma unroll
            for (int j = 0; j < C::NTV; ++j) {
                st.o[sg][j][0] *= ro0;
                st.o[sg][j][1] *= ro1;
                st.o[sg][j][2] *= ro0;
                st.o[sg][j][3] *= ro1;
            }
    }
#pragma unroll
    for (int u = 0; u < (C::TS + 63) / 64; ++u) {
        const int t = 2 * (lane + 32 * u);
        if (t < n) {
#pragma unroll
            for (int h = 0; h < NQB; ++h) {
                float2* px = reinterpret_cast<float2*>(lg + h * C::LS + lg_phys(t));
                const float2 x = *px;
                const float p0 = ex2(x.x - st.m[h]);
                const float p1 = t + 1 < n ? ex2(x.y - st.m[h]) : 0.0f;
                st.l[h] += p0 + p1;
                *px = make_float2(p0, p1);
            }
        }
    }
    __syncwarp();
}

// N consecutive floats from shared memory at p (aligned to 4 N bytes, up to
// 16), in 16-byte pieces where N allows.
template <int N>
__device__ __forceinline__ void load_vec(float (&v)[N], const float* p)
{
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const float4 x = *reinterpret_cast<const float4*>(p + i);
            v[i] = x.x;
            v[i + 1] = x.y;
            v[i + 2] = x.z;
            v[i + 3] = x.w;
        }
    } else if constexpr (N == 2) {
        const float2 x = *reinterpret_cast<const float2*>(p);
        v[0] = x.x;
        v[1] = x.y;
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i)
            v[i] = p[i];
    }
}

// Value weights of the stage's tokens [tb, tb + UB) below n: for unit
// (group gg, head h) = gg NQB + h, ub[part][unit][t - tb] holds the hi
// (part 0) and lo (part 1) fp16 terms of u = p_ht s_tg fv, and the lane's
// zero terms gather p_ht z_tg.  Token pairs per lane.
template <class C, int NQB, int NG>
__device__ __forceinline__ void value_weights(ConsumerState<C, NQB>& st, const float* lg, const uint8_t* slot,
                                              int tb, int n, float fv, uint16_t* ub)
{
    const int lane = threadIdx.x & 31;
    const float* vs = reinterpret_cast<const float*>(slot + C::O_VS);
    const float* vz = reinterpret_cast<const float*>(slot + C::O_VZ);
    uint32_t* ub32 = reinterpret_cast<uint32_t*>(ub);
#pragma unroll
    for (int u = 0; u < (C::UB + 63) / 64; ++u) {
        const int i = lane + 32 * u;  // pair within the batch
        const int t = tb + 2 * i;
        if (2 * i >= C::UB || t >= n)
            continue;
        // statistics of tokens t, t + 1: 2 NG consecutive floats, read as
        // vectors (scalar reads at a stride of 2 NG floats conflict on banks)
        float s01[2 * NG], z01[2 * NG];
        load_vec<2 * NG>(s01, vs + t * NG);
        load_vec<2 * NG>(z01, vz + t * NG);
        float s0[NG], s1[NG], z0[NG], z1[NG];
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) {
            s0[gg] = s01[gg] * fv;
            s1[gg] = s01[NG + gg] * fv;
            z0[gg] = z01[gg];
            z1[gg] = z01[NG + gg];
        }
#pragma unroll
        for (int h = 0; h < NQB; ++h) {
            const float2 p = *reinterpret_cast<const float2*>(lg + h * C::LS + lg_phys(t));
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) {
                st.z[h][gg] = fmaf(p.x, z0[gg], fmaf(p.y, z1[gg], st.z[h][gg]));
                uint32_t hi, lo;
                split_hi_lo(p.x * s0[gg], p.y * s1[gg], hi, lo);
                const int unit = gg * NQB + h;
                ub32[(unit * C::UTS) / 2 + i] = hi;
                ub32[((C::UNITS + unit) * C::UTS) / 2 + i] = lo;
            }
        }
    }
}

// p . V_hat of the 16-token slices k0 .. k1 of the stage (weights of the
// batch at tb in ub), accumulated into st.o.
template <int BV, int NQB, int D, class C>
__device__ __forceinline__ void pv_slices(ConsumerState<C, NQB>& st, int lgG, const uint8_t* slot,
                                          const uint16_t* ub, int tb, int k0, int k1)
{
    using VT = ValTile<BV>;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tg = lane & 3;
    const int mi = lane >> 3, lrow = (lane & 7) + 8 * (mi & 1), lseg = C::SPL == 2 ? mi >> 1 : 0;
    const uint32_t vbase = smem_addr(slot + C::O_VW) + (uint32_t)(lrow * C::DW * 4 + lseg * 16);
    const uint32_t* ub32 = reinterpret_cast<const uint32_t*>(ub);
    // B column of this lane: unit within a fragment and weight part
    const int ucol = C::HLV ? g >> 1 : g, part = g & 1;
#pragma unroll 2
    for (int k = k0; k < k1; ++k) {
        const int pi = (16 * k - tb) / 2 + tg;  // pair index of tokens 2 tg, 2 tg + 1 of the slice
#pragma unroll
        for (int sp = 0; sp < C::NSEG / C::SPL; ++sp) {
            uint32_t R[4];
            const uint32_t addr = vbase + (uint32_t)(16 * k * C::DW * 4 + sp * C::SPL * 16);
            if constexpr (C::SPL == 2)
                ldsm_x4_t(R, addr);
            else
                ldsm_x2_t(R, addr);
#pragma unroll
            for (int s2 = 0; s2 < C::SPL; ++s2) {
                const int sg = sp * C::SPL + s2;
                // first unit of the segment's fragment: its first group times NQB, rounded to a fragment
                const int gfirst = (sg * VT::CS) >> lgG;
                const int frag0 = (gfirst * NQB) / C::UF * C::UF;
                const int unit = frag0 + ucol;
                uint32_t b0, b1, c0 = 0, c1 = 0;
                if constexpr (C::HLV) {
                    const int row = (part * C::UNITS + unit) * C::UTS / 2;
                    b0 = ub32[row + pi];
                    b1 = ub32[row + pi + 4];
                } else {
                    const int rh = unit * C::UTS / 2, rl = (C::UNITS + unit) * C::UTS / 2;
                    b0 = ub32[rh + pi];
                    b1 = ub32[rh + pi + 4];
                    c0 = ub32[rl + pi];
                    c1 = ub32[rl + pi + 4];
                }
                const uint32_t Rl = R[2 * s2], Rh = R[2 * s2 + 1];
                const uint32_t Rls = Rl >> VT::SHIFT, Rhs = Rh >> VT::SHIFT;
#pragma unroll
                for (int j = 0; j < VT::NT; ++j) {
                    const int m0 = 2 * j, m1 = 2 * j + 1;
                    const uint32_t mk0 = half_pair_mask<BV>(VT::bitpos(m0));
                    const uint32_t mk1 = half_pair_mask<BV>(VT::bitpos(m1));
                    const uint32_t x0 = (VT::shifted(m0) ? Rls : Rl) & mk0;
                    const uint32_t x1 = (VT::shifted(m1) ? Rls : Rl) & mk1;
                    const uint32_t x2 = (VT::shifted(m0) ? Rhs : Rh) & mk0;
                    const uint32_t x3 = (VT::shifted(m1) ? Rhs : Rh) & mk1;
                    mma_f16(st.o[sg][j], x0, x1, x2, x3, b0, b1);
                    if constexpr (!C::HLV)
                        mma_f16(st.o[sg][j], x0, x1, x2, x3, c0, c1);
                }
            }
        }
    }
    (void)D;
}

// --------------------------------------------------------------- residual ---

// q . K of a residual stage (n fp16 tokens, padded rows) on the tensor cores:
// A = the keys (ldmatrix), B = the row's fp16 query heads (column h = head
// h, qrow in the warp's scratch),
// logits sl2 q . k into lg (sl2 = sm_scale log2 e).
template <int NQB, int D, class C>
__device__ __forceinline__ void qk_residual_stage(const uint8_t* slot, const uint16_t* qrow, int n, float sl2,
                                                  float* lg)
{
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tg = lane & 3;
    const int mi = lane >> 3, lrow = (lane & 7) + 8 * (mi & 1), lch = mi >> 1;
    const uint32_t kb = smem_addr(slot + C::O_KR) + (uint32_t)(lrow * C::RROW + lch * 16);
    const uint16_t* qh = qrow + (g < NQB ? g : 0) * D;
#pragma unroll 1
    for (int mt = 0; mt < (n + 15) / 16; ++mt) {
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t A[4];
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(A[0]), "=r"(A[1]), "=r"(A[2]), "=r"(A[3])
                         : "r"(kb + (uint32_t)(mt * 16 * C::RROW + ks * 32)));
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(qh + 16 * ks + 2 * tg);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(qh + 16 * ks + 8 + 2 * tg);
            mma_f16(acc, A[0], A[1], A[2], A[3], b0, b1);
        }
        // rows g, g + 8 (tokens), columns 2 tg, 2 tg + 1 (heads)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int h = 2 * tg + cc;
            if (h < NQB) {
                const int t0 = 16 * mt + g, t1 = t0 + 8;
                if (t0 < n)
                    lg[h * C::LS + lg_phys(t0)] = sl2 * acc[cc];
                if (t1 < n)
                    lg[h * C::LS + lg_phys(t1)] = sl2 * acc[2 + cc];
            }
        }
    }
}

// p . V of a residual stage in fp32: the lane's channels lane*CPL .. +CPL-1.
template <int NQB, int D, class C>
__device__ __forceinline__ void pv_residual_stage(ConsumerState<C, NQB>& st, const uint8_t* slot, int n,
                                                  const float* lg)
{
    const int lane = threadIdx.x & 31;
    const uint8_t* vr = slot + C::O_VR + lane * C::CPL * 2;
#pragma unroll 2
    for (int t = 0; t < n; ++t) {
        uint16_t v[C::CPL];
        if constexpr (C::CPL == 4) {
            const uint2 x = *reinterpret_cast<const uint2*>(vr + t * C::RROW);
            v[0] = (uint16_t)x.x;
            v[1] = (uint16_t)(x.x >> 16);
            v[2] = (uint16_t)x.y;
            v[3] = (uint16_t)(x.y >> 16);
        } else {
#pragma unroll
            for (int i = 0; i < C::CPL; ++i)
                v[i] = reinterpret_cast<const uint16_t*>(vr + t * C::RROW)[i];
        }
#pragma unroll
        for (int h = 0; h < NQB; ++h) {
            const float p = lg[h * C::LS + lg_phys(t)];
#pragma unroll
            for (int i = 0; i < C::CPL; ++i)
                st.r[h][i] = fmaf(p, __half2float(__ushort_as_half(v[i])), st.r[h][i]);
        }
    }
}

// ------------------------------------------------------------------ merge ---

// Publishes the warp's state for the row segment in the merge area: o (the
// MMA-layout sums times their code and value scales, plus the residual sums),
// the zero terms per (head, group), m and the warp's l.
template <int BV, int NQB, int D, class C>
__device__ __forceinline__ void state_publish(const ConsumerState<C, NQB>& st, int lgG, int cw, float* mb)
{
    using VT = ValTile<BV>;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tg = lane & 3;
    float* mo = mb + C::M_O + cw * NQB * D;
    const float invfv = __frcp_rn(st.fv);
    // each (head, channel) of the MMA layout is held by exactly one lane
#pragma unroll
    for (int sg = 0; sg < C::NSEG; ++sg) {
        const int ch0 = sg * VT::CS + g * VT::HC;
        const int grp = ch0 >> lgG;
        const int gfirst = (sg * VT::CS) >> lgG;
        const int frag0 = (gfirst * NQB) / C::UF * C::UF;
#pragma unroll
        for (int cc = 0; cc < (C::HLV ? 1 : 2); ++cc) {
            const int unit = frag0 + (C::HLV ? tg : 2 * tg + cc);
            if (unit / NQB != grp)
                continue;
            const int h = unit % NQB;
#pragma unroll
            for (int j = 0; j < VT::NT; ++j) {
                const float f0 = code_unscale_bits(VT::bitpos(2 * j)) * invfv;
                const float f1 = code_unscale_bits(VT::bitpos(2 * j + 1)) * invfv;
                float a, b;
                if constexpr (C::HLV) {
                    a = st.o[sg][j][0] + st.o[sg][j][1];
                    b = st.o[sg][j][2] + st.o[sg][j][3];
                } else {
                    a = st.o[sg][j][cc];
                    b = st.o[sg][j][2 + cc];
                }
                mo[h * D + ch0 + 2 * j] = a * f0;
                mo[h * D + ch0 + 2 * j + 1] = b * f1;
            }
        }
    }
    __syncwarp();
#pragma unroll
    for (int h = 0; h < NQB; ++h)
#pragma unroll
        for (int i = 0; i < C::CPL; ++i)
            mo[h * D + lane * C::CPL + i] += st.r[h][i];
    float* mz = mb + C::M_Z + cw * NQB * C::NGM;
#pragma unroll
    for (int h = 0; h < NQB; ++h) {
        float l = st.l[h];
#pragma unroll
        for (int k = 16; k > 0; k >>= 1)
            l += __shfl_xor_sync(0xffffffffu, l, k);
#pragma unroll
        for (int gg = 0; gg < C::NGM; ++gg) {
            float z = st.z[h][gg];
#pragma unroll
            for (int k = 16; k > 0; k >>= 1)
                z += __shfl_xor_sync(0xffffffffu, z, k);
            if (lane == 0)
                mz[h * C::NGM + gg] = z;
        }
        if (lane == 0) {
            mb[C::M_M + cw * NQB + h] = st.m[h];
            mb[C::M_L + cw * NQB + h] = l;
        }
    }
}

// ------------------------------------------------------- one quantized stage ---

// Tokens [t0, t0 + n) of a quantized stage, by one consumer warp (qh: the
// row's NQB query heads, fp16, in the warp's scratch): weight
// scales (keys from max|q| and the largest key scale, values from the largest
// value scale, valid rows only), q . K_hat into the logit rows, the online
// softmax, then the value weights and p . V_hat in batches of UB tokens.
// FULL: n == TS, so that every loop bound and mask is a constant.
template <int BK, int BV, int NQB, int D, class C, bool FULL>
__device__ __forceinline__ void consume_quant(ConsumerState<C, NQB>& st, const uint8_t* sl, const uint16_t* qh,
                                              int t0, int n_rt, int lgG, float sl2, float* lg, float* qw,
                                              uint16_t* ub)
{
    const int lane = threadIdx.x & 31;
    const int n = FULL ? C::TS : n_rt;
    const int NG = D >> lgG;
    const int ngr = ((t0 + n - 1) >> lgG) - (t0 >> lgG) + 1;
    float smax_k, smax_v;
    warp_max_stats2<C::KSR * D, C::TS * C::NGM>(reinterpret_cast<const float*>(sl + C::O_KS), ngr * D,
                                               reinterpret_cast<const float*>(sl + C::O_VS), n * NG, smax_k,
                                               smax_v);
    float fac[NQB];
#pragma unroll
    for (int hh = 0; hh < NQB; ++hh) {
        if (st.qmax[hh] < 0.0f) {
            float mx = 0.0f;
#pragma unroll
            for (int d = lane; d < D; d += 32)
                mx = fmaxf(mx, fabsf(__half2float(__ushort_as_half(qh[hh * D + d]))));
            st.qmax[hh] = warp_max_nonneg(mx);
        }
        const float fk = weight_scale_pow2(st.qmax[hh] * smax_k);
        fac[hh] = sl2 * __frcp_rn(fk);
#pragma unroll
        for (int d = lane; d < D; d += 32)
            qw[hh * C::QWS + d] = __half2float(__ushort_as_half(qh[hh * D + d])) * fk;
    }
    __syncwarp();
#pragma unroll 1
    for (int tok0 = 0; tok0 < n; tok0 += C::TOK)
        qk_warp_tile<BK, NQB, D, C>(lgG, t0, tok0, n, sl, qw, fac, lg);
    __syncwarp();
    softmax_stage<C, NQB>(st, lg, n, weight_scale_pow2(smax_v));
#pragma unroll 1
    for (int tb = 0; tb < n; tb += C::UB) {
        switch (NG) {
        case 1: value_weights<C, NQB, 1>(st, lg, sl, tb, n, st.fv, ub); break;
        case 2: value_weights<C, NQB, 2>(st, lg, sl, tb, n, st.fv, ub); break;
        case 4: value_weights<C, NQB, cmin(4, C::NGM)>(st, lg, sl, tb, n, st.fv, ub); break;
        default: value_weights<C, NQB, C::NGM>(st, lg, sl, tb, n, st.fv, ub); break;
        }
        __syncwarp();
        pv_slices<BV, NQB, D, C>(st, lgG, sl, ub, tb, tb / 16, min(n, tb + C::UB) / 16);
        __syncwarp();
    }
}

// ---------------------------------------------------------------- kernel ---

template <int BK, int BV, int NQB, int D, int NC>
__global__ void __launch_bounds__(32 * kStreamWarps, 1)
decode_stream_kernel(const kivi_cache c, const uint16_t* __restrict__ q, int Hq, float sm_scale,
                     float* __restrict__ out, float* __restrict__ ws)
{
    using C = StreamCfg<BK, BV, NQB, D, NC>;
    constexpr int ns = stream_stages<C>();  // stages of the ring
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ long long red[2 * (C::THREADS / 32)];
    __shared__ RangeStart sh_range[2];
    __shared__ int abort_flag;
    // per merge buffer: warps published (bit mask), tiles published, last segment merged
    __shared__ int pmask[C::NMB], ptiles[C::NMB], merged[C::NMB];
    __shared__ unsigned long long next_tile;  // the consumers' tile counter
    __shared__ int consumed[kStreamMaxStages];  // tiles finished per slot

    // Launched as a programmatic dependent: the CTAs may be scheduled while
    // the previous kernel of the stream drains, and wait here for its
    // results before reading anything.  The combine kernel may start once
    // every CTA of this grid is running; it waits for this grid's results in
    // its own griddepcontrol.wait.
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NQ = Hq / c.H, NP = NQ / NQB, RB = c.H * NP;
    const float sl2 = sm_scale * 1.44269504088896341f;  // logits in log2 units
    const int lgG = ilog2(c.G);
    uint8_t* slots = smem;
    float* wscr = reinterpret_cast<float*>(smem + (size_t)ns * C::SLOT);
    float* mbuf = wscr + NC * C::WARP_FLOATS;
    uint64_t* full = reinterpret_cast<uint64_t*>(mbuf + C::NMB * C::M_END);
    uint64_t* empty = full + ns;
    int* wsi = reinterpret_cast<int*>(ws);

    RangeStart r0, r1;
    long long W = 0;  // split weight of all tiles
    locate_range<C::THREADS, NQB>(c, RB, C::TS, C::RT, blockIdx.x, gridDim.x, r0, r1, red, sh_range, &W);
    // zero outputs of empty sequences b = blockIdx.x mod gridDim.x (no tile writes them)
    for (int b = blockIdx.x; b < c.B; b += gridDim.x)
        if (c.len[b] == 0)
            for (int x = threadIdx.x; x < Hq * D; x += C::THREADS)
                out[(size_t)b * Hq * D + x] = 0.0f;
    if (threadIdx.x == 0) {
        // The row in which this range ends, for the combine kernel: cut (the
        // range ends inside it and holds its first tile), its sequence and
        // row, the partial slot of this CTA's piece, and the last range with
        // a piece: the last k whose split point W k / N lies before the
        // row's end weight r1.wend.
        int* dsc = wsi + kStreamHeaderFloats + stream_partial_floats(D, NQB, gridDim.x) +
                   (size_t)blockIdx.x * kStreamDescInts;
        const long long g0 = r0.g, g1 = r1.g, row_first = g1 - r1.j;
        const bool cut = g1 > g0 && r1.j != 0 && r1.b < c.B && row_first >= g0;
        int last = 0;
        if (cut)
            last = (int)min((long long)gridDim.x - 1, (r1.wend * gridDim.x - 1) / W);
        dsc[0] = cut ? 1 : 0;
        dsc[1] = r1.b;
        dsc[2] = r1.rr;
        dsc[3] = row_first == g0 ? 0 : 1;
        dsc[4] = last;
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full[s], 2);  // the key and the value producer
            mbar_init(&empty[s], 1);
            consumed[s] = 0;
        }
        mbar_fence_init();
        abort_flag = 0;
        for (int i = 0; i < C::NMB; ++i) {
            pmask[i] = 0;
            ptiles[i] = 0;
            merged[i] = i - C::NMB;
        }
        next_tile = 0ull;
#ifndef KIVI_CHECKS
        if (blockIdx.x == 0)
            wsi[0] = KIVI_OK;  // status word: KIVI_ETIMEOUT if a bounded wait gives up
#endif
    }
    __syncthreads();
    const long long ntiles = r1.g - r0.g;
    if (ntiles <= 0) {
        // an empty range inside a cut row: its slot 0 holds no piece, which
        // the combine reads as the maximum -inf
        if (threadIdx.x < NQB && kivi_check((int)blockIdx.x < kMaxStreamCTAs, wsi))
            ws[kStreamHeaderFloats + (size_t)blockIdx.x * 2 * NQB * (D + 2) + NQB * D + threadIdx.x] = -INFINITY;
        return;
    }
    Walk w0{r0.b, r0.rr, r0.j, 0, 0, 0, 0};
    walk_load(w0, c, C::TS, C::RT);

    if (warp >= kStreamConsumerWarps) {
        // the third warpgroup hands registers back (every warp of it, before
        // any leaves)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kStreamOtherRegs));
        // ----------------------------------------------------- producers
        // Lane 0 of warp 8 issues the key copies of every stage, lane 0 of
        // warp 9 the value copies (three bulk copies each per quantized
        // stage); each announces its own bytes on the stage's full barrier.
        // The issuing thread's own latency per copy bounds the stream, hence
        // two issuers, row base pointers formed once per row, 32-bit offsets
        // inside a row and shared-memory addresses kept converted.
        if (warp >= kStreamConsumerWarps + 2 || lane != 0)
            return;
        const bool kp = warp == kStreamConsumerWarps;  // the key producer
        Walk w = w0;
        int slot = 0;
        uint32_t round = 0;
        long long issued = 0;
        const int NG = D >> lgG;
        const int RG = c.R + c.G;
        const uint32_t s_slots = smem_addr(slots), s_full = smem_addr(full);
        const int32_t* kq_r = nullptr;
        const int32_t* vq_r = nullptr;
        const float *ks_r = nullptr, *kz_r = nullptr, *vs_r = nullptr, *vz_r = nullptr;
        const uint16_t *kr_r = nullptr, *vr_r = nullptr;
        bool new_row = true;
        for (long long k = 0; k < ntiles; ++k) {
            // the empty barrier of a slot completes once per tile taken from
            // it, in order, so its phase never runs more than one ahead
            if (k >= ns && !mbar_wait_bounded(&empty[slot], (round & 1u) ^ 1u, &abort_flag)) {
                atomicExch(&abort_flag, 1);
                atomicExch(wsi, KIVI_ETIMEOUT);
                break;
            }
            if (new_row) {
                const size_t bh = (size_t)w.b * c.H + w.rr / NP;
                kq_r = c.kq + bh * (size_t)(c.Tmax / C::PK) * D;
                ks_r = c.kscale + bh * (size_t)(c.Tmax >> lgG) * D;
                kz_r = c.kzero + bh * (size_t)(c.Tmax >> lgG) * D;
                vq_r = c.vq + bh * (size_t)c.Tmax * C::DW;
                vs_r = c.vscale + bh * (size_t)c.Tmax * NG;
                vz_r = c.vzero + bh * (size_t)c.Tmax * NG;
                kr_r = c.kres + bh * (size_t)RG * D;
                vr_r = c.vres + bh * (size_t)RG * D;
            }
            const uint32_t sb = s_slots + (uint32_t)slot * C::SLOT;
            const uint32_t bar = s_full + (uint32_t)slot * 8u;
            if (w.j < w.nq) {
                const int t0 = w.j * C::TS, n = min(C::TS, w.Tq - t0);
                const int g0 = t0 >> lgG, ngr = ((t0 + n - 1) >> lgG) - g0 + 1;
                const uint32_t bw = (uint32_t)(n / C::PK) * (D * 4), bs = (uint32_t)ngr * (D * 4);
                const uint32_t bv = (uint32_t)n * (C::DW * 4), bz = (uint32_t)(n * NG) * 4u;
                // the tile lies in the row's quantized tokens and in Tmax, each copy in its region
                if (!kivi_check(w.b < c.B && w.rr < RB && t0 >= 0 && n > 0 && t0 + n <= w.Tq &&
                                    w.Tq <= c.Tmax && t0 % C::PK == 0 && n % C::PK == 0 &&
                                    g0 + ngr <= (c.Tmax >> lgG) && C::O_KW + bw <= (uint32_t)C::O_KS &&
                                    C::O_KS + bs <= (uint32_t)C::O_KZ && C::O_KZ + bs <= (uint32_t)C::O_VW &&
                                    C::O_VW + bv <= (uint32_t)C::O_VS && C::O_VS + bz <= (uint32_t)C::O_VZ &&
                                    C::O_VZ + bz <= (uint32_t)C::SLOT,
                                wsi)) {
                    mbar_arrive(&full[slot]);  // the stage completes without data
                } else if (kp) {
                    mbar_arrive_tx_a(bar, bw + 2 * bs);
                    bulk_g2s_a(sb + C::O_KW, kq_r + (t0 / C::PK) * D, bw, bar);
                    bulk_g2s_a(sb + C::O_KS, ks_r + g0 * D, bs, bar);
                    bulk_g2s_a(sb + C::O_KZ, kz_r + g0 * D, bs, bar);
                } else {
                    mbar_arrive_tx_a(bar, bv + 2 * bz);
                    bulk_g2s_a(sb + C::O_VW, vq_r + t0 * C::DW, bv, bar);
                    bulk_g2s_a(sb + C::O_VS, vs_r + t0 * NG, bz, bar);
                    bulk_g2s_a(sb + C::O_VZ, vz_r + t0 * NG, bz, bar);
                }
            } else {
                // ring slots of tokens t0 .. t0+n-1: contiguous up to the ring's end
                const int t0 = w.Tq + (w.j - w.nq) * C::RT, n = min(C::RT, w.len - t0);
                const int s0 = t0 % RG, n1 = min(n, RG - s0);
                // the tile lies in the row's residual tokens, inside the ring, each copy in its region
                if (kivi_check(w.b < c.B && w.rr < RB && t0 >= w.Tq && n > 0 && n <= C::RT &&
                                   t0 + n <= w.len && n <= RG && s0 + n1 <= RG && n - n1 <= s0 &&
                                   C::O_KR + n * C::RROW <= C::O_VR && C::O_VR + n * C::RROW <= C::SLOT,
                               wsi)) {
                    const uint32_t o = kp ? C::O_KR : C::O_VR;
                    const uint16_t* r = kp ? kr_r : vr_r;
                    mbar_arrive_tx_a(bar, (uint32_t)n * D * 2);
                    bulk_g2s_a(sb + o, r + s0 * D, n1 * D * 2, bar);
                    if (n1 < n)
                        bulk_g2s_a(sb + o + n1 * C::RROW, r, (n - n1) * D * 2, bar);
                } else {
                    mbar_arrive(&full[slot]);
                }
            }
            ++issued;
            new_row = ++w.j >= w.nt;
            if (new_row) {
                --w.j;
                walk_next(w, c, RB, C::TS, C::RT);
            }
            if (++slot == ns) {
                slot = 0;
                ++round;
            }
        }
        // leave only once the copies issued have landed (the consumers
        // normally wait for every one of them already)
        if (*(volatile int*)&abort_flag) {
            const volatile int never = 0;
            for (long long k = issued - 1; k >= 0 && k >= issued - ns; --k)
                (void)mbar_wait_bounded(&full[(int)(k % ns)], (uint32_t)((k / ns) & 1), &never);
        }
        return;
    }

    // ------------------------------------------------------------ consumer
    // the two consumer warpgroups take the registers the third gave back
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kStreamConsumerRegs));
    if (warp >= NC)
        return;  // a consumer warp this shape has no shared memory for
    // The consumers take the range's tiles in order from a shared counter, so
    // a warp that falls behind (a merge, a slow tile) takes fewer of them and
    // holds up no one.  A row segment is the range's tiles of one row; a warp
    // keeps one open segment and, when its next tile lies in another one (or
    // the range is done), publishes its state for it in merge buffer
    // (segment mod NMB) with the number of the segment's tiles it took.  The
    // publisher that completes the segment's count merges the states and
    // writes the segment's output or partial.  Which warp takes which tile
    // varies from run to run, so the merged results agree to rounding order.
    using CS = ConsumerState<C, NQB>;
    CS st;
    state_reset<C, NQB>(st);
    float* lg = wscr + warp * C::WARP_FLOATS + C::W_LG;
    float* qw = wscr + warp * C::WARP_FLOATS + C::W_QW;
    uint16_t* ub = reinterpret_cast<uint16_t*>(wscr + warp * C::WARP_FLOATS + C::W_UB);
    uint4* wq = reinterpret_cast<uint4*>(wscr + warp * C::WARP_FLOATS + C::W_Q);
    constexpr int QPL = (C::QPIECES + 31) / 32;  // query pieces per lane
    Walk w = w0;
    long long kw = 0;            // tile of the walker
    int seg = 0;                 // segment of the walker's tile
    long long seg_start = 0;     // its first tile
    // the open segment
    int o_seg = -1, o_tiles = 0, o_b = 0, o_hq0 = 0;
    long long o_start = 0, o_rowend = 0;
    auto publish = [&]() {
        const long long seg_end = o_rowend < ntiles ? o_rowend : ntiles - 1;
        const int seg_len = (int)(seg_end - o_start + 1);
        const int buf = o_seg % C::NMB;
        const bool whole = (o_seg > 0 || r0.j == 0) && o_rowend < ntiles;
        float* mb = mbuf + buf * C::M_END;
        // the buffer's previous segment must have been merged
        {
            const uint64_t t0 = global_ns();
            for (uint32_t it = 0; *(volatile int*)&merged[buf] != o_seg - C::NMB; ++it)
                if ((it & 63u) == 0 && global_ns() - t0 > kStreamWaitNs) {
                    if (lane == 0) {
                        atomicExch(&abort_flag, 1);
                        atomicExch(wsi, KIVI_ETIMEOUT);
                    }
                    break;
                }
            __syncwarp();
            __threadfence_block();
        }
        state_publish<BV, NQB, D, C>(st, lgG, warp, mb);
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();  // this warp's published state before its count
            atomicOr(&pmask[buf], 1 << warp);
            __threadfence_block();
            last = atomicAdd(&ptiles[buf], o_tiles) + o_tiles == seg_len;
            __threadfence_block();  // the others' states after the completing count
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();
        if (last) {
            const unsigned mask = (unsigned)*(volatile int*)&pmask[buf];
            float* dst_o;
            float* dst_ml = nullptr;
            const bool row_ok = kivi_check(o_b < c.B && o_hq0 + NQB <= Hq && (int)blockIdx.x < kMaxStreamCTAs, wsi);
            if (whole) {
                dst_o = out + ((size_t)o_b * Hq + o_hq0) * D;
            } else {
                dst_o = ws + kStreamHeaderFloats + ((size_t)blockIdx.x * 2 + (o_seg == 0 ? 0 : 1)) * NQB * (D + 2);
                dst_ml = dst_o + NQB * D;
            }
#pragma unroll
            for (int hh = 0; hh < NQB; ++hh) {
                if (!row_ok)
                    break;
                float M = -INFINITY;
#pragma unroll
                for (int cw = 0; cw < NC; ++cw)
                    if (mask >> cw & 1u)
                        M = fmaxf(M, mb[C::M_M + cw * NQB + hh]);
                float e[NC], L = 0.0f;
#pragma unroll
                for (int cw = 0; cw < NC; ++cw) {
                    const float mw = mb[C::M_M + cw * NQB + hh];
                    e[cw] = (mask >> cw & 1u) && mw > -INFINITY ? ex2(mw - M) : 0.0f;
                    L = fmaf(e[cw], (mask >> cw & 1u) ? mb[C::M_L + cw * NQB + hh] : 0.0f, L);
                }
                const float inv_l = whole ? 1.0f / L : 1.0f;
                for (int d = lane; d < D; d += 32) {
                    const int gg = d >> lgG;
                    float o = 0.0f;
#pragma unroll
                    for (int cw = 0; cw < NC; ++cw)
                        if (e[cw] != 0.0f)
                            o = fmaf(e[cw],
                                     mb[C::M_O + (cw * NQB + hh) * D + d] + mb[C::M_Z + (cw * NQB + hh) * C::NGM + gg],
                                     o);
                    dst_o[hh * D + d] = o * inv_l;
                }
                if (!whole && lane == 0) {
                    dst_ml[hh] = M;
                    dst_ml[NQB + hh] = L;
                }
            }
            __syncwarp();
            if (lane == 0) {
                pmask[buf] = 0;
                ptiles[buf] = 0;
                __threadfence_block();
                atomicExch(&merged[buf], o_seg);
            }
        }
        state_reset<C, NQB>(st);
        o_seg = -1;
        o_tiles = 0;
    };
    // The warp reserves its next tile while it works on the current one (the
    // counter's round trip is then off the critical path).  The smallest
    // unfinished tile is always some warp's current tile, whose slot's
    // previous tile is finished, so the reservations cannot deadlock.
    unsigned long long kk_next = 0;
    if (lane == 0)
        kk_next = atomicAdd(&next_tile, 1ull);
    for (;;) {
        const long long k = (long long)__shfl_sync(0xffffffffu, kk_next, 0);
        if (k >= ntiles)
            break;
        if (lane == 0)
            kk_next = atomicAdd(&next_tile, 1ull);
        const int crossed = walk_skip(w, c, RB, C::TS, C::RT, (int)(k - kw));
        kw = k;
        if (crossed) {
            seg += crossed;
            seg_start = k - w.j;
        }
        if (o_seg >= 0 && o_seg != seg)
            publish();
        // a new segment (a new row): its query heads go to the warp's scratch
        // once the tile's wait is over; the loads start now
        const bool newq = o_seg < 0;
        uint4 qv[QPL];
        if (newq) {
            const int h = w.rr / NP, pass = w.rr - h * NP;
            const int hq0 = h * NQ + pass * NQB;
            o_seg = seg;
            o_start = seg_start;
            o_rowend = k + (w.nt - 1 - w.j);
            o_b = w.b;
            o_hq0 = hq0;
            const uint4* q4 = reinterpret_cast<const uint4*>(q + ((size_t)w.b * Hq + hq0) * D);
#pragma unroll
            for (int i = 0; i < QPL; ++i)
                if (lane + 32 * i < C::QPIECES)
                    qv[i] = __ldg(q4 + lane + 32 * i);
        }
        ++o_tiles;
        const int slot = (int)((unsigned long long)k % ns);
        const uint32_t round = (uint32_t)((unsigned long long)k / ns);
        const bool aborted = __shfl_sync(0xffffffffu, *(volatile int*)&abort_flag, 0) != 0;
        if (!aborted) {
            // A parity wait cannot tell phase `round` from phase `round` - 2:
            // wait on the full barrier only once the slot's previous tile is
            // done (then its phase `round` - 1 has completed, and the parity
            // names phase `round`).  Tiles are taken in order, so this almost
            // never waits.
            bool ok = true;
            if (*(volatile int*)&consumed[slot] < (int)round) {
                const uint64_t tw = global_ns();
                for (uint32_t it = 0; *(volatile int*)&consumed[slot] < (int)round; ++it)
                    if ((it & 63u) == 0 && (global_ns() - tw > kStreamWaitNs || *(volatile int*)&abort_flag)) {
                        ok = false;
                        break;
                    }
            }
            ok = __all_sync(0xffffffffu, ok) &&
                 __all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], round & 1u, &abort_flag));
            if (!ok && lane == 0) {
                atomicExch(&abort_flag, 1);
                atomicExch(wsi, KIVI_ETIMEOUT);
            }
            if (ok) {
                const uint8_t* sl = slots + (size_t)slot * C::SLOT;
                if (newq) {
#pragma unroll
                    for (int i = 0; i < QPL; ++i)
                        if (lane + 32 * i < C::QPIECES)
                            wq[lane + 32 * i] = qv[i];
                    __syncwarp();
                }
                const uint16_t* qh = reinterpret_cast<const uint16_t*>(wq);
                const int t0 = walk_t0(w, C::TS, C::RT), n = walk_n(w, C::TS, C::RT);
                if (!kivi_check(w.b < c.B && t0 >= 0 && n > 0 && t0 + n <= w.len &&
                                    n <= (walk_quant(w) ? C::TS : C::RT),
                                wsi)) {
                    // nothing to compute
                } else if (walk_quant(w)) {
                    if (n == C::TS)
                        consume_quant<BK, BV, NQB, D, C, true>(st, sl, qh, t0, n, lgG, sl2, lg, qw, ub);
                    else
                        consume_quant<BK, BV, NQB, D, C, false>(st, sl, qh, t0, n, lgG, sl2, lg, qw, ub);
                } else {
                    qk_residual_stage<NQB, D, C>(sl, qh, n, sl2, lg);
                    __syncwarp();
                    softmax_stage<C, NQB>(st, lg, n, st.fv);
                    pv_residual_stage<NQB, D, C>(st, sl, n, lg);
                    __syncwarp();
                }
                if (lane == 0) {
                    *(volatile int*)&consumed[slot] = (int)round + 1;
                    mbar_arrive(&empty[slot]);
                }
            }
        }
    }
    if (o_seg >= 0)
        publish();
}

// --------------------------------------------------------------- combine ---

// Merges the partials of the rows that CTA ranges cut: CTA i of this grid
// takes the row in which range i ends, if range i is not empty, ends inside
// a row, and holds that row's first tile; the ranges after it up to the one
// holding the row's last tile hold its other pieces (their first row
// segment, slot 0), or nothing if they are empty (their slot 0 then holds
// the maximum -inf, a piece of weight zero).  Decode CTA i leaves that row
// in its descriptor (cut or not, the row, the slot of its own piece, the
// last range with a piece), so after its wait this kernel reads the
// descriptor, then the pieces' (m, l) pairs, then their o rows, four pieces
// at a time; a row of at most four pieces (the usual case) has its pairs and
// rows read in one round.  The sums run over the pieces in order, so the
// result does not depend on timing.
template <int NQB, int D, int TS, int RT>
__global__ void __launch_bounds__(128)
decode_stream_combine_kernel(const kivi_cache c, int Hq, int NP, const float* __restrict__ ws,
                             float* __restrict__ out)
{
    constexpr int T = 128;
    const int N = gridDim.x, i = blockIdx.x;
    const int NQ = Hq / c.H;
    __shared__ float s_m[T][NQB], s_l[T][NQB];
    // the next decode kernel may be scheduled once every CTA of this grid
    // runs (it waits for this grid's results before it reads anything)
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int* dsc = reinterpret_cast<const int*>(ws) + kStreamHeaderFloats + stream_partial_floats(D, NQB, N) +
                     (size_t)i * kStreamDescInts;
    if (dsc[0] == 0)
        return;
    const int rb = dsc[1], rr = dsc[2], slot_i = dsc[3], last = dsc[4];
    const int P = last - i + 1;  // ranges i .. last; an empty one holds no piece
    const float* part = ws + kStreamHeaderFloats;
    const size_t pstride = (size_t)NQB * (D + 2);
    auto piece = [&](int k) { return part + ((size_t)k * 2 + (k == i ? slot_i : 0)) * pstride; };
    const int h = rr / NP, pass = rr - h * NP;
    float* dst = out + ((size_t)rb * Hq + h * NQ + pass * NQB) * D;
    // the pieces are the grid's partial slots, the row one of the output's
    if (!kivi_check(last < N && P >= 1 && rb < c.B && h * NQ + pass * NQB + NQB <= Hq,
                    reinterpret_cast<int*>(const_cast<float*>(ws))))
        return;

    constexpr int ND = (D + T - 1) / T;  // channels per thread
    const int t = (int)threadIdx.x;
    if (P <= 4) {
        // the common case: every load of the row in one round (the sums run
        // in the same order as below, so the result is the same)
        float mr[4][NQB], lr[4][NQB], v[4][NQB][ND];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int k = i + r;
            const bool hk = r < P;
            const float* pc = piece(k);
#pragma unroll
            for (int hh = 0; hh < NQB; ++hh) {
                mr[r][hh] = hk ? pc[NQB * D + hh] : -INFINITY;
                lr[r][hh] = hk ? pc[NQB * D + NQB + hh] : 0.0f;
#pragma unroll
                for (int u = 0; u < ND; ++u)
                    v[r][hh][u] = hk && t + u * T < D ? pc[hh * D + t + u * T] : 0.0f;
            }
        }
#pragma unroll
        for (int hh = 0; hh < NQB; ++hh) {
            float Mh = -INFINITY;
#pragma unroll
            for (int r = 0; r < 4; ++r)
                Mh = fmaxf(Mh, mr[r][hh]);
            float Lh = 0.0f, oh[ND];
#pragma unroll
            for (int u = 0; u < ND; ++u)
                oh[u] = 0.0f;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float e = mr[r][hh] > -INFINITY ? ex2(mr[r][hh] - Mh) : 0.0f;
                if (e == 0.0f)
                    continue;
                Lh = fmaf(e, lr[r][hh], Lh);
#pragma unroll
                for (int u = 0; u < ND; ++u)
                    oh[u] = fmaf(e, v[r][hh][u], oh[u]);
            }
#pragma unroll
            for (int u = 0; u < ND; ++u)
                if (t + u * T < D)
                    dst[hh * D + t + u * T] = oh[u] / Lh;
        }
        return;
    }
    float M[NQB], L[NQB], o[NQB][ND];
#pragma unroll
    for (int hh = 0; hh < NQB; ++hh) {
        M[hh] = -INFINITY;
        L[hh] = 0.0f;
#pragma unroll
        for (int u = 0; u < ND; ++u)
            o[hh][u] = 0.0f;
    }
    auto load_ml = [&](int c0) {
        const int k = i + c0 + t;
        const bool hk = c0 + t < P;
#pragma unroll
        for (int hh = 0; hh < NQB; ++hh) {
            s_m[t][hh] = hk ? piece(k)[NQB * D + hh] : -INFINITY;
            s_l[t][hh] = hk ? piece(k)[NQB * D + NQB + hh] : 0.0f;
        }
    };
    // pass 1: the maxima (a single chunk of pairs stays in shared memory)
    for (int c0 = 0; c0 < P; c0 += T) {
        load_ml(c0);
        __syncthreads();
        const int nq = min(T, P - c0);
        for (int qq = 0; qq < nq; ++qq)
#pragma unroll
            for (int hh = 0; hh < NQB; ++hh)
                M[hh] = fmaxf(M[hh], s_m[qq][hh]);
        __syncthreads();
    }
    // pass 2: weights and sums, four pieces' rows loaded at a time
    for (int c0 = 0; c0 < P; c0 += T) {
        if (P > T) {
            load_ml(c0);
            __syncthreads();
        }
        const int nq = min(T, P - c0);
        for (int q0 = 0; q0 < nq; q0 += 4) {
            float e[4][NQB], v[4][NQB][ND];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int hh = 0; hh < NQB; ++hh) {
                    const float m = q0 + r < nq ? s_m[q0 + r][hh] : -INFINITY;
                    e[r][hh] = m > -INFINITY ? ex2(m - M[hh]) : 0.0f;
                    const float* pq = piece(i + c0 + q0 + r) + hh * D;
#pragma unroll
                    for (int u = 0; u < ND; ++u) {
                        const int d = t + u * T;
                        v[r][hh][u] = e[r][hh] != 0.0f && d < D ? pq[d] : 0.0f;
                    }
                }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int hh = 0; hh < NQB; ++hh) {
                    if (e[r][hh] == 0.0f)
                        continue;
                    L[hh] = fmaf(e[r][hh], s_l[q0 + r][hh], L[hh]);
#pragma unroll
                    for (int u = 0; u < ND; ++u)
                        o[hh][u] = fmaf(e[r][hh], v[r][hh][u], o[hh][u]);
                }
        }
        if (P > T)
            __syncthreads();
    }
#pragma unroll
    for (int hh = 0; hh < NQB; ++hh)
#pragma unroll
        for (int u = 0; u < ND; ++u) {
            const int d = (int)threadIdx.x + u * T;
            if (d < D)
                dst[hh * D + d] = o[hh][u] / L[hh];
        }
}

// ---------------------------------------------------------------- launch ---

template <int D, int BK, int BV, int NQB, int NC>
cudaError_t stream_launch(const kivi_cache& c, const uint16_t* q, int Hq, float sm, float* out, float* ws,
                          cudaStream_t s)
{
    using C = StreamCfg<BK, BV, NQB, D, NC>;
    auto kern = decode_stream_kernel<BK, BV, NQB, D, NC>;
    constexpr int ns = stream_stages<C>();
    static_assert(ns >= 2, "the shared memory holds at least two stages");
    const size_t smem = (size_t)ns * C::SLOT + C::FIXED_BYTES - kStreamStaticSmem + 2 * (size_t)ns * 8;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    // the register split needs the block launched with kStreamLaunchRegs per
    // thread: otherwise the consumers' setmaxnreg.inc could never be granted
    static int launch_regs = -1;
    if (launch_regs < 0) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess)
            return e;
        launch_regs = fa.numRegs;
    }
    if (launch_regs != kStreamLaunchRegs)
        return cudaErrorInvalidConfiguration;
    const int N = cmin(sm_count(), kMaxStreamCTAs);
#ifdef KIVI_CHECKS
    // the status word starts at KIVI_OK before any CTA can record a check
    e = cudaMemsetAsync(ws, 0, sizeof(int32_t), s);
    if (e != cudaSuccess)
        return e;
#endif
    {
        cudaLaunchConfig_t cf = {};
        cf.gridDim = dim3(N);
        cf.blockDim = dim3(C::THREADS);
        cf.dynamicSmemBytes = smem;
        cf.stream = s;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cf.attrs = at;
        cf.numAttrs = 1;
        e = cudaLaunchKernelEx(&cf, kern, c, q, Hq, sm, out, ws);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            kern<<<N, C::THREADS, smem, s>>>(c, q, Hq, sm, out, ws);
        }
    }
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const int NP = (Hq / c.H) / NQB;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(N);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto comb = decode_stream_combine_kernel<NQB, D, C::TS, C::RT>;
    e = cudaLaunchKernelEx(&cfg, comb, c, Hq, NP, (const float*)ws, out);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        comb<<<N, 128, 0, s>>>(c, Hq, NP, ws, out);
    }
    return cudaGetLastError();
}

// Dispatch of the key and value widths and the query heads per pass for head
// dimension D.
template <int D, int BK, int BV>
cudaError_t stream_launch_nq(const kivi_cache& c, const uint16_t* q, int Hq, float sm, float* out, float* ws,
                             cudaStream_t s)
{
    switch (heads_per_pass(Hq / c.H)) {
    case 4: return stream_launch<D, BK, BV, 4, stream_consumers<BK, BV, 4, D>()>(c, q, Hq, sm, out, ws, s);
    case 2: return stream_launch<D, BK, BV, 2, stream_consumers<BK, BV, 2, D>()>(c, q, Hq, sm, out, ws, s);
    default: return stream_launch<D, BK, BV, 1, stream_consumers<BK, BV, 1, D>()>(c, q, Hq, sm, out, ws, s);
    }
}

template <int D, int BK>
cudaError_t stream_launch_bv(const kivi_cache& c, const uint16_t* q, int Hq, float sm, float* out, float* ws,
                             cudaStream_t s)
{
    switch (c.bits_v) {
    case 2: return stream_launch_nq<D, BK, 2>(c, q, Hq, sm, out, ws, s);
    case 4: return stream_launch_nq<D, BK, 4>(c, q, Hq, sm, out, ws, s);
    default: return stream_launch_nq<D, BK, 8>(c, q, Hq, sm, out, ws, s);
    }
}

template <int D, int BK>
cudaError_t launch_decode_stream(const kivi_cache& c, const uint16_t* q, int Hq, float sm, float* out, float* ws,
                                 cudaStream_t s)
{
    return stream_launch_bv<D, BK>(c, q, Hq, sm, out, ws, s);
}

// Instantiates the streamed decode for one head dimension and key width (one
// translation unit each, so that they compile in parallel).
#define KIVI_STREAM_INSTANTIATE(DIM, BK)                                                                      \
    template cudaError_t launch_decode_stream<DIM, BK>(const kivi_cache&, const uint16_t*, int, float, float*, \
                                                       float*, cudaStream_t);

}  // namespace kivi
