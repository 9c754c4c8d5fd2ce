// decode.cu -- decode attention over the packed KIVI cache plus the fp16
// residual, with dequantization fused into the loads (the decode-time consumer
// of the cache: q . K_hat^T, softmax, p . V_hat).
//
// Both GEMVs factor the statistics out of the inner loop:
//   keys   (per-channel stats s_d, z_d of a G-token group):
//          q . k_hat_t = sum_d (q_d s_d) c_td + sum_d q_d z_d
//   values (per-token stats s_t, z_t of a G-channel group):
//          sum_t p_t v_hat_td = sum_t (p_t s_t) c_td + sum_t p_t z_t
// so each code costs one mask (window_value) and one FMA per query head.
// HBM-bound: K and V are each read once per KV head (grouped-query heads share
// the load), b/8 bytes of code + 8/G bytes of statistics per element.
#include <math.h>

#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

constexpr int kDecodeThreads = 128;
constexpr int kSegChans = 32;               // channels per lane in decode_qk
constexpr int kSegStride = kSegChans + 4;   // padded shared-memory row (bank spread)

// --------------------------------------------------------------- q . K^T ---
//
// CTA = (chunk of TC tokens, b, h).  Quantized part: a lane owns 16 tokens x
// 32 channels; the D/32 lanes of a 16-token row are adjacent and reduce with
// shuffles.  Residual part: a lane owns one token x 32 channels.
template <int BITS, int NQB>
__global__ void __launch_bounds__(kDecodeThreads)
decode_qk_kernel(kivi_cache c, const uint16_t* __restrict__ q, int Hq, float sm_scale,
                 float* __restrict__ logits, int ldl, int TC)
{
    using Cd = Codec<BITS>;
    using Win = Window<BITS>;
    extern __shared__ __align__(16) float qsm[];  // [NQB][D/32][kSegStride]

    const int D = c.D, H = c.H;
    const int LPR = D / kSegChans;
    const int chunk = blockIdx.y;
    const size_t bh = blockIdx.x;
    const int b = (int)(bh / H), h = (int)(bh % H);
    const int NQ = Hq / H;
    const int n = c.len[b];
    const int t_begin = chunk * TC;
    if (t_begin >= n)
        return;
    const int t_end = min(t_begin + TC, n);
    const int Tq = quantized_tokens(n, c.G, c.R);
    const int RG = c.R + c.G;
    const int lane = threadIdx.x & 31;
    const int seg = threadIdx.x % LPR;
    const unsigned rmask = (((1u << LPR) - 1u) << (lane & ~(LPR - 1)));
    const int rows_per_cta = kDecodeThreads / LPR;
    const int hq_stride = (D / kSegChans) * kSegStride;
    const int TPL = kLaneTokens / LPR;  // logits each lane stores per row
    const uint32_t one = one_bits();

    for (int pass = 0; pass < NQ / NQB; ++pass) {
        const int hq0 = h * NQ + pass * NQB;
        __syncthreads();
        for (int i = threadIdx.x; i < NQB * D; i += kDecodeThreads) {
            const int hq = i / D, d = i % D;
            qsm[hq * hq_stride + (d / kSegChans) * kSegStride + d % kSegChans] =
                __half2float(__ushort_as_half(q[((size_t)b * Hq + hq0 + hq) * D + d]));
        }
        __syncthreads();
        const float* qseg = qsm + seg * kSegStride;

        // ---- quantized rows (Tq and t_begin are multiples of 16) ----
        const int tq_end = min(t_end, Tq);
        for (int t0 = t_begin + (threadIdx.x / LPR) * kLaneTokens; t0 < tq_end;
             t0 += rows_per_cta * kLaneTokens) {
            const int g = t0 / c.G;
            const int32_t* kw = c.kq + (bh * (size_t)(c.Tmax / Cd::P) + t0 / Cd::P) * D +
                                seg * kSegChans;
            const size_t so = (bh * (size_t)(c.Tmax / c.G) + g) * D + seg * kSegChans;
            float acc[NQB][kLaneTokens];
            float Ssum[NQB], Zsum[NQB];
#pragma unroll
            for (int hq = 0; hq < NQB; ++hq) {
                Ssum[hq] = Zsum[hq] = 0.0f;
#pragma unroll
                for (int i = 0; i < kLaneTokens; ++i)
                    acc[hq][i] = 0.0f;
            }
            // Load phases of LB channel batches (4 channels each): every load
            // of a phase is issued before any of its data is used.
            constexpr int LB = BITS == 2 ? 8 : BITS == 4 ? 4 : 2;
#pragma unroll 1
            for (int cb0 = 0; cb0 < kSegChans / 4; cb0 += LB) {
                uint4 W[LB][Cd::kWordRows];
                float4 SC[LB], ZR[LB];
#pragma unroll
                for (int l = 0; l < LB; ++l) {
#pragma unroll
                    for (int w = 0; w < Cd::kWordRows; ++w)
                        W[l][w] = ld_nc(kw + (size_t)w * D + (cb0 + l) * 4);
                    SC[l] = ld_nc_f4(c.kscale + so + (cb0 + l) * 4);
                    ZR[l] = ld_nc_f4(c.kzero + so + (cb0 + l) * 4);
                }
#pragma unroll
                for (int l = 0; l < LB; ++l) {
                    const int cb = cb0 + l;
                    const float scv[4] = {SC[l].x, SC[l].y, SC[l].z, SC[l].w};
                    const float zrv[4] = {ZR[l].x, ZR[l].y, ZR[l].z, ZR[l].w};
                    float qsw[NQB][4][Win::kNumPos];
#pragma unroll
                    for (int hq = 0; hq < NQB; ++hq) {
                        const float4 qv = *reinterpret_cast<const float4*>(qseg + hq * hq_stride + cb * 4);
                        const float qq[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float qs = qq[k] * scv[k];
                            Ssum[hq] += qs;
                            Zsum[hq] = fmaf(qq[k], zrv[k], Zsum[hq]);
#pragma unroll
                            for (int p = 0; p < Win::kNumPos; ++p)
                                qsw[hq][k][p] = qs * Win::mult_of_index(p);
                        }
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int w = 0; w < Cd::kWordRows; ++w) {
                            float f[Cd::P];
                            window_values<BITS>(u4_word(W[l][w], k), one, f);
#pragma unroll
                            for (int ci = 0; ci < Cd::P; ++ci)
#pragma unroll
                                for (int hq = 0; hq < NQB; ++hq)
                                    acc[hq][w * Cd::P + ci] = fmaf(qsw[hq][k][Win::pos_index(ci)], f[ci],
                                                                   acc[hq][w * Cd::P + ci]);
                        }
                }
            }
#pragma unroll
            for (int hq = 0; hq < NQB; ++hq)
#pragma unroll
                for (int i = 0; i < kLaneTokens; ++i) {
                    const float mult = Win::mult_of_index(Win::pos_index(i % Cd::P));
                    acc[hq][i] = fmaf(-mult, Ssum[hq], acc[hq][i]) + Zsum[hq];
                }
            for (int m = 1; m < LPR; m <<= 1)
#pragma unroll
                for (int hq = 0; hq < NQB; ++hq)
#pragma unroll
                    for (int i = 0; i < kLaneTokens; ++i)
                        acc[hq][i] += __shfl_xor_sync(rmask, acc[hq][i], m);
#pragma unroll
            for (int hq = 0; hq < NQB; ++hq) {
                float* lrow = logits + ((size_t)b * Hq + hq0 + hq) * ldl + t0;
#pragma unroll
                for (int i = 0; i < kLaneTokens; ++i)
                    if (i / TPL == seg)
                        lrow[i] = sm_scale * acc[hq][i];
            }
        }

        // ---- residual rows ----
        for (int t = max(t_begin, Tq) + threadIdx.x / LPR; t < t_end; t += rows_per_cta) {
            const uint16_t* kr = c.kres + (bh * RG + t % RG) * D + seg * kSegChans;
            float acc[NQB];
#pragma unroll
            for (int hq = 0; hq < NQB; ++hq)
                acc[hq] = 0.0f;
#pragma unroll
            for (int u = 0; u < kSegChans / 8; ++u) {
                const uint4 kv = ld_nc(kr + u * 8);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float kf = __half2float(__ushort_as_half(u4_half(kv, e)));
#pragma unroll
                    for (int hq = 0; hq < NQB; ++hq)
                        acc[hq] = fmaf(qseg[hq * hq_stride + u * 8 + e], kf, acc[hq]);
                }
            }
            for (int m = 1; m < LPR; m <<= 1)
#pragma unroll
                for (int hq = 0; hq < NQB; ++hq)
                    acc[hq] += __shfl_xor_sync(rmask, acc[hq], m);
            if (seg == 0)
#pragma unroll
                for (int hq = 0; hq < NQB; ++hq)
                    logits[((size_t)b * Hq + hq0 + hq) * ldl + t] = sm_scale * acc[hq];
        }
    }
}

// ---------------------------------------------------------------- p . V ---
//
// CTA = (chunk of TC tokens, b, h).  Phase 1: the chunk's logits go to shared
// memory, p = exp(s - m_chunk), l_chunk = sum p.  Phase 2: a lane owns one
// token x CPL channels (one channel group segment); it accumulates
// (p s_t) * code per channel.  Phase 3: lanes and warps are summed through
// shared memory and the chunk's (m, l, o) goes to the workspace.
template <int NQB>
__device__ __forceinline__ void block_reduce(float (&v)[NQB], float* red, bool is_max)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NW = kDecodeThreads / 32;
#pragma unroll
    for (int hq = 0; hq < NQB; ++hq)
        for (int m = 16; m > 0; m >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, v[hq], m);
            v[hq] = is_max ? fmaxf(v[hq], o) : v[hq] + o;
        }
    __syncthreads();
    if (lane == 0)
#pragma unroll
        for (int hq = 0; hq < NQB; ++hq)
            red[warp * NQB + hq] = v[hq];
    __syncthreads();
#pragma unroll
    for (int hq = 0; hq < NQB; ++hq) {
        float r = red[hq];
#pragma unroll
        for (int w = 1; w < NW; ++w)
            r = is_max ? fmaxf(r, red[w * NQB + hq]) : r + red[w * NQB + hq];
        v[hq] = r;
    }
}

template <int BITS, int NQB, int CPL>
__global__ void __launch_bounds__(kDecodeThreads)
decode_pv_kernel(kivi_cache c, const float* __restrict__ logits, int ldl, int Hq,
                 float* __restrict__ ws_o, float* __restrict__ ws_m, float* __restrict__ ws_l,
                 int TC, int nchunks)
{
    using Cd = Codec<BITS>;
    using Win = Window<BITS>;
    constexpr int WPL = CPL / Cd::P;  // words per lane per token
    extern __shared__ __align__(16) float pv_smem[];
    float* p_sm = pv_smem;           // [TC][NQB]; reused for the phase-3 partials
    __shared__ float red[(kDecodeThreads / 32) * NQB];

    const int D = c.D, H = c.H;
    const int chunk = blockIdx.y;
    const size_t bh = blockIdx.x;
    const int b = (int)(bh / H), h = (int)(bh % H);
    const int NQ = Hq / H;
    const int n = c.len[b];
    const int t_begin = chunk * TC;
    if (t_begin >= n)
        return;
    const int t_end = min(t_begin + TC, n);
    const int Tq = quantized_tokens(n, c.G, c.R);
    const int RG = c.R + c.G;
    const int LPT = D / CPL;                 // lanes per token
    const int TPW = 32 / LPT;                // tokens per warp step
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = lane % LPT, tl = lane / LPT;
    constexpr int NW = kDecodeThreads / 32;
    const int g = (seg * CPL) / c.G;         // channel group of this segment
    const uint32_t one = one_bits();
    const int NGv = D / c.G;

    for (int pass = 0; pass < NQ / NQB; ++pass) {
        const int hq0 = h * NQ + pass * NQB;
        __syncthreads();
        // ---- phase 1: chunk softmax statistics ----
        float mloc[NQB];
#pragma unroll
        for (int hq = 0; hq < NQB; ++hq)
            mloc[hq] = -INFINITY;
        for (int t = t_begin + threadIdx.x; t < t_end; t += kDecodeThreads)
#pragma unroll
            for (int hq = 0; hq < NQB; ++hq) {
                const float sv = logits[((size_t)b * Hq + hq0 + hq) * ldl + t];
                p_sm[(t - t_begin) * NQB + hq] = sv;
                mloc[hq] = fmaxf(mloc[hq], sv);
            }
        block_reduce<NQB>(mloc, red, true);
        float lloc[NQB];
#pragma unroll
        for (int hq = 0; hq < NQB; ++hq)
            lloc[hq] = 0.0f;
        for (int t = t_begin + threadIdx.x; t < t_end; t += kDecodeThreads)
#pragma unroll
            for (int hq = 0; hq < NQB; ++hq) {
                const float pe = expf(p_sm[(t - t_begin) * NQB + hq] - mloc[hq]);
                p_sm[(t - t_begin) * NQB + hq] = pe;
                lloc[hq] += pe;
            }
        block_reduce<NQB>(lloc, red, false);  // its barriers also publish p_sm

        // ---- phase 2: weighted sum of dequantized values ----
        float acc[NQB][CPL];
        float Ssum[NQB], Zsum[NQB];
#pragma unroll
        for (int hq = 0; hq < NQB; ++hq) {
            Ssum[hq] = Zsum[hq] = 0.0f;
#pragma unroll
            for (int k = 0; k < CPL; ++k)
                acc[hq][k] = 0.0f;
        }
        const int tq_end = min(t_end, Tq);
        constexpr int UNR = NQB == 1 ? 8 : 4;  // tokens whose loads are in flight per lane
        for (int t0 = t_begin + warp * TPW + tl; t0 < tq_end; t0 += NW * TPW * UNR) {
            uint32_t W[UNR][WPL];
            float SV[UNR], ZV[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int t = t0 + u * NW * TPW;
                SV[u] = ZV[u] = 0.0f;
#pragma unroll
                for (int w = 0; w < WPL; ++w)
                    W[u][w] = 0u;
                if (t < tq_end) {
                    const size_t vrow = bh * (size_t)c.Tmax + t;
                    const int32_t* vw = c.vq + vrow * (D / Cd::P) + seg * WPL;
                    if constexpr (WPL == 1) {
                        W[u][0] = (uint32_t)__ldg(vw);
                    } else if constexpr (WPL == 2) {
                        const uint2 x = __ldg(reinterpret_cast<const uint2*>(vw));
                        W[u][0] = x.x;
                        W[u][1] = x.y;
                    } else {
#pragma unroll
                        for (int w = 0; w < WPL; w += 4) {
                            const uint4 x = ld_nc(vw + w);
                            W[u][w] = x.x;
                            W[u][w + 1] = x.y;
                            W[u][w + 2] = x.z;
                            W[u][w + 3] = x.w;
                        }
                    }
                    SV[u] = __ldg(c.vscale + vrow * NGv + g);
                    ZV[u] = __ldg(c.vzero + vrow * NGv + g);
                }
            }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int t = t0 + u * NW * TPW;
                if (t >= tq_end)
                    break;
                float psw[NQB][Win::kNumPos];
#pragma unroll
                for (int hq = 0; hq < NQB; ++hq) {
                    const float pt = p_sm[(t - t_begin) * NQB + hq];
                    const float ps = pt * SV[u];
                    Ssum[hq] += ps;
                    Zsum[hq] = fmaf(pt, ZV[u], Zsum[hq]);
#pragma unroll
                    for (int p = 0; p < Win::kNumPos; ++p)
                        psw[hq][p] = ps * Win::mult_of_index(p);
                }
#pragma unroll
                for (int w = 0; w < WPL; ++w) {
                    float f[Cd::P];
                    window_values<BITS>(W[u][w], one, f);
#pragma unroll
                    for (int i = 0; i < Cd::P; ++i)
#pragma unroll
                        for (int hq = 0; hq < NQB; ++hq)
                            acc[hq][w * Cd::P + i] =
                                fmaf(psw[hq][Win::pos_index(i)], f[i], acc[hq][w * Cd::P + i]);
                }
            }
        }
#pragma unroll
        for (int hq = 0; hq < NQB; ++hq)
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
                const float mult = Win::mult_of_index(Win::pos_index(k % Cd::P));
                acc[hq][k] = fmaf(-mult, Ssum[hq], acc[hq][k]) + Zsum[hq];
            }
        // residual tokens: exact fp16 values
        for (int t = max(t_begin, Tq) + warp * TPW + tl; t < t_end; t += NW * TPW) {
            const uint16_t* vr = c.vres + (bh * RG + t % RG) * D + seg * CPL;
            float pt[NQB];
#pragma unroll
            for (int hq = 0; hq < NQB; ++hq)
                pt[hq] = p_sm[(t - t_begin) * NQB + hq];
#pragma unroll
            for (int u = 0; u < CPL / 8; ++u) {
                const uint4 x = ld_nc(vr + u * 8);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float vf = __half2float(__ushort_as_half(u4_half(x, e)));
#pragma unroll
                    for (int hq = 0; hq < NQB; ++hq)
                        acc[hq][u * 8 + e] = fmaf(pt[hq], vf, acc[hq][u * 8 + e]);
                }
            }
        }

        // ---- phase 3: sum the NW*TPW token lanes of each channel ----
        __syncthreads();  // every warp is done reading p_sm
        float* part = p_sm;  // [NW*TPW][NQB][D]
        const int slot = warp * TPW + tl;
#pragma unroll
        for (int hq = 0; hq < NQB; ++hq)
#pragma unroll
            for (int k = 0; k < CPL; ++k)
                part[((size_t)slot * NQB + hq) * D + seg * CPL + k] = acc[hq][k];
        __syncthreads();
        const int nslots = NW * TPW;
        for (int idx = threadIdx.x; idx < NQB * D; idx += kDecodeThreads) {
            const int hq = idx / D, d = idx % D;
            float sum = 0.0f;
            for (int sl = 0; sl < nslots; ++sl)
                sum += part[((size_t)sl * NQB + hq) * D + d];
            const size_t row = ((size_t)b * Hq + hq0 + hq) * nchunks + chunk;
            ws_o[row * D + d] = sum;
        }
#pragma unroll
        for (int hq = 0; hq < NQB; ++hq)
            if (threadIdx.x == hq) {
                const size_t row = ((size_t)b * Hq + hq0 + hq) * nchunks + chunk;
                ws_m[row] = mloc[hq];
                ws_l[row] = lloc[hq];
            }
    }
}

// out[b][hq][d] = sum_c o_c[d] e^(m_c - M) / sum_c l_c e^(m_c - M), M = max m_c.
__global__ void __launch_bounds__(256)
decode_combine_kernel(const int32_t* __restrict__ len, int Hq, int D, int TC, int nchunks,
                      const float* __restrict__ ws_o, const float* __restrict__ ws_m,
                      const float* __restrict__ ws_l, float* __restrict__ out)
{
    const size_t bhq = blockIdx.x;
    const int b = (int)(bhq / Hq);
    const int n = len[b];
    const int nv = (n + TC - 1) / TC;
    const float* mrow = ws_m + bhq * nchunks;
    const float* lrow = ws_l + bhq * nchunks;
    float M = -INFINITY;
    for (int k = 0; k < nv; ++k)
        M = fmaxf(M, mrow[k]);
    float L = 0.0f;
    for (int k = 0; k < nv; ++k)
        L += lrow[k] * expf(mrow[k] - M);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float o = 0.0f;
        for (int k = 0; k < nv; ++k)
            o = fmaf(ws_o[(bhq * nchunks + k) * D + d], expf(mrow[k] - M), o);
        out[bhq * D + d] = nv > 0 ? o / L : 0.0f;
    }
}

// ---------------------------------------------------------------- launch ---

int qk_chunk_tokens(int D) { return 2 * (kDecodeThreads / (D / kSegChans)) * kLaneTokens; }
int pv_chunk_tokens(int) { return 1024; }
int pv_chunks(const kivi_cache& c)
{
    const int TC = pv_chunk_tokens(c.D);
    return (c.Tmax + TC - 1) / TC;
}

static int heads_per_pass(int NQ) { return NQ % 4 == 0 ? 4 : NQ % 2 == 0 ? 2 : 1; }

template <int BITS>
static cudaError_t qk_bits(const kivi_cache& c, const uint16_t* q, int Hq, float sm,
                           float* logits, int ldl, cudaStream_t s)
{
    const int NQB = heads_per_pass(Hq / c.H);
    const int TC = qk_chunk_tokens(c.D);
    const dim3 grid(c.B * c.H, (c.Tmax + TC - 1) / TC);
    const size_t smem = (size_t)NQB * (c.D / kSegChans) * kSegStride * sizeof(float);
    switch (NQB) {
    case 4: decode_qk_kernel<BITS, 4><<<grid, kDecodeThreads, smem, s>>>(c, q, Hq, sm, logits, ldl, TC); break;
    case 2: decode_qk_kernel<BITS, 2><<<grid, kDecodeThreads, smem, s>>>(c, q, Hq, sm, logits, ldl, TC); break;
    default: decode_qk_kernel<BITS, 1><<<grid, kDecodeThreads, smem, s>>>(c, q, Hq, sm, logits, ldl, TC); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_decode_qk(const kivi_cache& c, const uint16_t* q, int Hq, float sm_scale,
                             float* logits, int ld_logits, cudaStream_t s)
{
    switch (c.bits_k) {
    case 2: return qk_bits<2>(c, q, Hq, sm_scale, logits, ld_logits, s);
    case 4: return qk_bits<4>(c, q, Hq, sm_scale, logits, ld_logits, s);
    default: return qk_bits<8>(c, q, Hq, sm_scale, logits, ld_logits, s);
    }
}

template <int BITS, int NQB, int CPL>
static void pv_launch(const kivi_cache& c, const float* logits, int ldl, int Hq, float* ws_o,
                      float* ws_m, float* ws_l, int TC, int nch, cudaStream_t s)
{
    const int LPT = c.D / CPL;
    const int slots = (kDecodeThreads / 32) * (32 / LPT);
    const size_t p_bytes = (size_t)TC * NQB * sizeof(float);
    const size_t part_bytes = (size_t)slots * NQB * c.D * sizeof(float);
    const size_t smem = p_bytes > part_bytes ? p_bytes : part_bytes;
    auto kern = decode_pv_kernel<BITS, NQB, CPL>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const dim3 grid(c.B * c.H, nch);
    kern<<<grid, kDecodeThreads, smem, s>>>(c, logits, ldl, Hq, ws_o, ws_m, ws_l, TC, nch);
}

template <int BITS>
static void pv_bits(const kivi_cache& c, const float* logits, int ldl, int Hq, float* ws_o,
                    float* ws_m, float* ws_l, int TC, int nch, cudaStream_t s)
{
    switch (heads_per_pass(Hq / c.H)) {
    case 4: pv_launch<BITS, 4, 16>(c, logits, ldl, Hq, ws_o, ws_m, ws_l, TC, nch, s); break;
    case 2: pv_launch<BITS, 2, 32>(c, logits, ldl, Hq, ws_o, ws_m, ws_l, TC, nch, s); break;
    default: pv_launch<BITS, 1, 32>(c, logits, ldl, Hq, ws_o, ws_m, ws_l, TC, nch, s); break;
    }
}

cudaError_t launch_decode_pv(const kivi_cache& c, const float* logits, int ld_logits, int Hq,
                             float* out, float* ws_o, float* ws_m, float* ws_l, cudaStream_t s)
{
    const int TC = pv_chunk_tokens(c.D);
    const int nch = pv_chunks(c);
    switch (c.bits_v) {
    case 2: pv_bits<2>(c, logits, ld_logits, Hq, ws_o, ws_m, ws_l, TC, nch, s); break;
    case 4: pv_bits<4>(c, logits, ld_logits, Hq, ws_o, ws_m, ws_l, TC, nch, s); break;
    default: pv_bits<8>(c, logits, ld_logits, Hq, ws_o, ws_m, ws_l, TC, nch, s); break;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    decode_combine_kernel<<<c.B * Hq, c.D < 256 ? c.D : 256, 0, s>>>(c.len, Hq, c.D, TC, nch,
                                                                     ws_o, ws_m, ws_l, out);
    return cudaGetLastError();
}

}  // namespace kivi
