// dequant.cu -- materialize: unpack codes and dequantize to fp16
// (x_hat = fp16_rne(fmaf(code, scale, zero))), residual rows copied from the
// ring.  CacheSeek PR #4 change notes: only the compact codes, scales and
// offsets travel back to the device, and dequantization happens there.
//
// HBM-bound: reads b/8 bytes of code plus the statistics per element and
// writes 2 bytes per element with 16-byte stores.  2-D grids (x: token tiles,
// y: (b, h) slices), 32-bit index arithmetic.
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

constexpr int kDequantThreads = 256;

__device__ __forceinline__ int lg2(int x) { return __ffs(x) - 1; }

// Keys: one lane = 16 tokens x 8 channels of a G-token group.
template <int BITS>
__global__ void __launch_bounds__(kDequantThreads)
dequant_keys_kernel(kivi_cache c, uint16_t* __restrict__ out, int T_out)
{
    using Cd = Codec<BITS>;
    const int D = c.D;
    const int S = c.G / kLaneTokens, lgS = lg2(S);
    const int NC = D / kLaneChans, lgNC = lg2(NC);
    const int id = blockIdx.x * kDequantThreads + threadIdx.x;  // lane task within the slice
    const int s = id & (S - 1);
    const int j = (id >> lgS) & (NC - 1);
    const int g = id >> (lgS + lgNC);
    const int t0 = g * c.G + s * kLaneTokens;
    const int RG = c.R + c.G;
    const uint32_t two23 = two23_bits();

    for (int bh = blockIdx.y; bh < c.B * c.H; bh += gridDim.y) {
        const int len = ld_checked(c.len + bh / c.H);
        const int n = min(len, T_out);
        if (t0 >= n)
            continue;
        const int Tq = quantized_tokens(len, c.G, c.R);
        uint16_t* dst = out + (size_t)bh * T_out * D + j * kLaneChans;
        if (t0 + kLaneTokens <= Tq) {
            const int32_t* src = c.kq + ((size_t)bh * (c.Tmax / Cd::P) + t0 / Cd::P) * D +
                                 j * kLaneChans;
            uint4 wlo[Cd::kWordRows], whi[Cd::kWordRows];
#pragma unroll
            for (int w = 0; w < Cd::kWordRows; ++w) {
                wlo[w] = ld_stream(src + (size_t)w * D);
                whi[w] = ld_stream(src + (size_t)w * D + 4);
            }
            const size_t so = ((size_t)bh * (c.Tmax / c.G) + g) * D + j * kLaneChans;
            const float4 s0 = ld_nc_f4(c.kscale + so), s1 = ld_nc_f4(c.kscale + so + 4);
            const float4 z0 = ld_nc_f4(c.kzero + so), z1 = ld_nc_f4(c.kzero + so + 4);
            const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
            const float zr[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
            for (int i = 0; i < kLaneTokens; ++i) {
                if (t0 + i >= n)
                    break;  // out holds only T_out rows
                const int w = i / Cd::P, sh = (i % Cd::P) * BITS;
                uint32_t h2[4];
#pragma unroll
                for (int k = 0; k < 8; k += 2) {
                    const uint32_t w0 = k < 4 ? u4_word(wlo[w], k) : u4_word(whi[w], k - 4);
                    const uint32_t w1 = k < 4 ? u4_word(wlo[w], k + 1) : u4_word(whi[w], k - 3);
                    h2[k / 2] = dequant_h2(code_float(w0 >> sh, Cd::M, two23),
                                           code_float(w1 >> sh, Cd::M, two23), sc[k], zr[k],
                                           sc[k + 1], zr[k + 1]);
                }
                st_stream(dst + (size_t)(t0 + i) * D, make_uint4(h2[0], h2[1], h2[2], h2[3]));
            }
        } else {
            for (int i = 0; i < kLaneTokens; ++i) {
                const int t = t0 + i;
                if (t >= Tq && t < n)
                    st_stream(dst + (size_t)t * D,
                              ld_nc(c.kres + ((size_t)bh * RG + t % RG) * D + j * kLaneChans));
            }
        }
    }
}

// Values: one lane = one channel group (G channels) of U token rows: the
// group's words, scale and zero are loaded once and G fp16 values produced.
// A lane's 16-byte output chunks lie 64 bytes apart (G = 32), so each warp
// passes its rows through shared memory and stores them back with every
// instruction writing 512 contiguous bytes.  In shared memory chunk c of warp
// row r sits at c ^ ((r NG ^ c / (G/8)) & 7), which keeps both the group-wise
// writes and the row-wise reads free of bank conflicts.
template <int BITS, int G>
__global__ void __launch_bounds__(kDequantThreads)
dequant_values_kernel(kivi_cache c, uint16_t* __restrict__ out, int T_out)
{
    using Cd = Codec<BITS>;
    constexpr int U = G == 32 ? 4 : G == 64 ? 2 : 1;
    constexpr int NW = G * BITS / 32;  // words per group
    constexpr int NV = G / 8;          // 16-byte chunks per group
    constexpr int lgNV = G == 32 ? 2 : G == 64 ? 3 : 4;
    extern __shared__ __align__(16) uint4 dq_rows[];
    const int D = c.D;
    const int NG = D / G, lgNG = lg2(NG);
    const int CPR = D / 8, lgCPR = lg2(CPR);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gi = threadIdx.x & (NG - 1);
    const int rows_per_pass = kDequantThreads >> lgNG;
    const int rows_w = 32 >> lgNG;                      // rows per warp and pass
    const int wr = lane >> lgNG;                        // this lane's row in the warp
    const int r0 = blockIdx.x * rows_per_pass * U + (threadIdx.x >> lgNG);
    const int RG = c.R + c.G;
    const uint32_t two23 = two23_bits();
    uint4* wsm = dq_rows + (size_t)warp * rows_w * CPR;
    auto phys = [&](int r, int ch) { return ch ^ (((r << lgNG) ^ (ch >> lgNV)) & 7); };

    for (int bh = blockIdx.y; bh < c.B * c.H; bh += gridDim.y) {
        const int len = ld_checked(c.len + bh / c.H);
        const int n = min(len, T_out);
        const int Tq = quantized_tokens(len, c.G, c.R);
        uint32_t words[U][NW];
        float sc[U], zr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = r0 + u * rows_per_pass;
            sc[u] = zr[u] = 0.0f;
            if (t < Tq && t < n) {
                const size_t row = (size_t)bh * c.Tmax + t;
                const uint32_t* src = reinterpret_cast<const uint32_t*>(c.vq) + row * (D / Cd::P) + gi * NW;
                if constexpr (NW == 2) {
                    const uint2 x = KIVI_IN_RANGE(src, 8) ? __ldcs(reinterpret_cast<const uint2*>(src))
                                                          : make_uint2(0u, 0u);
                    words[u][0] = x.x;
                    words[u][1] = x.y;
                } else {
#pragma unroll
                    for (int w = 0; w < NW; w += 4) {
                        const uint4 x = ld_stream(src + w);
                        words[u][w] = x.x;
                        words[u][w + 1] = x.y;
                        words[u][w + 2] = x.z;
                        words[u][w + 3] = x.w;
                    }
                }
                sc[u] = KIVI_IN_RANGE(c.vscale + row * NG + gi, 4) ? __ldcs(c.vscale + row * NG + gi) : 0.0f;
                zr[u] = KIVI_IN_RANGE(c.vzero + row * NG + gi, 4) ? __ldcs(c.vzero + row * NG + gi) : 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int tw = r0 - (threadIdx.x >> lgNG) + warp * rows_w + u * rows_per_pass;  // warp's first row
            if (tw >= n)
                break;  // uniform over the warp
            const int t = r0 + u * rows_per_pass;
            if (t < n) {
                uint4* dst = wsm + (size_t)wr * CPR;
                if (t < Tq) {
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        uint32_t h2[4];
#pragma unroll
                        for (int k = 0; k < 8; k += 2) {
                            const int e = v * 8 + k;
                            h2[k / 2] = dequant_h2(
                                code_float(words[u][e / Cd::P] >> ((e % Cd::P) * BITS), Cd::M, two23),
                                code_float(words[u][(e + 1) / Cd::P] >> (((e + 1) % Cd::P) * BITS), Cd::M, two23),
                                sc[u], zr[u], sc[u], zr[u]);
                        }
                        dst[phys(wr, gi * NV + v)] = make_uint4(h2[0], h2[1], h2[2], h2[3]);
                    }
                } else {
                    const uint16_t* rs = c.vres + ((size_t)bh * RG + t % RG) * D + gi * G;
#pragma unroll
                    for (int v = 0; v < NV; ++v)
                        dst[phys(wr, gi * NV + v)] = ld_nc(rs + v * 8);
                }
            }
            __syncwarp();
            uint16_t* orow = out + ((size_t)bh * T_out + tw) * D;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int q = k * 32 + lane;
                const int rr = q >> lgCPR, x = q & (CPR - 1);
                if (tw + rr < n)
                    st_stream(orow + (size_t)rr * D + x * 8, wsm[(size_t)rr * CPR + phys(rr, x)]);
            }
            __syncwarp();
        }
    }
}

static dim3 dq_grid(const kivi_cache& c, int tiles)
{
    const int bh = c.B * c.H;
    return dim3((unsigned)(tiles > 0 ? tiles : 1), (unsigned)(bh < 65535 ? bh : 65535));
}

template <int BITS>
static void dequant_values_bits(const kivi_cache& c, uint16_t* out, int T_out, cudaStream_t s)
{
    const int U = c.G == 32 ? 4 : c.G == 64 ? 2 : 1;
    const int rows_per_cta = kDequantThreads / (c.D / c.G) * U;
    const dim3 grid = dq_grid(c, (T_out + rows_per_cta - 1) / rows_per_cta);
    // per warp: (32 / (D/G)) rows of D fp16 values
    const size_t smem = (size_t)(kDequantThreads / 32) * 64 * c.G;
    switch (c.G) {
    case 32: dequant_values_kernel<BITS, 32><<<grid, kDequantThreads, smem, s>>>(c, out, T_out); break;
    case 64: dequant_values_kernel<BITS, 64><<<grid, kDequantThreads, smem, s>>>(c, out, T_out); break;
    default:
        cudaFuncSetAttribute(dequant_values_kernel<BITS, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        dequant_values_kernel<BITS, 128><<<grid, kDequantThreads, smem, s>>>(c, out, T_out);
        break;
    }
}

cudaError_t launch_dequant(const kivi_cache& c, int which, uint16_t* out, int T_out,
                           cudaStream_t s)
{
    if (T_out <= 0)
        return cudaGetLastError();
    KIVI_SET_CHECK_RANGES(c, s, {{out, (size_t)c.B * c.H * T_out * c.D * 2}});
    if (which == 0) {
        const int lanes = ((T_out + c.G - 1) / c.G) * (c.G / kLaneTokens) * (c.D / kLaneChans);
        const dim3 grid = dq_grid(c, (lanes + kDequantThreads - 1) / kDequantThreads);
        switch (c.bits_k) {
        case 2: dequant_keys_kernel<2><<<grid, kDequantThreads, 0, s>>>(c, out, T_out); break;
        case 4: dequant_keys_kernel<4><<<grid, kDequantThreads, 0, s>>>(c, out, T_out); break;
        default: dequant_keys_kernel<8><<<grid, kDequantThreads, 0, s>>>(c, out, T_out); break;
        }
    } else {
        switch (c.bits_v) {
        case 2: dequant_values_bits<2>(c, out, T_out, s); break;
        case 4: dequant_values_bits<4>(c, out, T_out, s); break;
        default: dequant_values_bits<8>(c, out, T_out, s); break;
        }
    }
    return cudaGetLastError();
}

#ifdef KIVI_CHECKS
int32_t check_word_dequant() { return take_check_word(); }
#endif

}  // namespace kivi
