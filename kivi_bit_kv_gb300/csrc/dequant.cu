// dequant.cu -- materialize: unpack codes and dequantize to fp16
// (x_hat = fp16_rne(fmaf(code, scale, zero))), residual rows copied from the
// ring.  CacheSeek PR #4 change notes: "decode after materialize" moves only
// the compact qdata/scale/offset to the device and dequantizes there.
//
// HBM-bound: reads b/8 bytes of code plus the statistics per element and
// writes 2 bytes per element with 16-byte stores.
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

// Keys: one lane = 16 tokens x 8 channels of a G-token group.
template <int BITS>
__global__ void __launch_bounds__(256)
dequant_keys_kernel(kivi_cache c, uint16_t* __restrict__ out, int T_out, int units_per_bh)
{
    using Cd = Codec<BITS>;
    const int D = c.D;
    const int S = c.G / kLaneTokens;
    const int NC = D / kLaneChans;
    const int lanes_per_unit = S * NC;
    const long long total = (long long)c.B * c.H * units_per_bh * lanes_per_unit;
    const long long stride = (long long)gridDim.x * blockDim.x;
    const int RG = c.R + c.G;

    for (long long task = (long long)blockIdx.x * blockDim.x + threadIdx.x; task < total;
         task += stride) {
        const int s = (int)(task % S);
        const int j = (int)((task / S) % NC);
        const long long unit = task / lanes_per_unit;
        const int g = (int)(unit % units_per_bh);
        const size_t bh = (size_t)(unit / units_per_bh);
        const int b = (int)(bh / c.H);
        const int len = c.len[b];
        const int n = min(len, T_out);
        const int t0 = g * c.G + s * kLaneTokens;
        if (t0 >= n)
            continue;
        const int Tq = quantized_tokens(len, c.G, c.R);
        uint16_t* dst = out + (bh * T_out) * D + (size_t)j * kLaneChans;

        if (t0 + kLaneTokens <= Tq) {
            const int32_t* src = c.kq + (bh * (size_t)(c.Tmax / Cd::P) + t0 / Cd::P) * D +
                                 (size_t)j * kLaneChans;
            uint4 wlo[Cd::kWordRows], whi[Cd::kWordRows];
#pragma unroll
            for (int w = 0; w < Cd::kWordRows; ++w) {
                wlo[w] = ld_stream(src + (size_t)w * D);
                whi[w] = ld_stream(src + (size_t)w * D + 4);
            }
            const size_t so = (bh * (size_t)(c.Tmax / c.G) + g) * D + (size_t)j * kLaneChans;
            const float4 s0 = ld_nc_f4(c.kscale + so), s1 = ld_nc_f4(c.kscale + so + 4);
            const float4 z0 = ld_nc_f4(c.kzero + so), z1 = ld_nc_f4(c.kzero + so + 4);
            const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
            const float zr[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
            for (int i = 0; i < kLaneTokens; ++i) {
                if (t0 + i >= n)
                    break;  // out holds only T_out rows
                const int w = i / Cd::P, sh = (i % Cd::P) * BITS;
                uint32_t h[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t word = k < 4 ? u4_word(wlo[w], k) : u4_word(whi[w], k - 4);
                    h[k] = dequant_h((word >> sh) & Cd::M, sc[k], zr[k]);
                }
                st_stream(dst + (size_t)(t0 + i) * D,
                          make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16),
                                     h[4] | (h[5] << 16), h[6] | (h[7] << 16)));
            }
        } else {
            for (int i = 0; i < kLaneTokens; ++i) {
                const int t = t0 + i;
                if (t >= Tq && t < n)
                    st_stream(dst + (size_t)t * D,
                              ld_nc(c.kres + (bh * RG + t % RG) * D + (size_t)j * kLaneChans));
            }
        }
    }
}

// Values: one lane = 8 channels of one token; four rows in flight per thread.
template <int BITS>
__global__ void __launch_bounds__(256)
dequant_values_kernel(kivi_cache c, uint16_t* __restrict__ out, int T_out)
{
    using Cd = Codec<BITS>;
    constexpr int U = 4;
    const int D = c.D;
    const int NC = D / kLaneChans;
    const int LPG = c.G / kLaneChans;
    const long long total = (long long)c.B * c.H * T_out * NC;
    const long long stride = (long long)gridDim.x * blockDim.x;
    const int RG = c.R + c.G;

    for (long long base = (long long)blockIdx.x * blockDim.x + threadIdx.x; base < total;
         base += U * stride) {
        uint32_t wl[U], wh[U];
        float sc[U], zr[U];
        uint4 rr[U];
        int kind[U];  // 0 nothing, 1 quantized, 2 residual
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long task = base + u * stride;
            kind[u] = 0;
            wl[u] = wh[u] = 0u;
            sc[u] = zr[u] = 0.0f;
            rr[u] = make_uint4(0u, 0u, 0u, 0u);
            if (task >= total)
                continue;
            const int j = (int)(task % NC);
            const long long row = task / NC;
            const int t = (int)(row % T_out);
            const size_t bh = (size_t)(row / T_out);
            const int len = c.len[(int)(bh / c.H)];
            if (t >= len)
                continue;
            const int Tq = quantized_tokens(len, c.G, c.R);
            if (t < Tq) {
                kind[u] = 1;
                const size_t vrow = bh * (size_t)c.Tmax + t;
                const int32_t* vw = c.vq + vrow * (D / Cd::P);
                if (BITS == 2) {
                    wl[u] = (uint32_t)__ldcs(vw + (j >> 1)) >> ((j & 1) * 16);
                } else if (BITS == 4) {
                    wl[u] = (uint32_t)__ldcs(vw + j);
                } else {
                    const uint2 p = __ldcs(reinterpret_cast<const uint2*>(vw) + j);
                    wl[u] = p.x;
                    wh[u] = p.y;
                }
                const size_t so = vrow * (D / c.G) + j / LPG;
                sc[u] = __ldg(c.vscale + so);
                zr[u] = __ldg(c.vzero + so);
            } else {
                kind[u] = 2;
                rr[u] = ld_nc(c.vres + (bh * RG + t % RG) * D + (size_t)j * kLaneChans);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (kind[u] == 0)
                continue;
            const long long task = base + u * stride;
            const int j = (int)(task % NC);
            const long long row = task / NC;
            uint4 v = rr[u];
            if (kind[u] == 1) {
                uint32_t h[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t code = BITS == 8 ? ((k < 4 ? wl[u] : wh[u]) >> ((k & 3) * 8)) & 0xffu
                                                    : (wl[u] >> (k * BITS)) & Cd::M;
                    h[k] = dequant_h(code, sc[u], zr[u]);
                }
                v = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                               h[6] | (h[7] << 16));
            }
            st_stream(out + (size_t)row * D + (size_t)j * kLaneChans, v);
        }
    }
}

cudaError_t launch_dequant(const kivi_cache& c, int which, uint16_t* out, int T_out,
                           cudaStream_t s)
{
    if (T_out <= 0)
        return cudaGetLastError();
    const int cap = sm_count() * 16;
    if (which == 0) {
        const int units = (T_out + c.G - 1) / c.G;
        const long long threads = (long long)c.B * c.H * units * (c.G / kLaneTokens) *
                                  (c.D / kLaneChans);
        long long grid = (threads + 255) / 256;
        if (grid > cap)
            grid = cap;
        switch (c.bits_k) {
        case 2: dequant_keys_kernel<2><<<(int)grid, 256, 0, s>>>(c, out, T_out, units); break;
        case 4: dequant_keys_kernel<4><<<(int)grid, 256, 0, s>>>(c, out, T_out, units); break;
        default: dequant_keys_kernel<8><<<(int)grid, 256, 0, s>>>(c, out, T_out, units); break;
        }
    } else {
        const long long threads = (long long)c.B * c.H * T_out * (c.D / kLaneChans);
        long long grid = ((threads + 3) / 4 + 255) / 256;
        if (grid > cap)
            grid = cap;
        switch (c.bits_v) {
        case 2: dequant_values_kernel<2><<<(int)grid, 256, 0, s>>>(c, out, T_out); break;
        case 4: dequant_values_kernel<4><<<(int)grid, 256, 0, s>>>(c, out, T_out); break;
        default: dequant_values_kernel<8><<<(int)grid, 256, 0, s>>>(c, out, T_out); break;
        }
    }
    return cudaGetLastError();
}

}  // namespace kivi
