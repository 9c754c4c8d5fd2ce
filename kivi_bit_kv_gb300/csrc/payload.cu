// payload.cu -- the compact payload of a cache (include/kivi.h, "compact
// payload"): export to and import from caller memory, in the format the
// header documents.  CacheSeek PR #4 (change notes) stores a quantized layer
// as its codes, scales and offsets, copied to host memory; here one kernel
// gathers the packed codes, statistics and fp16 residual of every slice
// straight into the destination (pinned host memory is written over the
// CPU-GPU link without a staging copy), and one kernel scatters a payload
// back into a cache.
//
// Each row of CTAs takes a contiguous range of slices and computes the first
// slice's offset from len[] (a prefix sum of kivi_cache_bytes over the
// sequences, one block-wide scan), the others by adding slice sizes, so the
// kernels need no scratch memory and no second launch; the copies move
// 16-byte units.
#include <algorithm>

#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

constexpr int kPayloadThreads = 256;

// Sections of one (b, h) slice of a sequence of n tokens, in 16-byte units:
// kq, kscale, kzero, vq, vscale, vzero, key residual, value residual.
struct SliceGeom {
    int Tq, res;
    uint32_t u[8];
};

__host__ __device__ __forceinline__ SliceGeom slice_geom(int n, int D, int bits_k, int bits_v, int G, int R)
{
    SliceGeom g;
    g.Tq = quantized_tokens(n, G, R);
    g.res = n - g.Tq;
    const uint64_t Tq = (uint64_t)g.Tq, d = (uint64_t)D, ng = (uint64_t)G;
    g.u[0] = (uint32_t)(Tq * d * (uint64_t)bits_k / 128u);  // Tq D b / 8 bytes
    g.u[1] = g.u[2] = (uint32_t)((Tq / ng) * d / 4u);
    g.u[3] = (uint32_t)(Tq * d * (uint64_t)bits_v / 128u);
    g.u[4] = g.u[5] = (uint32_t)(Tq * (d / ng) / 4u);
    g.u[6] = g.u[7] = (uint32_t)((uint64_t)g.res * d / 8u);
    return g;
}

__host__ __device__ __forceinline__ size_t slice_units(const SliceGeom& g)
{
    size_t s = 0;
    for (int i = 0; i < 8; ++i)
        s += g.u[i];
    return s;
}

// Header plus the padded len[] table, in 16-byte units.
__host__ __device__ __forceinline__ size_t head_units(int B) { return 4 + (size_t)(B + 3) / 4; }

// Payload offset (16-byte units) of the slices of sequence b0, and the total
// payload size, from lens[0 .. B): a block-wide prefix over the sequences.
// `bad` receives whether any length lies outside [0, Tmax].  Whole CTA.
struct PayloadScan {
    size_t base, total;
    bool bad;
};

__device__ __forceinline__ PayloadScan payload_scan(const kivi_cache& c, const int32_t* lens, int b0)
{
    __shared__ unsigned long long sb[kPayloadThreads / 32], st[kPayloadThreads / 32];
    __shared__ int sbad[kPayloadThreads / 32];
    unsigned long long before = 0, total = 0;
    int bad = 0;
    for (int b = threadIdx.x; b < c.B; b += kPayloadThreads) {
        const int n = ld_checked(lens + b);
        if (n < 0 || n > c.Tmax) {
            bad = 1;
            continue;
        }
        const unsigned long long u =
            (unsigned long long)c.H * slice_units(slice_geom(n, c.D, c.bits_k, c.bits_v, c.G, c.R));
        total += u;
        if (b < b0)
            before += u;
    }
    for (int m = 16; m > 0; m >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, m);
        total += __shfl_xor_sync(0xffffffffu, total, m);
        bad |= __shfl_xor_sync(0xffffffffu, bad, m);
    }
    const int warp = threadIdx.x >> 5;
    __syncthreads();  // the arrays may still be read by a previous call
    if ((threadIdx.x & 31) == 0) {
        sb[warp] = before;
        st[warp] = total;
        sbad[warp] = bad;
    }
    __syncthreads();
    PayloadScan r{head_units(c.B), head_units(c.B), false};
    for (int w = 0; w < kPayloadThreads / 32; ++w) {
        r.base += sb[w];
        r.total += st[w];
        r.bad |= sbad[w] != 0;
    }
    return r;
}

// Source (export) or destination (import) of unit r of section s of slice bh
// in the cache.
__device__ __forceinline__ uint4* cache_unit(const kivi_cache& c, size_t bh, const SliceGeom& g, int s,
                                             uint32_t r)
{
    const size_t D = c.D, T = c.Tmax, G = c.G, RG = (size_t)c.R + c.G;
    switch (s) {
    case 0: return reinterpret_cast<uint4*>(c.kq + bh * (T / (32 / c.bits_k)) * D) + r;
    case 1: return reinterpret_cast<uint4*>(c.kscale + bh * (T / G) * D) + r;
    case 2: return reinterpret_cast<uint4*>(c.kzero + bh * (T / G) * D) + r;
    case 3: return reinterpret_cast<uint4*>(c.vq + bh * T * (D / (32 / c.bits_v))) + r;
    case 4: return reinterpret_cast<uint4*>(c.vscale + bh * T * (D / G)) + r;
    case 5: return reinterpret_cast<uint4*>(c.vzero + bh * T * (D / G)) + r;
    default: {
        const uint32_t upr = (uint32_t)D / 8;  // units per fp16 row
        const uint32_t row = r / upr, col = r - row * upr;
        const size_t slot = ((size_t)g.Tq + row) % RG;
        uint16_t* ring = s == 6 ? c.kres : c.vres;
        return reinterpret_cast<uint4*>(ring + (bh * RG + slot) * D) + col;
    }
    }
}

// Section and unit within it of slice unit u.
__device__ __forceinline__ int section_of(const SliceGeom& g, uint32_t u, uint32_t& r)
{
    int s = 0;
#pragma unroll
    for (int i = 0; i < 7; ++i)
        if (s == i && u >= g.u[i]) {
            u -= g.u[i];
            s = i + 1;
        }
    r = u;
    return s;
}

// Slices of CTA row blockIdx.y: a contiguous range [bh0, bh1) of the B H
// slices, so one prefix scan gives the first offset and the others follow.
__device__ __forceinline__ bool slice_range(const kivi_cache& c, int& bh0, int& bh1)
{
    const int BH = c.B * c.H;
    const int per = (BH + gridDim.y - 1) / gridDim.y;
    bh0 = blockIdx.y * per;
    bh1 = min(BH, bh0 + per);
    return bh0 < bh1;
}

__global__ void __launch_bounds__(kPayloadThreads)
export_kernel(kivi_cache c, uint4* __restrict__ dst, size_t dst_units, uint64_t fingerprint, int32_t* status)
{
    int bh0, bh1;
    if (!slice_range(c, bh0, bh1))
        return;
    const PayloadScan ps = payload_scan(c, c.len, bh0 / c.H);
    if (ps.bad)
        return;  // len[] is the library's own state: cannot happen
    if (ps.total > dst_units) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            st_checked(status, (int32_t)KIVI_EWORKSPACE);
        return;
    }
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        uint32_t* hd = reinterpret_cast<uint32_t*>(dst);
        const int32_t fields[7] = {c.B, c.H, c.D, c.bits_k, c.bits_v, c.G, c.R};
        for (int i = threadIdx.x; i < 16 + 4 * (int)(head_units(c.B) - 4); i += kPayloadThreads) {
            uint32_t w = 0;
            if (i == 0) w = KIVI_PAYLOAD_MAGIC;
            else if (i == 1) w = KIVI_PAYLOAD_VERSION;
            else if (i == 2) w = (uint32_t)fingerprint;
            else if (i == 3) w = (uint32_t)(fingerprint >> 32);
            else if (i < 11) w = (uint32_t)fields[i - 4];
            else if (i >= 16 && i - 16 < c.B) w = (uint32_t)ld_checked(c.len + (i - 16));
            st_checked(hd + i, w);
        }
    }
    size_t off = ps.base;  // offset of slice (bh0 / H, 0)
    for (int bh = bh0 - bh0 % c.H; bh < bh1; ++bh) {
        const SliceGeom g = slice_geom(ld_checked(c.len + bh / c.H), c.D, c.bits_k, c.bits_v, c.G, c.R);
        const uint32_t U = (uint32_t)slice_units(g);
        if (bh >= bh0)
            for (uint32_t u = blockIdx.x * kPayloadThreads + threadIdx.x; u < U; u += gridDim.x * kPayloadThreads) {
                uint32_t r;
                const int s = section_of(g, u, r);
                st_checked(dst + off + u, ld_nc(reinterpret_cast<const uint16_t*>(cache_unit(c, bh, g, s, r))));
            }
        off += U;
    }
}

__global__ void __launch_bounds__(kPayloadThreads)
import_kernel(kivi_cache c, const uint4* __restrict__ src, size_t src_units, uint64_t fingerprint,
              int32_t* status)
{
    const uint32_t* hd = reinterpret_cast<const uint32_t*>(src);
    const int32_t fields[7] = {c.B, c.H, c.D, c.bits_k, c.bits_v, c.G, c.R};
    bool ok = ld_checked(hd) == KIVI_PAYLOAD_MAGIC && ld_checked(hd + 1) == KIVI_PAYLOAD_VERSION &&
              ld_checked(hd + 2) == (uint32_t)fingerprint && ld_checked(hd + 3) == (uint32_t)(fingerprint >> 32);
#pragma unroll
    for (int i = 0; i < 7; ++i)
        ok = ok && (int32_t)ld_checked(hd + 4 + i) == fields[i];
    if (!ok) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            st_checked(status, (int32_t)KIVI_EINVAL);
        return;
    }
    const int32_t* lens = reinterpret_cast<const int32_t*>(hd + 16);
    int bh0, bh1;
    if (!slice_range(c, bh0, bh1))
        return;
    const PayloadScan ps = payload_scan(c, lens, bh0 / c.H);
    if (ps.bad || ps.total > src_units) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            st_checked(status, (int32_t)(ps.bad ? KIVI_ECAPACITY : KIVI_EWORKSPACE));
        return;
    }
    size_t off = ps.base;  // offset of slice (bh0 / H, 0)
    for (int bh = bh0 - bh0 % c.H; bh < bh1; ++bh) {
        const int b = bh / c.H, n = ld_checked(lens + b);
        const SliceGeom g = slice_geom(n, c.D, c.bits_k, c.bits_v, c.G, c.R);
        const uint32_t U = (uint32_t)slice_units(g);
        if (bh >= bh0) {
            for (uint32_t u = blockIdx.x * kPayloadThreads + threadIdx.x; u < U; u += gridDim.x * kPayloadThreads) {
                uint32_t r;
                const int s = section_of(g, u, r);
                st_checked(cache_unit(c, bh, g, s, r), ld_checked(src + off + u));
            }
            if (bh % c.H == 0 && blockIdx.x == 0 && threadIdx.x == 0)
                st_checked(c.len + b, n);
        }
        off += U;
    }
}

// Rows of CTAs over contiguous slice ranges (at most four rows per SM), and
// CTAs per row splitting each slice's units when there are few slices.
static dim3 payload_grid(const kivi_cache& c)
{
    const int BH = c.B * c.H;
    const int y = std::min(BH, 4 * sm_count());
    const int x = std::max(1, std::min(64, (4 * sm_count() + BH - 1) / BH));
    return dim3((unsigned)x, (unsigned)y);
}

size_t payload_bytes(const kivi_cache& c, const int32_t* lens)
{
    size_t u = head_units(c.B);
    for (int b = 0; b < c.B; ++b)
        u += (size_t)c.H * slice_units(slice_geom(lens[b], c.D, c.bits_k, c.bits_v, c.G, c.R));
    return 16 * u;
}

cudaError_t launch_export(const kivi_cache& c, void* dst, size_t dst_bytes, uint64_t fingerprint,
                          int32_t* status, cudaStream_t s)
{
    KIVI_SET_CHECK_RANGES(c, s, {{dst, dst_bytes}, {status, 4}});
    export_kernel<<<payload_grid(c), kPayloadThreads, 0, s>>>(c, static_cast<uint4*>(dst), dst_bytes / 16,
                                                             fingerprint, status);
    return cudaGetLastError();
}

cudaError_t launch_import(const kivi_cache& c, const void* src, size_t src_bytes, uint64_t fingerprint,
                          int32_t* status, cudaStream_t s)
{
    KIVI_SET_CHECK_RANGES(c, s, {{src, src_bytes}, {status, 4}});
    import_kernel<<<payload_grid(c), kPayloadThreads, 0, s>>>(c, static_cast<const uint4*>(src), src_bytes / 16,
                                                             fingerprint, status);
    return cudaGetLastError();
}

#ifdef KIVI_CHECKS
int32_t check_word_payload() { return take_check_word(); }
#endif

}  // namespace kivi
