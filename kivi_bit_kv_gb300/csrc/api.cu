// api.cu -- the C ABI of libkivi (include/kivi.h): argument validation,
// status codes, byte accounting and dispatch to the kernel launchers.
//
// Unknown or unsupported configurations are rejected with a message that
// names the accepted values, the way the vLLM TurboQuant config rejects an
// unknown preset (vllm/model_executor/layers/quantization/turboquant/config.py,
// `from_cache_dtype`).
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdarg>
#include <cstdio>
#include <string>

#include "kivi.h"
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace {

thread_local std::string g_last_error;

int32_t fail(int32_t status, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int32_t ok()
{
    g_last_error.clear();
    return KIVI_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// An NVTX range around each call that launches work, named after the call,
// so that a timeline tool shows the host call above its kernels (the NVTX
// calls do nothing unless such a tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
bool bits_ok(int b) { return b == 2 || b == 4 || b == 8; }

int32_t check_sizes(const kivi_cache* c)
{
    if (!c)
        return fail(KIVI_EINVAL, "cache descriptor is NULL");
    if (c->B < 1 || c->H < 1)
        return fail(KIVI_EINVAL, "B=%d H=%d: both must be >= 1", c->B, c->H);
    if (c->D != 64 && c->D != 128 && c->D != 256)
        return fail(KIVI_EINVAL, "head dim D=%d unsupported; valid: 64, 128, 256", c->D);
    if (!bits_ok(c->bits_k) || !bits_ok(c->bits_v))
        return fail(KIVI_EINVAL, "bits_k=%d bits_v=%d unsupported; valid: 2, 4, 8", c->bits_k,
                    c->bits_v);
    if (c->G != 32 && c->G != 64 && c->G != 128)
        return fail(KIVI_EINVAL, "group size G=%d unsupported; valid: 32, 64, 128", c->G);
    if (c->D % c->G != 0)
        return fail(KIVI_EINVAL, "D=%d is not a multiple of G=%d (value groups span channels)",
                    c->D, c->G);
    if (c->R < 0 || c->R % c->G != 0)
        return fail(KIVI_EINVAL, "residual R=%d must be >= 0 and a multiple of G=%d", c->R, c->G);
    if (c->Tmax < 1 || c->Tmax % c->G != 0)
        return fail(KIVI_EINVAL, "capacity Tmax=%d must be >= 1 and a multiple of G=%d", c->Tmax,
                    c->G);
    if (c->Tmax > (1 << 24) || c->R > (1 << 24))
        return fail(KIVI_EINVAL, "capacity Tmax=%d / residual R=%d above 2^24 tokens", c->Tmax, c->R);
    return KIVI_OK;
}

int32_t check_cache(const kivi_cache* c)
{
    int32_t st = check_sizes(c);
    if (st != KIVI_OK)
        return st;
    const void* ptrs[] = {c->kq, c->kscale, c->kzero, c->vq, c->vscale,
                          c->vzero, c->kres, c->vres, c->len};
    const char* names[] = {"kq", "kscale", "kzero", "vq", "vscale", "vzero", "kres", "vres", "len"};
    for (int i = 0; i < 9; ++i) {
        if (!ptrs[i])
            return fail(KIVI_EINVAL, "cache buffer %s is NULL", names[i]);
        if (!aligned16(ptrs[i]))
            return fail(KIVI_EINVAL, "cache buffer %s is not 16-byte aligned", names[i]);
    }
    return KIVI_OK;
}

int32_t check_ptr(const void* p, const char* name, bool need16 = true)
{
    if (!p)
        return fail(KIVI_EINVAL, "%s is NULL", name);
    if (need16 ? !aligned16(p) : ((uintptr_t)p & 3u) != 0)
        return fail(KIVI_EINVAL, "%s is not %d-byte aligned", name, need16 ? 16 : 4);
    return KIVI_OK;
}

int32_t launched(cudaError_t e)
{
    if (e != cudaSuccess)
        return fail(KIVI_ECUDA, "CUDA launch failed: %s", cudaGetErrorString(e));
    return ok();
}

size_t ws_bytes(const kivi_cache& c, int Hq)
{
    const size_t rows = (size_t)c.B * Hq * kivi::pv_chunks(c, Hq);
    return rows * ((size_t)c.D + 2) * sizeof(float);
}

}  // namespace

extern "C" {

int32_t kivi_abi_version(void) { return KIVI_ABI_VERSION; }

const char* kivi_status_string(int32_t status)
{
    switch (status) {
    case KIVI_OK: return "ok";
    case KIVI_EINVAL: return "invalid argument";
    case KIVI_ECAPACITY: return "sequence capacity (Tmax) exceeded";
    case KIVI_ECUDA: return "CUDA error";
    case KIVI_ETIMEOUT: return "device wait timed out";
    case KIVI_EWORKSPACE: return "workspace too small";
    case KIVI_ECHECK: return "device bounds check failed";
    default: return "unknown status";
    }
}

const char* kivi_last_error(void) { return g_last_error.c_str(); }

int32_t kivi_cache_validate(const kivi_cache* c)
{
    const int32_t st = check_cache(c);
    return st != KIVI_OK ? st : ok();
}

size_t kivi_buffer_bytes(const kivi_cache* c, int32_t buffer)
{
    if (check_sizes(c) != KIVI_OK)
        return 0;
    const size_t BH = (size_t)c->B * c->H, D = c->D, T = c->Tmax, G = c->G;
    const size_t Pk = 32 / c->bits_k, Pv = 32 / c->bits_v, RG = (size_t)c->R + c->G;
    switch (buffer) {
    case KIVI_BUF_KQ: return BH * (T / Pk) * D * 4;
    case KIVI_BUF_KSCALE:
    case KIVI_BUF_KZERO: return BH * (T / G) * D * 4;
    case KIVI_BUF_VQ: return BH * T * (D / Pv) * 4;
    case KIVI_BUF_VSCALE:
    case KIVI_BUF_VZERO: return BH * T * (D / G) * 4;
    case KIVI_BUF_KRES:
    case KIVI_BUF_VRES: return BH * RG * D * 2;
    case KIVI_BUF_LEN: return (size_t)c->B * 4;
    default: return 0;
    }
}

size_t kivi_cache_bytes(int32_t T, int32_t D, int32_t bits, int32_t G, int32_t R, int32_t which)
{
    if (T < 0 || D < 1 || !bits_ok(bits) || G < 1 || D % G != 0 || R < 0 ||
        (which != 0 && which != 1))
        return 0;
    const size_t Tq = (size_t)kivi::quantized_tokens(T, G, R);
    const size_t res = (size_t)T - Tq;
    const size_t codes = Tq * (size_t)D * bits / 8;
    const size_t stats = which == 0 ? (Tq / G) * (size_t)D * 8 : Tq * (size_t)(D / G) * 8;
    return codes + stats + res * (size_t)D * 2;
}

int32_t kivi_quant_keys(const kivi_cache* c, const uint16_t* K, int32_t T,
                        const int32_t* seq_lens, void* stream)
{
    NvtxRange range_("kivi_quant_keys");
    int32_t st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if (T < 0 || T > c->Tmax)
        return fail(KIVI_EINVAL, "T=%d outside [0, Tmax=%d]", T, c->Tmax);
    if (T > 0 && (st = check_ptr(K, "K")) != KIVI_OK)
        return st;
    if (seq_lens && ((uintptr_t)seq_lens & 3u))
        return fail(KIVI_EINVAL, "seq_lens is not 4-byte aligned");
    return launched(kivi::launch_quant_keys(*c, K, T, seq_lens, (cudaStream_t)stream));
}

int32_t kivi_quant_values(const kivi_cache* c, const uint16_t* V, int32_t T,
                          const int32_t* seq_lens, void* stream)
{
    NvtxRange range_("kivi_quant_values");
    int32_t st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if (T < 0 || T > c->Tmax)
        return fail(KIVI_EINVAL, "T=%d outside [0, Tmax=%d]", T, c->Tmax);
    if (T > 0 && (st = check_ptr(V, "V")) != KIVI_OK)
        return st;
    if (seq_lens && ((uintptr_t)seq_lens & 3u))
        return fail(KIVI_EINVAL, "seq_lens is not 4-byte aligned");
    return launched(kivi::launch_quant_values(*c, V, T, seq_lens, (cudaStream_t)stream));
}

int32_t kivi_dequant(const kivi_cache* c, int32_t which, uint16_t* out, int32_t T_out,
                     void* stream)
{
    NvtxRange range_("kivi_dequant");
    int32_t st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if (which != 0 && which != 1)
        return fail(KIVI_EINVAL, "which=%d; valid: 0 (keys), 1 (values)", which);
    if (T_out < 0 || T_out > c->Tmax)
        return fail(KIVI_EINVAL, "T_out=%d outside [0, Tmax=%d]", T_out, c->Tmax);
    if (T_out > 0 && (st = check_ptr(out, "out")) != KIVI_OK)
        return st;
    return launched(kivi::launch_dequant(*c, which, out, T_out, (cudaStream_t)stream));
}

int32_t kivi_append_token(const kivi_cache* c, const uint16_t* k, const uint16_t* v,
                          int32_t* status, void* stream)
{
    NvtxRange range_("kivi_append_token");
    int32_t st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if ((st = check_ptr(k, "k")) != KIVI_OK || (st = check_ptr(v, "v")) != KIVI_OK ||
        (st = check_ptr(status, "status", false)) != KIVI_OK)
        return st;
    return launched(kivi::launch_append(*c, k, v, status, (cudaStream_t)stream));
}

static int32_t check_heads(const kivi_cache* c, int32_t Hq)
{
    if (Hq < c->H || Hq % c->H != 0 || Hq / c->H > 16)
        return fail(KIVI_EINVAL, "Hq=%d must be a multiple of H=%d with Hq/H <= 16", Hq, c->H);
    // one CTA per (b, h, chunk) in a 1-D grid
    const long long ctas = (long long)c->B * c->H * kivi::pv_chunks(*c, Hq);
    if (ctas >= (1ll << 31))
        return fail(KIVI_EINVAL, "B*H*chunks = %lld decode CTAs; the grid holds fewer than 2^31", ctas);
    return KIVI_OK;
}

static int32_t check_logits(const kivi_cache* c, const float* logits, int32_t ld)
{
    int32_t st = check_ptr(logits, "logits");
    if (st != KIVI_OK)
        return st;
    if (ld < c->Tmax || ld % 4 != 0)
        return fail(KIVI_EINVAL, "ld_logits=%d must be >= Tmax=%d and a multiple of 4", ld,
                    c->Tmax);
    return KIVI_OK;
}

}  // extern "C"

namespace kivi {

// The argument checks of kivi_decode_pv other than the workspace's, for
// entry points that bring their own workspace.
int32_t check_decode_pv_args(const kivi_cache* c, const float* logits, int32_t ld_logits, int32_t Hq,
                             const float* out)
{
    int32_t st = check_cache(c);
    if (st != KIVI_OK || (st = check_heads(c, Hq)) != KIVI_OK ||
        (st = check_logits(c, logits, ld_logits)) != KIVI_OK || (st = check_ptr(out, "out")) != KIVI_OK)
        return st;
    return KIVI_OK;
}

}  // namespace kivi

extern "C" {

int32_t kivi_decode_qk(const kivi_cache* c, const uint16_t* q, int32_t Hq, float sm_scale,
                       float* logits, int32_t ld_logits, void* stream)
{
    NvtxRange range_("kivi_decode_qk");
    int32_t st = check_cache(c);
    if (st != KIVI_OK || (st = check_heads(c, Hq)) != KIVI_OK ||
        (st = check_ptr(q, "q")) != KIVI_OK || (st = check_logits(c, logits, ld_logits)) != KIVI_OK)
        return st;
    return launched(
        kivi::launch_decode_qk(*c, q, Hq, sm_scale, logits, ld_logits, (cudaStream_t)stream));
}

size_t kivi_workspace_bytes(const kivi_cache* c, int32_t Hq)
{
    if (check_sizes(c) != KIVI_OK || Hq < 1)
        return 0;
    const size_t pv = ws_bytes(*c, Hq), fused = kivi::stream_ws_bytes(*c, Hq);
    return pv > fused ? pv : fused;
}

int32_t kivi_decode_pv(const kivi_cache* c, const float* logits, int32_t ld_logits, int32_t Hq,
                       float* out, void* ws, size_t ws_bytes_given, void* stream)
{
    NvtxRange range_("kivi_decode_pv");
    int32_t st = check_cache(c);
    if (st != KIVI_OK || (st = check_heads(c, Hq)) != KIVI_OK ||
        (st = check_logits(c, logits, ld_logits)) != KIVI_OK ||
        (st = check_ptr(out, "out")) != KIVI_OK || (st = check_ptr(ws, "ws")) != KIVI_OK)
        return st;
    const size_t need = ws_bytes(*c, Hq);
    if (ws_bytes_given < need)
        return fail(KIVI_EWORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes_given, need);
    const size_t rows = (size_t)c->B * Hq * kivi::pv_chunks(*c, Hq);
    float* ws_o = static_cast<float*>(ws);
    float* ws_m = ws_o + rows * c->D;
    float* ws_l = ws_m + rows;
    return launched(kivi::launch_decode_pv(*c, logits, ld_logits, Hq, out, ws_o, ws_m, ws_l,
                                           (cudaStream_t)stream));
}

int32_t kivi_decode_attention(const kivi_cache* c, const uint16_t* q, int32_t Hq, float sm_scale,
                              float* out, void* ws, size_t ws_bytes_given, void* stream)
{
    NvtxRange range_("kivi_decode_attention");
    int32_t st = check_cache(c);
    if (st != KIVI_OK || (st = check_heads(c, Hq)) != KIVI_OK || (st = check_ptr(q, "q")) != KIVI_OK ||
        (st = check_ptr(out, "out")) != KIVI_OK || (st = check_ptr(ws, "ws")) != KIVI_OK)
        return st;
    const size_t need = kivi::stream_ws_bytes(*c, Hq);
    if (ws_bytes_given < need)
        return fail(KIVI_EWORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes_given, need);
    return launched(kivi::launch_decode_attention(*c, q, Hq, sm_scale, out, static_cast<float*>(ws),
                                                  (cudaStream_t)stream));
}

// ------------------------------------------------------ compact payload ---

uint64_t kivi_codec_fingerprint(const kivi_cache* c)
{
    if (check_sizes(c) != KIVI_OK)
        return 0;
    // FNV-1a 64 over "KIVI" + int32 {layout 1, D, bits_k, bits_v, G, R, 4}, little-endian
    const int32_t f[7] = {1, c->D, c->bits_k, c->bits_v, c->G, c->R, 4};
    uint8_t bytes[32] = {'K', 'I', 'V', 'I'};
    for (int i = 0; i < 7; ++i)
        for (int k = 0; k < 4; ++k)
            bytes[4 + 4 * i + k] = (uint8_t)((uint32_t)f[i] >> (8 * k));
    uint64_t hsh = 0xcbf29ce484222325ull;
    for (int i = 0; i < 32; ++i) {
        hsh ^= bytes[i];
        hsh *= 0x100000001b3ull;
    }
    return hsh;
}

size_t kivi_payload_bytes(const kivi_cache* c, const int32_t* lens)
{
    if (check_sizes(c) != KIVI_OK || !lens)
        return 0;
    for (int b = 0; b < c->B; ++b)
        if (lens[b] < 0 || lens[b] > c->Tmax)
            return 0;
    return kivi::payload_bytes(*c, lens);
}

static int32_t check_payload_buffer(const void* p, size_t bytes, const kivi_cache* c, const char* name)
{
    int32_t st = check_ptr(p, name);
    if (st != KIVI_OK)
        return st;
    const size_t head = KIVI_PAYLOAD_HEADER_BYTES + (size_t)(c->B + 3) / 4 * 16;
    if (bytes < head)
        return fail(KIVI_EINVAL, "%s holds %zu bytes, fewer than the %zu of the header and lengths", name,
                    bytes, head);
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return fail(KIVI_EINVAL, "%s: cudaPointerGetAttributes failed", name);
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeHost && a.type != cudaMemoryTypeManaged)
        return fail(KIVI_EINVAL, "%s must be device memory or pinned (page-locked) host memory", name);
    return KIVI_OK;
}

int32_t kivi_export(const kivi_cache* c, void* dst, size_t dst_bytes, int32_t* status, void* stream)
{
    NvtxRange range_("kivi_export");
    int32_t st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if ((st = check_payload_buffer(dst, dst_bytes, c, "dst")) != KIVI_OK ||
        (st = check_ptr(status, "status", false)) != KIVI_OK)
        return st;
    return launched(kivi::launch_export(*c, dst, dst_bytes, kivi_codec_fingerprint(c), status,
                                        (cudaStream_t)stream));
}

int32_t kivi_import(const kivi_cache* c, const void* src, size_t src_bytes, int32_t* status, void* stream)
{
    NvtxRange range_("kivi_import");
    int32_t st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if ((st = check_payload_buffer(src, src_bytes, c, "src")) != KIVI_OK ||
        (st = check_ptr(status, "status", false)) != KIVI_OK)
        return st;
    return launched(kivi::launch_import(*c, src, src_bytes, kivi_codec_fingerprint(c), status,
                                        (cudaStream_t)stream));
}

int32_t kivi_check_status(int32_t* status)
{
    if (!status)
        return fail(KIVI_EINVAL, "status is NULL");
    int32_t first = KIVI_OK;
#ifdef KIVI_CHECKS
    const int32_t words[] = {kivi::check_word_quant(),    kivi::check_word_dequant(),
                             kivi::check_word_append(),   kivi::check_word_payload(),
                             kivi::check_word_decode(),   kivi::check_word_decode_d64(),
                             kivi::check_word_decode_d128(), kivi::check_word_decode_d256()};
    for (const int32_t w : words) {
        if (w == KIVI_ECUDA)
            return fail(KIVI_ECUDA, "reading the device check words failed");
        if (first == KIVI_OK)
            first = w;
    }
#endif
    *status = first;
    return ok();
}

}  // extern "C"

namespace kivi {

int sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 152;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace kivi

namespace kivi {

// Lets entry points defined in other translation units report through
// kivi_last_error().
int32_t record_error(int32_t status, const char* message)
{
    return fail(status, "%s", message);
}

}  // namespace kivi
