/*
 * kivi_ref.c -- CPU oracle for KIVI grouped asymmetric KV-cache quantization.
 *
 * TEST INFRASTRUCTURE ONLY (see kivi_ref.h for the sources and the contract).
 * Every function walks its elements one at a time in the order the method
 * states them: group statistics, then codes, then packing; unpack, then
 * dequantization; append, then flush; logits, softmax, weighted sum.  No
 * blocking, no fusion.  Build with -ffp-contract=off so that no
 * multiply-add is fused behind the code's back.
 */
#include "kivi_ref.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* binary16 <-> binary32                                                     */
/* ------------------------------------------------------------------------ */

float kref_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    float v;
    if (expo == 0)
        v = ldexpf((float)mant, -24); /* zero or subnormal: mant * 2^-24 */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexpf((float)(mant | 0x400), expo - 25); /* 1.mant * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a non-negative double holding an exact value to an integer, ties to
 * even.  Used only on values that are exact in double. */
static double round_half_even(double n)
{
    double r = floor(n);
    double diff = n - r;
    if (diff > 0.5 || (diff == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    return r;
}

uint16_t kref_float_to_half(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(f))
        return (uint16_t)(sign | 0x7e00u);
    double a = fabs((double)f); /* exact */
    if (a >= 65520.0)           /* at or past the midpoint above 65504 */
        return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: a multiple of 2^-24 */
        double n = round_half_even(a * ldexp(1.0, 24));
        return (uint16_t)(sign | (uint16_t)n); /* n == 1024 encodes 2^-14 */
    }
    int ex;
    (void)frexp(a, &ex);          /* a = fr * 2^ex, fr in [0.5, 1) */
    int e = ex - 1;               /* a in [2^e, 2^(e+1)) */
    double n = round_half_even(a * ldexp(1.0, 10 - e)); /* in [1024, 2048] */
    if (n == 2048.0) {
        n = 1024.0;
        e += 1;
    }
    if (e + 15 >= 31)
        return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(n - 1024.0));
}

/* fp16 bits -> fp32 with -0 mapped to +0, so that equal values share bits. */
static float canon(uint16_t h)
{
    return kref_half_to_float(h) + 0.0f;
}

/* ------------------------------------------------------------------------ */
/* Split, statistics, codes, packing                                         */
/* ------------------------------------------------------------------------ */

int kref_quantized_tokens(int T, int G, int R)
{
    int n = T - R;
    if (n <= 0)
        return 0;
    return (n / G) * G;
}

void kref_group_quantize(const uint16_t* x, int n, long stride, int bits,
                         float* scale, float* zero, int32_t* codes)
{
    int M = (1 << bits) - 1;
    /* min / max: a sequential scan in index order */
    float mn = canon(x[0]);
    float mx = mn;
    for (int i = 1; i < n; ++i) {
        float v = canon(x[i * stride]);
        if (v < mn)
            mn = v;
        if (v > mx)
            mx = v;
    }
    volatile float range = mx - mn;           /* fp32 subtraction */
    float s = range / (float)M;               /* IEEE fp32 division */
    *scale = s;
    *zero = mn;
    for (int i = 0; i < n; ++i) {
        float v = canon(x[i * stride]);
        int c;
        if (s == 0.0f) {
            c = 0; /* constant group: every element equals the zero point */
        } else {
            volatile float a = v - mn;           /* fp32 subtraction */
            volatile float qf = a / s;           /* IEEE fp32 division */
            c = (int)nearbyintf(qf);             /* ties to even */
            if (c < 0)
                c = 0;
            if (c > M)
                c = M;
        }
        codes[i] = c;
    }
}

int32_t kref_pack_word(const int32_t* codes, int bits)
{
    int P = 32 / bits;
    uint32_t w = 0;
    for (int i = 0; i < P; ++i)
        w |= ((uint32_t)codes[i]) << (i * bits); /* code i at bits [i*b, i*b+b) */
    int32_t out;
    memcpy(&out, &w, sizeof out);
    return out;
}

void kref_unpack_word(int32_t word, int bits, int32_t* codes)
{
    int P = 32 / bits;
    uint32_t w;
    memcpy(&w, &word, sizeof w);
    uint32_t mask = (1u << bits) - 1u;
    for (int i = 0; i < P; ++i)
        codes[i] = (int32_t)((w >> (i * bits)) & mask);
}

static uint16_t dequant_half(int32_t code, float scale, float zero)
{
    return kref_float_to_half(fmaf((float)code, scale, zero));
}

/* ------------------------------------------------------------------------ */
/* Prefix encode                                                             */
/* ------------------------------------------------------------------------ */

void kref_encode_keys(const uint16_t* K, int T, int D, int bits, int G, int R,
                      int32_t* kq, float* ks, float* kz, uint16_t* kres)
{
    int P = 32 / bits;
    int RG = R + G;
    int Tq = kref_quantized_tokens(T, G, R);
    int32_t* codes = (int32_t*)malloc(sizeof(int32_t) * (size_t)G);
    for (int g = 0; g < Tq / G; ++g) {
        for (int d = 0; d < D; ++d) {
            /* per channel d: the G tokens g*G .. g*G+G-1 */
            const uint16_t* col = K + (size_t)g * G * D + d;
            kref_group_quantize(col, G, D, bits, &ks[(size_t)g * D + d],
                                &kz[(size_t)g * D + d], codes);
            for (int w = 0; w < G / P; ++w) {
                size_t row = (size_t)g * (G / P) + w;
                kq[row * D + d] = kref_pack_word(codes + w * P, bits);
            }
        }
    }
    free(codes);
    for (int t = Tq; t < T; ++t)
        for (int d = 0; d < D; ++d)
            kres[(size_t)(t % RG) * D + d] = K[(size_t)t * D + d];
}

void kref_encode_values(const uint16_t* V, int T, int D, int bits, int G, int R,
                        int32_t* vq, float* vs, float* vz, uint16_t* vres)
{
    int P = 32 / bits;
    int RG = R + G;
    int Tq = kref_quantized_tokens(T, G, R);
    int NG = D / G;
    int32_t* codes = (int32_t*)malloc(sizeof(int32_t) * (size_t)G);
    for (int t = 0; t < Tq; ++t) {
        for (int g = 0; g < NG; ++g) {
            /* per token t: the G channels g*G .. g*G+G-1 */
            const uint16_t* row = V + (size_t)t * D + (size_t)g * G;
            kref_group_quantize(row, G, 1, bits, &vs[(size_t)t * NG + g],
                                &vz[(size_t)t * NG + g], codes);
            for (int w = 0; w < G / P; ++w)
                vq[(size_t)t * (D / P) + (size_t)g * (G / P) + w] =
                    kref_pack_word(codes + w * P, bits);
        }
    }
    free(codes);
    for (int t = Tq; t < T; ++t)
        for (int d = 0; d < D; ++d)
            vres[(size_t)(t % RG) * D + d] = V[(size_t)t * D + d];
}

/* ------------------------------------------------------------------------ */
/* Unpack + dequantize                                                       */
/* ------------------------------------------------------------------------ */

static int32_t key_code(const int32_t* kq, int t, int d, int D, int bits)
{
    int P = 32 / bits;
    int32_t codes[16];
    kref_unpack_word(kq[(size_t)(t / P) * D + d], bits, codes);
    return codes[t % P];
}

static int32_t value_code(const int32_t* vq, int t, int d, int D, int bits)
{
    int P = 32 / bits;
    int32_t codes[16];
    kref_unpack_word(vq[(size_t)t * (D / P) + d / P], bits, codes);
    return codes[d % P];
}

void kref_decode_keys(const int32_t* kq, const float* ks, const float* kz,
                      const uint16_t* kres, int len, int D, int bits, int G,
                      int R, uint16_t* out)
{
    int RG = R + G;
    int Tq = kref_quantized_tokens(len, G, R);
    for (int t = 0; t < len; ++t) {
        for (int d = 0; d < D; ++d) {
            uint16_t h;
            if (t < Tq) {
                size_t si = (size_t)(t / G) * D + d;
                h = dequant_half(key_code(kq, t, d, D, bits), ks[si], kz[si]);
            } else {
                h = kres[(size_t)(t % RG) * D + d];
            }
            out[(size_t)t * D + d] = h;
        }
    }
}

void kref_decode_values(const int32_t* vq, const float* vs, const float* vz,
                        const uint16_t* vres, int len, int D, int bits, int G,
                        int R, uint16_t* out)
{
    int RG = R + G;
    int NG = D / G;
    int Tq = kref_quantized_tokens(len, G, R);
    for (int t = 0; t < len; ++t) {
        for (int d = 0; d < D; ++d) {
            uint16_t h;
            if (t < Tq) {
                size_t si = (size_t)t * NG + d / G;
                h = dequant_half(value_code(vq, t, d, D, bits), vs[si], vz[si]);
            } else {
                h = vres[(size_t)(t % RG) * D + d];
            }
            out[(size_t)t * D + d] = h;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Append one token, flushing the oldest G residual tokens when full         */
/* ------------------------------------------------------------------------ */

int kref_append(int32_t* kq, float* ks, float* kz, uint16_t* kres,
                int32_t* vq, float* vs, float* vz, uint16_t* vres,
                int len, const uint16_t* k, const uint16_t* v,
                int D, int bits_k, int bits_v, int G, int R, int Tmax)
{
    int RG = R + G;
    if (len + 1 > Tmax)
        return -1;
    int Tq = kref_quantized_tokens(len, G, R);
    for (int d = 0; d < D; ++d) {
        kres[(size_t)(len % RG) * D + d] = k[d];
        vres[(size_t)(len % RG) * D + d] = v[d];
    }
    len += 1;
    if (len - Tq == RG) {
        /* Gather the G oldest residual tokens into a plain [G][D] block and
         * quantize it exactly as a prefix group. */
        uint16_t* kb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)G * D);
        uint16_t* vb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)G * D);
        for (int i = 0; i < G; ++i)
            for (int d = 0; d < D; ++d) {
                kb[(size_t)i * D + d] = kres[(size_t)((Tq + i) % RG) * D + d];
                vb[(size_t)i * D + d] = vres[(size_t)((Tq + i) % RG) * D + d];
            }
        int Pk = 32 / bits_k, Pv = 32 / bits_v;
        /* keys: one G-token group per channel, appended at row Tq/Pk */
        kref_encode_keys(kb, G, D, bits_k, G, 0,
                         kq + (size_t)(Tq / Pk) * D, ks + (size_t)(Tq / G) * D,
                         kz + (size_t)(Tq / G) * D, NULL);
        /* values: G tokens, appended at row Tq */
        kref_encode_values(vb, G, D, bits_v, G, 0,
                           vq + (size_t)Tq * (D / Pv), vs + (size_t)Tq * (D / G),
                           vz + (size_t)Tq * (D / G), NULL);
        free(kb);
        free(vb);
    }
    return len;
}

/* ------------------------------------------------------------------------ */
/* Decode attention                                                          */
/* ------------------------------------------------------------------------ */

/* Dequantized key / value at full precision: code * scale + zero in double. */
static double key_hat(const int32_t* kq, const float* ks, const float* kz,
                      const uint16_t* kres, int Tq, int t, int d, int D,
                      int bits, int G, int RG)
{
    if (t < Tq) {
        size_t si = (size_t)(t / G) * D + d;
        return (double)key_code(kq, t, d, D, bits) * (double)ks[si] + (double)kz[si];
    }
    return (double)kref_half_to_float(kres[(size_t)(t % RG) * D + d]);
}

static double value_hat(const int32_t* vq, const float* vs, const float* vz,
                        const uint16_t* vres, int Tq, int t, int d, int D,
                        int bits, int G, int RG)
{
    if (t < Tq) {
        size_t si = (size_t)t * (D / G) + d / G;
        return (double)value_code(vq, t, d, D, bits) * (double)vs[si] + (double)vz[si];
    }
    return (double)kref_half_to_float(vres[(size_t)(t % RG) * D + d]);
}

void kref_attention(const uint16_t* q, int NQ, float sm_scale, int len, int D,
                    int bits_k, int bits_v, int G, int R,
                    const int32_t* kq, const float* ks, const float* kz,
                    const uint16_t* kres,
                    const int32_t* vq, const float* vs, const float* vz,
                    const uint16_t* vres, float* logits, float* out)
{
    int RG = R + G;
    int Tq = kref_quantized_tokens(len, G, R);
    double* s = (double*)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
    for (int h = 0; h < NQ; ++h) {
        const uint16_t* qh = q + (size_t)h * D;
        /* s_t = sm_scale * sum_d q_d * K_hat[t][d] */
        for (int t = 0; t < len; ++t) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += (double)kref_half_to_float(qh[d]) *
                       key_hat(kq, ks, kz, kres, Tq, t, d, D, bits_k, G, RG);
            s[t] = (double)sm_scale * acc;
            logits[(size_t)h * len + t] = (float)s[t];
        }
        /* softmax with the maximum subtracted */
        double m = -INFINITY;
        for (int t = 0; t < len; ++t)
            if (s[t] > m)
                m = s[t];
        double sum = 0.0;
        for (int t = 0; t < len; ++t) {
            s[t] = exp(s[t] - m);
            sum += s[t];
        }
        /* o_d = sum_t p_t * V_hat[t][d] */
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int t = 0; t < len; ++t)
                acc += (s[t] / sum) *
                       value_hat(vq, vs, vz, vres, Tq, t, d, D, bits_v, G, RG);
            out[(size_t)h * D + d] = (float)acc;
        }
    }
    free(s);
}

/* ------------------------------------------------------------------------ */
/* Storage accounting                                                        */
/* ------------------------------------------------------------------------ */

size_t kref_cache_bytes(int T, int D, int bits, int G, int R, int which)
{
    size_t Tq = (size_t)kref_quantized_tokens(T, G, R);
    size_t res = (size_t)T - Tq;
    size_t codes = Tq * (size_t)D * (size_t)bits / 8;
    size_t stats = which == 0 ? (Tq / (size_t)G) * (size_t)D * 8
                              : Tq * (size_t)(D / G) * 8;
    return codes + stats + res * (size_t)D * 2;
}

/* ------------------------------------------------------------------------ */
/* Compact payload                                                           */
/* ------------------------------------------------------------------------ */

uint64_t kref_fnv1a64(const uint8_t* p, size_t n)
{
    uint64_t h = 14695981039346656037ull;
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= 1099511628211ull;
    }
    return h;
}

static void put_u32(uint8_t* out, uint32_t v)
{
    for (int k = 0; k < 4; ++k)
        out[k] = (uint8_t)(v >> (8 * k));
}

static uint32_t get_u32(const uint8_t* in)
{
    uint32_t v = 0;
    for (int k = 0; k < 4; ++k)
        v |= (uint32_t)in[k] << (8 * k);
    return v;
}

uint64_t kref_codec_fingerprint(int D, int bits_k, int bits_v, int G, int R)
{
    uint8_t b[32] = {'K', 'I', 'V', 'I'};
    const int32_t f[7] = {1, D, bits_k, bits_v, G, R, 4};
    for (int i = 0; i < 7; ++i)
        put_u32(b + 4 + 4 * i, (uint32_t)f[i]);
    return kref_fnv1a64(b, sizeof b);
}

size_t kref_payload_header(uint8_t* out, int B, int H, int D, int bits_k, int bits_v, int G, int R,
                           const int32_t* lens)
{
    const uint64_t fp = kref_codec_fingerprint(D, bits_k, bits_v, G, R);
    const int32_t f[7] = {B, H, D, bits_k, bits_v, G, R};
    size_t o = 0;
    put_u32(out + o, 0x5056494Bu); o += 4;  /* "KIVP" */
    put_u32(out + o, 1u); o += 4;
    put_u32(out + o, (uint32_t)fp); o += 4;
    put_u32(out + o, (uint32_t)(fp >> 32)); o += 4;
    for (int i = 0; i < 7; ++i) {
        put_u32(out + o, (uint32_t)f[i]);
        o += 4;
    }
    for (int i = 0; i < 5; ++i) {
        put_u32(out + o, 0u);
        o += 4;
    }
    const int nl = (B + 3) / 4 * 4;
    for (int b = 0; b < nl; ++b) {
        put_u32(out + o, b < B ? (uint32_t)lens[b] : 0u);
        o += 4;
    }
    return o;
}

/* Copies n 32-bit elements (put: array -> bytes; get: bytes -> array). */
static size_t words_io(uint8_t* bytes, void* words, size_t n, int put)
{
    uint8_t* w = (uint8_t*)words;
    for (size_t i = 0; i < n; ++i) {
        uint32_t v;
        if (put) {
            memcpy(&v, w + 4 * i, 4);
            put_u32(bytes + 4 * i, v);
        } else {
            v = get_u32(bytes + 4 * i);
            memcpy(w + 4 * i, &v, 4);
        }
    }
    return 4 * n;
}

/* Residual tokens Tq .. n-1 of a ring (slot t mod RG), D halves each. */
static size_t ring_io(uint8_t* bytes, uint16_t* ring, int Tq, int n, int D, int RG, int put)
{
    size_t o = 0;
    for (int t = Tq; t < n; ++t) {
        uint16_t* row = ring + (size_t)(t % RG) * D;
        for (int d = 0; d < D; ++d, o += 2) {
            if (put) {
                bytes[o] = (uint8_t)(row[d] & 0xFFu);
                bytes[o + 1] = (uint8_t)(row[d] >> 8);
            } else {
                row[d] = (uint16_t)(bytes[o] | (bytes[o + 1] << 8));
            }
        }
    }
    return o;
}

static size_t slice_io(uint8_t* io, int n, int D, int bits_k, int bits_v, int G, int R,
                       int32_t* kq, float* ks, float* kz, uint16_t* kres,
                       int32_t* vq, float* vs, float* vz, uint16_t* vres, int put)
{
    const int Tq = kref_quantized_tokens(n, G, R), RG = R + G;
    const size_t Pk = (size_t)(32 / bits_k), Pv = (size_t)(32 / bits_v);
    size_t o = 0;
    o += words_io(io + o, kq, (size_t)Tq / Pk * D, put);
    o += words_io(io + o, ks, (size_t)(Tq / G) * D, put);
    o += words_io(io + o, kz, (size_t)(Tq / G) * D, put);
    o += words_io(io + o, vq, (size_t)Tq * (D / Pv), put);
    o += words_io(io + o, vs, (size_t)Tq * (D / G), put);
    o += words_io(io + o, vz, (size_t)Tq * (D / G), put);
    o += ring_io(io + o, kres, Tq, n, D, RG, put);
    o += ring_io(io + o, vres, Tq, n, D, RG, put);
    return o;
}

size_t kref_payload_put_slice(uint8_t* out, int n, int D, int bits_k, int bits_v, int G, int R,
                              const int32_t* kq, const float* ks, const float* kz, const uint16_t* kres,
                              const int32_t* vq, const float* vs, const float* vz, const uint16_t* vres)
{
    return slice_io(out, n, D, bits_k, bits_v, G, R, (int32_t*)kq, (float*)ks, (float*)kz,
                    (uint16_t*)kres, (int32_t*)vq, (float*)vs, (float*)vz, (uint16_t*)vres, 1);
}

size_t kref_payload_get_slice(const uint8_t* in, int n, int D, int bits_k, int bits_v, int G, int R,
                              int32_t* kq, float* ks, float* kz, uint16_t* kres,
                              int32_t* vq, float* vs, float* vz, uint16_t* vres)
{
    return slice_io((uint8_t*)in, n, D, bits_k, bits_v, G, R, kq, ks, kz, kres, vq, vs, vz, vres, 0);
}
