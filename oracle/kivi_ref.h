/*
 * kivi_ref.h -- CPU oracle for KIVI grouped asymmetric KV-cache quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  This header and kivi_ref.c form a plain, slow,
 * one-element-at-a-time restatement of the method, used to check the CUDA
 * library.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline may build, load or call it.  It shares no code, header, table or
 * constant with the CUDA library, and the library never calls it.
 *
 * Sources (the pages print no code and no formula for the codec):
 *  - CacheForge README, "How it works": keys are quantized per channel and
 *    values per token; recent tokens stay at higher precision.
 *  - CacheForge README, "Example": k_bits, v_bits, group_size and
 *    residual_length (how many recent tokens stay in fp16).
 *  - CacheSeek PR #4, change notes: KIVI int4/int8 encode/decode with grouped
 *    statistics, codes packed into int32 words, a payload of codes, scales
 *    and offsets.
 *  - KIVI (Liu et al., ICML 2024), cited by the CacheForge README: asymmetric
 *    min/max quantization.
 * The arithmetic the pages leave open is fixed as follows (the same contract
 * the CUDA library documents in include/kivi.h):
 *    scale = (max - min) / (2^b - 1)   fp32 subtraction, IEEE fp32 division
 *    zero  = min
 *    code  = clamp(round_half_even((x - zero) / scale), 0, 2^b - 1)
 *            (0 when scale == 0)
 *    x_hat = fp16_rne(fmaf(code, scale, zero))
 *    codes packed little-endian, 32/b per int32 word, along the grouping axis.
 *
 * Layouts of one (batch, head) slice, all row-major:
 *    K, V input          fp16 bits [T][D]
 *    kq  (key codes)     int32 [Tq/P][D]   word (w, d) = tokens wP..wP+P-1 of channel d
 *    ks, kz              fp32  [Tq/G][D]
 *    vq  (value codes)   int32 [Tq][D/P]   word (t, w) = channels wP..wP+P-1 of token t
 *    vs, vz              fp32  [Tq][D/G]
 *    kres, vres (ring)   fp16 bits [R+G][D], token t in slot t mod (R+G)
 * with P = 32/b, Tq = max(0, floor((T-R)/G)*G) quantized tokens.
 */
#ifndef KIVI_REF_H
#define KIVI_REF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* IEEE binary16 <-> binary32, written out by hand (round half to even). */
float    kref_half_to_float(uint16_t h);
uint16_t kref_float_to_half(float f);

/* Number of quantized tokens of a T-token sequence. */
int kref_quantized_tokens(int T, int G, int R);

/* One group of n fp16 values read at x[i*stride]: statistics and codes. */
void kref_group_quantize(const uint16_t* x, int n, long stride, int bits,
                         float* scale, float* zero, int32_t* codes);

/* One int32 word from 32/bits codes, and back. */
int32_t kref_pack_word(const int32_t* codes, int bits);
void    kref_unpack_word(int32_t word, int bits, int32_t* codes);

/* Prefix encode of one slice of T tokens. */
void kref_encode_keys(const uint16_t* K, int T, int D, int bits, int G, int R,
                      int32_t* kq, float* ks, float* kz, uint16_t* kres);
void kref_encode_values(const uint16_t* V, int T, int D, int bits, int G, int R,
                        int32_t* vq, float* vs, float* vz, uint16_t* vres);

/* Materialize tokens [0, len) of one slice back to fp16. */
void kref_decode_keys(const int32_t* kq, const float* ks, const float* kz,
                      const uint16_t* kres, int len, int D, int bits, int G,
                      int R, uint16_t* out);
void kref_decode_values(const int32_t* vq, const float* vs, const float* vz,
                        const uint16_t* vres, int len, int D, int bits, int G,
                        int R, uint16_t* out);

/* Append one token to a slice holding len tokens; returns the new length,
 * or -1 (nothing written) when len + 1 > Tmax. */
int kref_append(int32_t* kq, float* ks, float* kz, uint16_t* kres,
                int32_t* vq, float* vs, float* vz, uint16_t* vres,
                int len, const uint16_t* k, const uint16_t* v,
                int D, int bits_k, int bits_v, int G, int R, int Tmax);

/* Decode attention of NQ query heads against one KV slice of len tokens.
 * Logits and softmax weights in double; results stored as fp32.
 * logits [NQ][len], out [NQ][D]. */
void kref_attention(const uint16_t* q, int NQ, float sm_scale, int len, int D,
                    int bits_k, int bits_v, int G, int R,
                    const int32_t* kq, const float* ks, const float* kz,
                    const uint16_t* kres,
                    const int32_t* vq, const float* vs, const float* vz,
                    const uint16_t* vres, float* logits, float* out);

/* Bytes one slice of T tokens occupies: codes + fp32 stats + fp16 residual.
 * which = 0 keys, 1 values. */
size_t kref_cache_bytes(int T, int D, int bits, int G, int R, int which);

/* Compact payload (the store format of the CUDA library's kivi_export /
 * kivi_import; CacheSeek PR #4 change notes: codes, scales and offsets are
 * copied to host memory for storage, and a fingerprint of the quantization
 * settings enters the prefix root hash).  Written
 * byte by byte, little-endian, independent of the host's byte order. */

/* FNV-1a, 64-bit: h = 14695981039346656037; for each byte: h ^= byte,
 * h *= 1099511628211 (mod 2^64). */
uint64_t kref_fnv1a64(const uint8_t* p, size_t n);

/* FNV-1a 64 of "KIVI" followed by the int32 values {1, D, bits_k, bits_v, G,
 * R, 4}, little-endian (32 bytes). */
uint64_t kref_codec_fingerprint(int D, int bits_k, int bits_v, int G, int R);

/* Header (64 bytes: magic "KIVP", format 1, fingerprint, B, H, D, bits_k,
 * bits_v, G, R, five zero words) and the len table (B int32, zero-padded to a
 * multiple of 4 entries).  Returns the bytes written. */
size_t kref_payload_header(uint8_t* out, int B, int H, int D, int bits_k, int bits_v, int G, int R,
                           const int32_t* lens);

/* One (b, h) slice of a sequence of n tokens: kq rows [0, Tq/Pk), ks and kz
 * rows [0, Tq/G), vq rows [0, Tq), vs and vz rows [0, Tq), then key and
 * value residual tokens Tq .. n-1 from their ring slots.  Returns the bytes
 * written (kref_cache_bytes(n, .., 0) + kref_cache_bytes(n, .., 1)). */
size_t kref_payload_put_slice(uint8_t* out, int n, int D, int bits_k, int bits_v, int G, int R,
                              const int32_t* kq, const float* ks, const float* kz, const uint16_t* kres,
                              const int32_t* vq, const float* vs, const float* vz, const uint16_t* vres);

/* The inverse of kref_payload_put_slice: fills the slice's arrays (the same
 * rows and ring slots) from `in`; returns the bytes read. */
size_t kref_payload_get_slice(const uint8_t* in, int n, int D, int bits_k, int bits_v, int G, int R,
                              int32_t* kq, float* ks, float* kz, uint16_t* kres,
                              int32_t* vq, float* vs, float* vz, uint16_t* vres);

#ifdef __cplusplus
}
#endif
#endif
