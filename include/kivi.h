/*
 * kivi.h -- C ABI of libkivi: KIVI grouped asymmetric KV-cache quantization
 * on one NVIDIA GB300 (sm_103a).
 *
 * The method (KIVI, Liu et al., ICML 2024, as the CacheForge README describes
 * it in its section "How it works", and as the CacheSeek PR #4 change notes
 * use it for exact-prefix reuse):
 * keys are quantized per channel over groups of G tokens, values per token
 * over groups of G channels, each group with its own min/max statistics; the
 * most recent tokens stay in fp16.  The pages print no formula; this library
 * fixes the arithmetic as follows, and every entry point below follows it:
 *
 *   M     = 2^b - 1, b in {2, 4, 8}            (CacheForge "Example": k_bits,
 *                                               v_bits; CacheSeek: int4/int8)
 *   scale = (max - min) / M     fp32 subtraction, IEEE fp32 division
 *   zero  = min                 (CacheSeek PR #4 change notes: the payload's
 *                                offset field)
 *   code  = clamp(rne((x - zero) / scale), 0, M)   fp32, IEEE division,
 *           round half to even; code = 0 when scale == 0
 *   x_hat = fp16_rne(fmaf(code, scale, zero))
 *
 * Inputs equal to -0 are treated as +0 when forming min/max, so the stored
 * statistics never hold -0.  NaN and infinity inputs are not supported.
 *
 * Codes are packed little-endian into int32 words, P = 32/b codes per word
 * (16 x int2, 8 x int4, 4 x int8; code i occupies bits [i*b, i*b+b)), along
 * the grouping axis: key words run along tokens, value words along channels.
 *
 * Residual (CacheForge README, "Example": the residual_length setting, the
 * count of recent tokens kept in fp16).  A sequence of T tokens keeps its first
 *     Tq = max(0, floor((T - R) / G) * G)
 * tokens quantized and the remaining T - Tq tokens (R <= T - Tq < R + G once
 * T >= R) in fp16, in a ring of R + G slots: token t lives in slot t mod (R+G).
 * Appending a token that makes the residual reach R + G quantizes its oldest
 * G tokens as one group and drops them from the ring (CacheForge README,
 * "How it works": the figure of how tokens move from fp16 into groups during
 * prefill and decoding).
 *
 * Conventions for every call:
 *   - All tensors are caller-allocated device memory (the library never
 *     allocates or frees), contiguous, row-major, 16-byte aligned.
 *   - fp16 tensors are passed as uint16_t bit patterns (IEEE binary16).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     only enqueues work on it and returns; no call synchronizes the host.
 *   - Every call returns KIVI_OK or an error code; a failed call enqueues
 *     nothing (argument errors) or reports the launch error (KIVI_ECUDA).
 *     kivi_last_error() then describes the problem (per host thread).
 *   - The per-sequence token counts `len` live on the device, so ragged
 *     batches never need a host round trip.
 */
#ifndef KIVI_H
#define KIVI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KIVI_ABI_VERSION 1

/* Status codes. */
#define KIVI_OK         0
#define KIVI_EINVAL     1 /* bad descriptor, shape, pointer or alignment       */
#define KIVI_ECAPACITY  2 /* a sequence would exceed Tmax tokens (device flag) */
#define KIVI_ECUDA      3 /* the CUDA launch reported an error                  */
#define KIVI_ETIMEOUT   4 /* a bounded device wait gave up (workspace status)  */
#define KIVI_EWORKSPACE 5 /* workspace smaller than kivi_workspace_bytes()      */
#define KIVI_ECHECK     6 /* a device bounds check failed (a library built with
                             KIVI_CHECKS defined; workspace status)           */

/*
 * Cache descriptor: a plain struct of sizes and device pointers, owned and
 * filled by the caller.  Shapes (P_k = 32/bits_k, P_v = 32/bits_v):
 *
 *   kq      int32 [B][H][Tmax/P_k][D]   key codes; word (w, d) = tokens
 *                                        w*P_k .. w*P_k+P_k-1 of channel d
 *   kscale  fp32  [B][H][Tmax/G][D]     per (token group, channel)
 *   kzero   fp32  [B][H][Tmax/G][D]
 *   vq      int32 [B][H][Tmax][D/P_v]   value codes; word (t, w) = channels
 *                                        w*P_v .. w*P_v+P_v-1 of token t
 *   vscale  fp32  [B][H][Tmax][D/G]     per (token, channel group)
 *   vzero   fp32  [B][H][Tmax][D/G]
 *   kres    fp16  [B][H][R+G][D]        residual ring of keys
 *   vres    fp16  [B][H][R+G][D]        residual ring of values
 *   len     int32 [B]                   tokens held by each sequence
 *
 * Constraints (checked, KIVI_EINVAL otherwise): B, H >= 1; D in {64, 128,
 * 256}; bits in {2, 4, 8}; G in {32, 64, 128} with D % G == 0; R >= 0 with
 * R % G == 0; 1 <= Tmax <= 2^24 with Tmax % G == 0; R <= 2^24; all pointers
 * non-NULL and 16-byte aligned.
 */
typedef struct kivi_cache {
    int32_t B, H, D;
    int32_t bits_k, bits_v;
    int32_t G, R, Tmax;
    int32_t*  kq;
    float*    kscale;
    float*    kzero;
    int32_t*  vq;
    float*    vscale;
    float*    vzero;
    uint16_t* kres;
    uint16_t* vres;
    int32_t*  len;
} kivi_cache;

/* Buffer ids for kivi_buffer_bytes(). */
#define KIVI_BUF_KQ     0
#define KIVI_BUF_KSCALE 1
#define KIVI_BUF_KZERO  2
#define KIVI_BUF_VQ     3
#define KIVI_BUF_VSCALE 4
#define KIVI_BUF_VZERO  5
#define KIVI_BUF_KRES   6
#define KIVI_BUF_VRES   7
#define KIVI_BUF_LEN    8

/* Library ABI version (KIVI_ABI_VERSION). */
int32_t kivi_abi_version(void);

/* Message for a status code; never NULL. */
const char* kivi_status_string(int32_t status);

/* Description of the last error returned on this host thread ("" if none). */
const char* kivi_last_error(void);

/* Checks the descriptor's sizes, pointers and alignment.  Host only. */
int32_t kivi_cache_validate(const kivi_cache* c);

/* Bytes the caller must allocate for one buffer of the descriptor (sizes
 * only are read; pointers may be NULL).  Returns 0 for a bad id or bad sizes. */
size_t kivi_buffer_bytes(const kivi_cache* c, int32_t buffer);

/*
 * Bytes a sequence of T tokens occupies in the cache for one (batch, head)
 * slice -- codes + fp32 scale/zero + fp16 residual (CacheSeek PR #4 change
 * notes: the store's size accounting counts a payload at its quantized
 * size):
 *   keys   (which = 0): Tq*D*b/8 + (Tq/G)*D*8 + (T-Tq)*D*2
 *   values (which = 1): Tq*D*b/8 + Tq*(D/G)*8 + (T-Tq)*D*2
 * Host only.  Returns 0 for invalid arguments.
 */
size_t kivi_cache_bytes(int32_t T, int32_t D, int32_t bits, int32_t G,
                        int32_t R, int32_t which);

/*
 * Prefix encode of keys (CacheForge "How it works": keys per channel).
 * K: fp16 [B][H][T][D].  Sequence b keeps its first n_b tokens, where
 * n_b = seq_lens[b] (device int32 [B], each 0 <= n_b <= T) or n_b = T when
 * seq_lens is NULL; T <= Tmax.  Writes kq, kscale, kzero for the Tq(n_b)
 * quantized tokens, copies tokens [Tq, n_b) into the key ring, and sets
 * len[b] = n_b.  One pass: each (channel, G-token group) tile is read once,
 * reduced to min/max, and its codes are packed in place.
 */
int32_t kivi_quant_keys(const kivi_cache* c, const uint16_t* K, int32_t T,
                        const int32_t* seq_lens, void* stream);

/*
 * Prefix encode of values (CacheForge "How it works": values per token).
 * V: fp16 [B][H][T][D]; seq_lens, T as for kivi_quant_keys.  Writes vq,
 * vscale, vzero, the value ring, and len[b] = n_b.
 */
int32_t kivi_quant_values(const kivi_cache* c, const uint16_t* V, int32_t T,
                          const int32_t* seq_lens, void* stream);

/*
 * Materialize (CacheSeek PR #4 change notes: a stored layer is dequantized
 * on the device once it has been brought back there): unpack and
 * dequantize keys (which = 0) or values (which = 1) into out, fp16
 * [B][H][T_out][D].  Rows t < len[b] are written (quantized rows as x_hat,
 * residual rows copied from the ring); rows t >= len[b] are not touched.
 * Requires len[b] <= T_out <= Tmax for every b (len is not checked on the
 * host; rows past T_out are never written).
 */
int32_t kivi_dequant(const kivi_cache* c, int32_t which, uint16_t* out,
                     int32_t T_out, void* stream);

/*
 * Append one decoded token to every sequence: k, v fp16 [B][H][D].
 * Writes them into ring slot len[b] mod (R+G) and increments len[b]; when
 * the residual reaches R + G tokens, the oldest G are quantized (keys: one
 * G-token group per channel; values: G tokens, per-token groups) and
 * appended to the packed cache.  A sequence with len[b] == Tmax is left
 * unchanged and *status (device int32, caller-owned) is set to
 * KIVI_ECAPACITY; *status is otherwise not written.  Two kernels on `stream`.
 */
int32_t kivi_append_token(const kivi_cache* c, const uint16_t* k,
                          const uint16_t* v, int32_t* status, void* stream);

/*
 * Decode logits with dequantization fused into the load.  The decode-time
 * consumer of the cache: CacheForge README, "How it works" (the cache is
 * quantized during prefill and read back at every decoding step) and
 * "Example" (generation with the quantized cache).  The pages print no
 * attention formula; this is standard scaled dot-product attention of one
 * query token over the dequantized keys:
 *   logits[b][hq][t] = sm_scale * sum_d q[b][hq][d] * K_hat[b][h][t][d]
 * for t < len[b], where h = hq / (Hq / H) (grouped-query attention) and
 * K_hat = code*scale + zero evaluated in fp32 (quantized tokens) or the fp16
 * residual.  q: fp16 [B][Hq][D]; logits: fp32 [B][Hq][ld_logits],
 * ld_logits >= Tmax, a multiple of 4; entries t >= len[b] are not written.
 * Hq must be a multiple of H with Hq / H <= 16.
 */
int32_t kivi_decode_qk(const kivi_cache* c, const uint16_t* q, int32_t Hq,
                       float sm_scale, float* logits, int32_t ld_logits,
                       void* stream);

/*
 * Decode output with dequantization fused into the load (the second half of
 * the decode-time consumer, same passages as kivi_decode_qk):
 *   p = softmax over t < len[b] of logits[b][hq][t]     (fp32, max-subtracted)
 *   out[b][hq][d] = sum_t p_t * V_hat[b][h][t][d]
 * out: fp32 [B][Hq][D].  The token range is split into chunks processed in
 * parallel; per-chunk partial results go to the caller's workspace `ws`
 * (device, >= kivi_workspace_bytes(c, Hq) bytes, 16-byte aligned) and a
 * second kernel combines them.  A sequence with len[b] == 0 gets out = 0.
 * The chunking and every sum's order are fixed, so kivi_decode_qk followed
 * by kivi_decode_pv gives the same bits from run to run (the fused
 * kivi_decode_attention is faster and agrees with it to rounding order).
 */
int32_t kivi_decode_pv(const kivi_cache* c, const float* logits,
                       int32_t ld_logits, int32_t Hq, float* out, void* ws,
                       size_t ws_bytes, void* stream);

/*
 * Decode attention in one pass over the cache: the logits of kivi_decode_qk,
 * the softmax and the weighted sum of kivi_decode_pv, fused so that the
 * logits stay on chip:
 *   out[b][hq][d] = sum_t softmax_t(sm_scale q . K_hat_t) V_hat[t][d]
 * over t < len[b] (the decode-time consumer: CacheForge README, "How it
 * works" and "Example", as for kivi_decode_qk).  Any bits_k, bits_v.
 * q: fp16 [B][Hq][D]; out: fp32 [B][Hq][D]; ws: device, >=
 * kivi_workspace_bytes(c, Hq) bytes, 16-byte aligned, contents need not be
 * initialized.  One persistent kernel (one CTA per SM, each taking a
 * contiguous share of all rows' tiles, the shares balanced by a weight that
 * counts each row's start as well as its tiles) and a combine kernel for the
 * rows that CTA shares cut: two kernels on `stream`.  A sequence with len[b] == 0 gets
 * out = 0.  The first 4 bytes of ws receive a status word: KIVI_OK, or
 * KIVI_ETIMEOUT if a bounded wait inside the kernel gave up (after two
 * seconds; the outputs are then invalid).  Calls that share a workspace must
 * not overlap on the GPU.  Which consumer warp takes which tile varies from
 * run to run, so results agree from run to run to rounding order, not bit
 * for bit; kivi_decode_qk + kivi_decode_pv is the deterministic path.
 */
int32_t kivi_decode_attention(const kivi_cache* c, const uint16_t* q,
                              int32_t Hq, float sm_scale, float* out,
                              void* ws, size_t ws_bytes, void* stream);

/*
 * Workspace bytes kivi_decode_pv and kivi_decode_attention need for this
 * descriptor and Hq: room for the per-chunk partial results of the split
 * token range.  An implementation detail of the decode-time consumer (the
 * pages have no counterpart).  Host only; 0 for invalid sizes.
 */
size_t kivi_workspace_bytes(const kivi_cache* c, int32_t Hq);

/* Size of the fixed device scratch behind kivi_decode_pv_noalloc. */
#define KIVI_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * kivi_decode_pv for callers that cannot allocate device memory.  This entry
 * point has no counterpart on the KIVI pages; it exists for callers with no
 * way to hand over a workspace -- an engine that reserves all of HBM for its
 * own KV pool and exposes no allocator, a custom op inside another runtime
 * that must not allocate outside that runtime's accounting, a decode loop
 * that must not call cudaMalloc / cudaFree because they can synchronize the
 * device.  Same arguments, results and validation as kivi_decode_pv, minus
 * ws / ws_bytes: the per-chunk partials go to a KIVI_NOALLOC_SCRATCH_BYTES
 * (16 MiB) array compiled into the library, one per GPU that loads it, held
 * until the process exits.  The call allocates nothing.
 *   - Shapes with kivi_workspace_bytes(c, Hq) > KIVI_NOALLOC_SCRATCH_BYTES are
 *     rejected with KIVI_EWORKSPACE before anything is launched.
 *   - The arguments are checked as kivi_decode_pv checks them (KIVI_EINVAL
 *     for a bad cache, Hq, logits or out) before the size test.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it for the
 *     rest of the process; make that first call before any stream capture.
 *     A device reset (cudaDeviceReset, or anything else that destroys the
 *     device's primary context) frees the array and leaves the cached address
 *     stale: do not call this entry point on a device after resetting it.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents.  Calls whose kernels may overlap on the GPU (unordered
 *     streams) race and corrupt each other's results: order them.  No part
 *     of the array needs to start at zero.
 */
int32_t kivi_decode_pv_noalloc(const kivi_cache* c, const float* logits,
                               int32_t ld_logits, int32_t Hq, float* out,
                               void* stream);

/* ------------------------------------------------ compact payload (store) */

/*
 * The exact-prefix store of CacheSeek PR #4 (change notes) keeps a quantized
 * layer as a compact payload of codes, scales and offsets that is copied to
 * host memory for storage, and folds a fingerprint of the quantization
 * settings into the prefix root hash, so that a quantized entry never matches
 * one stored under another codec.  These calls
 * move a cache's payload between the device and caller-owned memory (pinned
 * host memory: the copy kernels read and write it directly, over NVLink-C2C
 * on a Grace-Blackwell node) in this format, all little-endian:
 *
 *   header, 64 bytes:
 *     uint32 magic   KIVI_PAYLOAD_MAGIC ("KIVP")
 *     uint32 format  KIVI_PAYLOAD_VERSION
 *     uint64 kivi_codec_fingerprint(c)
 *     int32  B, H, D, bits_k, bits_v, G, R;  int32 reserved[5] = 0
 *   int32 len[B], zero-padded to a multiple of 4 entries
 *   then for b = 0..B-1, h = 0..H-1 (n = len[b], Tq = Tq(n), res = n - Tq):
 *     kq rows [0, Tq/Pk) of the slice     int32 [Tq/Pk][D]
 *     kscale, kzero rows [0, Tq/G)        fp32  [Tq/G][D] each
 *     vq rows [0, Tq)                     int32 [Tq][D/Pv]
 *     vscale, vzero rows [0, Tq)          fp32  [Tq][D/G] each
 *     key residual tokens Tq .. n-1       fp16  [res][D] (token order)
 *     value residual tokens Tq .. n-1     fp16  [res][D]
 *
 * A slice takes kivi_cache_bytes(n, ..., 0) + kivi_cache_bytes(n, ..., 1)
 * bytes, and every section starts 16-byte aligned.
 */
#define KIVI_PAYLOAD_MAGIC   0x5056494Bu /* bytes "KIVP" */
#define KIVI_PAYLOAD_VERSION 1
#define KIVI_PAYLOAD_HEADER_BYTES 64

/*
 * Codec fingerprint: FNV-1a 64 (offset basis 0xcbf29ce484222325, prime
 * 0x100000001b3) of the 32 bytes "KIVI" followed by the int32 values
 * {1 (layout version), D, bits_k, bits_v, G, R, 4 (bytes per statistic)},
 * little-endian.  Equal fingerprints mean payloads that decode identically
 * for any B, H and Tmax.  Host only; 0 for an invalid descriptor.
 */
uint64_t kivi_codec_fingerprint(const kivi_cache* c);

/*
 * Bytes of the payload of this descriptor when sequence b holds lens[b]
 * tokens (lens: host int32 [B], 0 <= lens[b] <= Tmax).  Host only; 0 for
 * invalid arguments.
 */
size_t kivi_payload_bytes(const kivi_cache* c, const int32_t* lens);

/*
 * Writes the payload of the cache (its current len[] on the device) to dst
 * (dst_bytes bytes, 16-byte aligned, device memory or pinned host memory).
 * If the payload would exceed dst_bytes, nothing is written and *status
 * (device int32) is set to KIVI_EWORKSPACE; *status is otherwise not
 * written.  One kernel on `stream`.
 */
int32_t kivi_export(const kivi_cache* c, void* dst, size_t dst_bytes,
                    int32_t* status, void* stream);

/*
 * Reads a payload from src (src_bytes bytes, 16-byte aligned, device memory
 * or pinned host memory) into the cache: codes, statistics, ring slots of the
 * residual tokens, and len[b].  The header is checked on the device before
 * anything is written: a wrong magic, format, fingerprint or B/H/D/bits/G/R
 * sets *status to KIVI_EINVAL, a sequence longer than Tmax to
 * KIVI_ECAPACITY, a payload longer than src_bytes to KIVI_EWORKSPACE; the
 * cache is then left unchanged.  One kernel on `stream`.
 */
int32_t kivi_import(const kivi_cache* c, const void* src, size_t src_bytes,
                    int32_t* status, void* stream);

/* ---------------------------------------------------- bounds-checked build */

/*
 * A library built with KIVI_CHECKS defined (the "checked" build variant)
 * checks, on the device, every global access of the encode, materialize,
 * append, payload and split-decode kernels against the arrays of the cache
 * and the buffers of the call, and skips an access that falls outside them;
 * the streamed fused decode checks its copies, tiles and output rows and
 * reports in its workspace status word (kivi_decode_attention).  This call
 * writes to *status (host memory) the status of the first failed check since
 * the previous call -- KIVI_ECHECK -- or KIVI_OK, and clears the record.  It
 * synchronizes the device.  In a library built without KIVI_CHECKS it writes
 * KIVI_OK.  Returns KIVI_OK, KIVI_EINVAL (status is NULL) or KIVI_ECUDA.
 */
int32_t kivi_check_status(int32_t* status);

#ifdef __cplusplus
}
#endif
#endif /* KIVI_H */
