// kivi_launch.h -- host-side launchers behind the C ABI (internal).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kivi.h"

namespace kivi {

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Number of decode chunks (one CTA per KV head and chunk) that cover Tmax.
int pv_chunks(const kivi_cache& c, int Hq);

cudaError_t launch_quant_keys(const kivi_cache& c, const uint16_t* K, int T,
                              const int32_t* seq_lens, cudaStream_t s);
cudaError_t launch_quant_values(const kivi_cache& c, const uint16_t* V, int T,
                                const int32_t* seq_lens, cudaStream_t s);
cudaError_t launch_dequant(const kivi_cache& c, int which, uint16_t* out, int T_out,
                           cudaStream_t s);
cudaError_t launch_append(const kivi_cache& c, const uint16_t* k, const uint16_t* v,
                          int32_t* status, cudaStream_t s);
cudaError_t launch_decode_qk(const kivi_cache& c, const uint16_t* q, int Hq, float sm_scale,
                             float* logits, int ld_logits, cudaStream_t s);
// ws_o: [B*Hq][nchunks][D], ws_m / ws_l: [B*Hq][nchunks] (fp32).
cudaError_t launch_decode_pv(const kivi_cache& c, const float* logits, int ld_logits, int Hq,
                             float* out, float* ws_o, float* ws_m, float* ws_l,
                             cudaStream_t s);

// q . K, softmax and p . V in one persistent pipelined kernel (one CTA per
// SM) plus a combine kernel for rows that CTA ranges cut; any bits_k, bits_v.
// ws: stream_ws_bytes(c, Hq) bytes.
cudaError_t launch_decode_attention(const kivi_cache& c, const uint16_t* q, int Hq, float sm_scale,
                                    float* out, float* ws, cudaStream_t s);
// Workspace bytes of launch_decode_attention (grid bounded by kMaxStreamCTAs).
size_t stream_ws_bytes(const kivi_cache& c, int Hq);

// The decode kernels of one head dimension D (64, 128, 256), without the
// combine step; instantiated in decode_d<D>.cu.
template <int D>
cudaError_t launch_decode_qk_d(const kivi_cache& c, const uint16_t* q, int Hq, float sm_scale, float* logits,
                               int ld_logits, cudaStream_t s);
template <int D>
cudaError_t launch_decode_pv_d(const kivi_cache& c, const float* logits, int ld_logits, int Hq, float* ws_o,
                               float* ws_m, float* ws_l, cudaStream_t s);
// The streamed fused decode of one head dimension D and key width BK (all
// value widths and query heads per pass), instantiated in
// decode_stream_d<D>_k<BK>.cu.
template <int D, int BK>
cudaError_t launch_decode_stream(const kivi_cache& c, const uint16_t* q, int Hq, float sm_scale, float* out,
                                 float* ws, cudaStream_t s);

// Compact payload (include/kivi.h): its size for host lengths lens[B], and
// the export / import kernels (header checks and size limits on the device).
size_t payload_bytes(const kivi_cache& c, const int32_t* lens);
cudaError_t launch_export(const kivi_cache& c, void* dst, size_t dst_bytes, uint64_t fingerprint,
                          int32_t* status, cudaStream_t s);
cudaError_t launch_import(const kivi_cache& c, const void* src, size_t src_bytes, uint64_t fingerprint,
                          int32_t* status, cudaStream_t s);

// The argument checks kivi_decode_pv makes before it looks at its workspace
// (cache, Hq, logits, out); KIVI_OK or the status it would return.
int32_t check_decode_pv_args(const kivi_cache* c, const float* logits, int32_t ld_logits, int32_t Hq,
                             const float* out);

#ifdef KIVI_CHECKS
// Read and clear the check word of each translation unit with checked kernels.
int32_t check_word_quant();
int32_t check_word_dequant();
int32_t check_word_append();
int32_t check_word_payload();
int32_t check_word_decode();
int32_t check_word_decode_d64();
int32_t check_word_decode_d128();
int32_t check_word_decode_d256();
#endif

// Sets the message kivi_last_error() returns on this host thread; returns status.
int32_t record_error(int32_t status, const char* message);

}  // namespace kivi
