// decode_stream_d64_k8.cu -- the streamed fused decode attention for head
// dimension 64 and 8-bit keys (every value width, 1, 2 or 4 query heads per pass).
#include "decode_stream.cuh"

namespace kivi {
KIVI_STREAM_INSTANTIATE(64, 8)
}  // namespace kivi
