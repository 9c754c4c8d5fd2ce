// decode_stream_d256_k2.cu -- the streamed fused decode attention for head
// dimension 256 and 2-bit keys (every value width, 1, 2 or 4 query heads per pass).
#include "decode_stream.cuh"

namespace kivi {
KIVI_STREAM_INSTANTIATE(256, 2)
}  // namespace kivi
