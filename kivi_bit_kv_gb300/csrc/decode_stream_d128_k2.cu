// decode_stream_d128_k2.cu -- the streamed fused decode attention for head
// dimension 128 and 2-bit keys (every value width, 1, 2 or 4 query heads per pass).
#include "decode_stream.cuh"

namespace kivi {
KIVI_STREAM_INSTANTIATE(128, 2)
}  // namespace kivi
