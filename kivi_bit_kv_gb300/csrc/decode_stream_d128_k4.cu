// decode_stream_d128_k4.cu -- the streamed fused decode attention for head
// dimension 128 and 4-bit keys (every value width, 1, 2 or 4 query heads per pass).
#include "decode_stream.cuh"

namespace kivi {
KIVI_STREAM_INSTANTIATE(128, 4)
}  // namespace kivi
