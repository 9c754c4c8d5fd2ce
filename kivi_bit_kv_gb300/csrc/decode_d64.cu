// decode_d64.cu -- the decode-attention kernels for head dimension 64.
#include "decode_kernels.cuh"

namespace kivi {
KIVI_DECODE_INSTANTIATE(64)
}  // namespace kivi
