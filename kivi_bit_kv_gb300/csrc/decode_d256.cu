// decode_d256.cu -- the decode-attention kernels for head dimension 256.
#include "decode_kernels.cuh"

namespace kivi {
KIVI_DECODE_INSTANTIATE(256)
}  // namespace kivi
