// decode_d128.cu -- the decode-attention kernels for head dimension 128.
#include "decode_kernels.cuh"

namespace kivi {
KIVI_DECODE_INSTANTIATE(128)
}  // namespace kivi
