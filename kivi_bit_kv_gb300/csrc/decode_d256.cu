// decode_d256.cu -- the decode-attention kernels for head dimension 256.
#include "decode_kernels.cuh"

namespace kivi {
KIVI_DECODE_INSTANTIATE(256)
#ifdef KIVI_CHECKS
int32_t check_word_decode_d256() { return take_check_word(); }
#endif
}  // namespace kivi
