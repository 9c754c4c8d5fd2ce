// decode_d64.cu -- the decode-attention kernels for head dimension 64.
#include "decode_kernels.cuh"

namespace kivi {
KIVI_DECODE_INSTANTIATE(64)
#ifdef KIVI_CHECKS
int32_t check_word_decode_d64() { return take_check_word(); }
#endif
}  // namespace kivi
