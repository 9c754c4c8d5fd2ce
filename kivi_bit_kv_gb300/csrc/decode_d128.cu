// decode_d128.cu -- the decode-attention kernels for head dimension 128.
#include "decode_kernels.cuh"

namespace kivi {
KIVI_DECODE_INSTANTIATE(128)
#ifdef KIVI_CHECKS
int32_t check_word_decode_d128() { return take_check_word(); }
#endif
}  // namespace kivi
