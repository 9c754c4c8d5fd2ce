// decode_noalloc.cu -- kivi_decode_pv_noalloc: the decode p.V step for
// callers that cannot allocate device memory.
//
// kivi_decode_pv needs a caller-provided workspace for its per-chunk partial
// results.  Some callers have no way to provide one: an inference engine that
// reserves all of HBM up front for its own KV pool and gives a plugin no
// handle to its allocator; a custom op hosted by another runtime that must not
// allocate outside that runtime's memory accounting; a latency-critical decode
// loop that must not call cudaMalloc / cudaFree, which can synchronize the
// device.  For them, the workspace lives here, in a fixed array compiled into
// the library.  This entry point has no counterpart on the KIVI pages.
//
// The array is KIVI_NOALLOC_SCRATCH_BYTES (16 MiB) per device and is held by
// every GPU that loads the library until the process exits.  All calls on a
// device share it, so calls whose kernels may overlap on the GPU (for
// instance on unordered streams) race; order them on one stream or with
// events.  Nothing in it has to start at zero: kivi_decode_pv writes every
// partial result before its combine step reads it, so contents left by an
// earlier call are never read.
#include <cuda_runtime.h>

#include <mutex>

#include "kivi.h"
#include "kivi_launch.h"

namespace {

__device__ __align__(256) unsigned char g_decode_scratch[KIVI_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached for the life of the
// process.  A device reset (cudaDeviceReset, or anything else that destroys
// the device's primary context) frees the array and leaves the cached address
// dangling: this entry point must not be used on a device after such a reset.
int32_t scratch_address(void** addr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return kivi::record_error(KIVI_ECUDA, "kivi_decode_pv_noalloc: no usable current device");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || p == nullptr)
            return kivi::record_error(KIVI_ECUDA,
                                      "kivi_decode_pv_noalloc: cannot locate the device scratch");
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return KIVI_OK;
}

}  // namespace

extern "C" int32_t kivi_decode_pv_noalloc(const kivi_cache* c, const float* logits,
                                          int32_t ld_logits, int32_t Hq, float* out, void* stream)
{
    // the same argument checks as kivi_decode_pv first, so that a bad cache or
    // Hq is reported as such and not as a size problem
    const int32_t valid = kivi::check_decode_pv_args(c, logits, ld_logits, Hq, out);
    if (valid != KIVI_OK)
        return valid;
    const size_t need = kivi_workspace_bytes(c, Hq);
    if (need > (size_t)KIVI_NOALLOC_SCRATCH_BYTES)
        return kivi::record_error(
            KIVI_EWORKSPACE,
            "kivi_decode_pv_noalloc: this shape needs more decode workspace than the fixed "
            "16 MiB scratch (KIVI_NOALLOC_SCRATCH_BYTES); use kivi_decode_pv with a caller workspace");
    void* ws = nullptr;
    if (need > 0) {
        const int32_t st = scratch_address(&ws);
        if (st != KIVI_OK)
            return st;
    }
    // Same validation, kernels and launch as kivi_decode_pv.
    return kivi_decode_pv(c, logits, ld_logits, Hq, out, ws, KIVI_NOALLOC_SCRATCH_BYTES, stream);
}
