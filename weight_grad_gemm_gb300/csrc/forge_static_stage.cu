// forge_static_stage.cu -- the fixed staging buffer behind
// forge_wgrad_adamw_noalloc.
//
// The buffer is a file-scope device array, so it lives in this translation
// unit's own module: with lazy module loading (the CUDA default) its device
// memory is reserved on a device only once the first no-allocation call
// there resolves its address, and stays reserved for the life of the process;
// with CUDA_MODULE_LOADING=EAGER every context the process creates reserves
// it at creation.  The address is cached per device ordinal and belongs to
// that device's primary context: after cudaDeviceReset (or from another
// context) the cached address is stale, so such calls are not supported.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "forge_static_stage.h"

namespace {

constexpr size_t kCapacity = size_t(256) << 20;  // 256 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_stage[kCapacity];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

}  // namespace

namespace forge {

size_t static_stage_capacity() { return kCapacity; }

cudaError_t static_stage_address(int dev, void** out)
{
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void* a = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&a, g_static_stage);
        if (e != cudaSuccess) return e;
        g_addr[dev] = a;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

}  // namespace forge
