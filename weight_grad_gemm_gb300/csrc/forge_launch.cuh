// forge_launch.cuh -- launch wrappers shared by the host API and the kernel
// translation units (one per input type, compiled in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "forge_kernel.cuh"

namespace forge {

// Sets the kernel's shared-memory limit on the current device (once per
// device) and launches it on `stream`.
template <int IT, int OP, int ST, bool GROUPED, bool MANUAL>
cudaError_t launch_wgrad(const CUtensorMap& tmA, const CUtensorMap& tmB, const Params& p,
                         int grid, cudaStream_t stream);

// Same for the CTA-pair kernel (grid: an even number of CTAs).
template <int IT, int OP, int ST>
cudaError_t launch_wgrad_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const Params& p,
                              int grid, cudaStream_t stream);

}  // namespace forge

#define FORGE_DEFINE_LAUNCH_PAIR()                                                             \
    namespace forge {                                                                          \
    template <int IT, int OP, int ST>                                                          \
    cudaError_t launch_wgrad_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,              \
                                  const Params& p, int grid, cudaStream_t stream)              \
    {                                                                                          \
        static unsigned long long attr_done = 0;                                               \
        int dev = 0;                                                                           \
        cudaError_t e = cudaGetDevice(&dev);                                                   \
        if (e != cudaSuccess) return e;                                                        \
        auto kern = forge_wgrad_pair_kernel<IT, OP, ST>;                                       \
        const unsigned long long bit = 1ull << (dev & 63);                                     \
        if (!(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & bit)) {                          \
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                     kSmemAlloc);                                              \
            if (e != cudaSuccess) return e;                                                    \
            __atomic_fetch_or(&attr_done, bit, __ATOMIC_ACQ_REL);                              \
        }                                                                                      \
        kern<<<grid, kThreads, kSmemAlloc, stream>>>(tmA, tmB, p);                             \
        return cudaGetLastError();                                                             \
    }                                                                                          \
    }

#define FORGE_INSTANTIATE_PAIR(IT, OP, ST)                                                     \
    template cudaError_t forge::launch_wgrad_pair<IT, OP, ST>(                                 \
        const CUtensorMap&, const CUtensorMap&, const forge::Params&, int, cudaStream_t);

#define FORGE_DEFINE_LAUNCH()                                                                  \
    namespace forge {                                                                          \
    template <int IT, int OP, int ST, bool GROUPED, bool MANUAL>                               \
    cudaError_t launch_wgrad(const CUtensorMap& tmA, const CUtensorMap& tmB, const Params& p,  \
                             int grid, cudaStream_t stream)                                    \
    {                                                                                          \
        static unsigned long long attr_done = 0; /* one bit per device ordinal < 64 */         \
        int dev = 0;                                                                           \
        cudaError_t e = cudaGetDevice(&dev);                                                   \
        if (e != cudaSuccess) return e;                                                        \
        auto kern = forge_wgrad_kernel<IT, OP, ST, GROUPED, MANUAL>;                                   \
        const unsigned long long bit = 1ull << (dev & 63);                                     \
        if (!(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & bit)) {                          \
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                     kSmemAlloc);                                              \
            if (e != cudaSuccess) return e;                                                    \
            __atomic_fetch_or(&attr_done, bit, __ATOMIC_ACQ_REL);                              \
        }                                                                                      \
        kern<<<grid, kThreads, kSmemAlloc, stream>>>(tmA, tmB, p);                             \
        return cudaGetLastError();                                                             \
    }                                                                                          \
    }

#define FORGE_INSTANTIATE(IT, OP, ST, G, MAN)                                                  \
    template cudaError_t forge::launch_wgrad<IT, OP, ST, G, MAN>(                              \
        const CUtensorMap&, const CUtensorMap&, const forge::Params&, int, cudaStream_t);
