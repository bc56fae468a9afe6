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
cudaError_t launch_wgrad(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmA1,
                         const CUtensorMap& tmB1, const CUtensorMap& tmAk,
                         const CUtensorMap& tmBk, const Params& p, int grid, cudaStream_t stream);

// Same for the CTA-pair kernels.  The grid is sized from the number of
// clusters of two CTAs that can be resident at once (a cluster must fit in
// one GPC), never more than `total_tiles` clusters.
template <int IT, int OP, int ST, bool GROUPED, bool MULTI>
cudaError_t launch_wgrad_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,
                              const CUtensorMap& tmA1, const CUtensorMap& tmB1,
                              const CUtensorMap& tmAk, const CUtensorMap& tmBk,
                              const MultiMaps& mm, const Params& p, int64_t total_tiles,
                              cudaStream_t stream);

}  // namespace forge

#define FORGE_DEFINE_LAUNCH_PAIR()                                                             \
    namespace forge {                                                                          \
    template <int IT, int OP, int ST, bool GROUPED, bool MULTI>                                \
    cudaError_t launch_wgrad_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,              \
                                  const CUtensorMap& tmA1, const CUtensorMap& tmB1,            \
                                  const CUtensorMap& tmAk, const CUtensorMap& tmBk,            \
                                  const MultiMaps& mm, const Params& p, int64_t total_tiles,   \
                                  cudaStream_t stream)                                         \
    {                                                                                          \
        static int max_clusters[64] = {0};                                                     \
        int dev = 0;                                                                           \
        cudaError_t e = cudaGetDevice(&dev);                                                   \
        if (e != cudaSuccess) return e;                                                        \
        auto kern = forge_wgrad_pair_kernel<IT, OP, ST, GROUPED, MULTI>;                       \
        int& mc = max_clusters[dev & 63];                                                      \
        constexpr int kSmemMax = PairRing<GROUPED>::Smem::alloc(kMaxExperts) < kSmemPerCtaMax   \
                                     ? PairRing<GROUPED>::Smem::alloc(kMaxExperts)             \
                                     : kSmemPerCtaMax;                                         \
        if (__atomic_load_n(&mc, __ATOMIC_ACQUIRE) == 0) {                                     \
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                     kSmemMax);                                                \
            if (e != cudaSuccess) return e;                                                    \
            cudaLaunchConfig_t cfg = {};                                                       \
            cfg.gridDim = dim3(2, 1, 1);                                                       \
            cfg.blockDim = dim3(EpiFor<GROUPED>::threads, 1, 1);                               \
            cfg.dynamicSmemBytes = kSmemMax;                                                   \
            int n = 0;                                                                         \
            e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);                                \
            if (e != cudaSuccess) return e;                                                    \
            if (n < 1) return cudaErrorInvalidConfiguration;                                   \
            __atomic_store_n(&mc, n, __ATOMIC_RELEASE);                                        \
        }                                                                                      \
        const int64_t nc = total_tiles < mc ? total_tiles : mc;                                \
        if (PairRing<GROUPED>::Smem::alloc(p.E) > kSmemMax) return cudaErrorInvalidValue;     \
        kern<<<static_cast<int>(2 * nc), EpiFor<GROUPED>::threads,                             \
               PairRing<GROUPED>::Smem::alloc(p.E),                                            \
               stream>>>(                                                                      \
            tmA, tmB, tmA1, tmB1, tmAk, tmBk, mm, p);                                          \
        return cudaGetLastError();                                                             \
    }                                                                                          \
    }

#define FORGE_INSTANTIATE_PAIR(IT, OP, ST, G, MU)                                              \
    template cudaError_t forge::launch_wgrad_pair<IT, OP, ST, G, MU>(                          \
        const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,        \
        const CUtensorMap&, const CUtensorMap&, const forge::MultiMaps&,                       \
        const forge::Params&, int64_t, cudaStream_t);

#define FORGE_DEFINE_LAUNCH()                                                                  \
    namespace forge {                                                                          \
    template <int IT, int OP, int ST, bool GROUPED, bool MANUAL>                               \
    cudaError_t launch_wgrad(const CUtensorMap& tmA, const CUtensorMap& tmB,                   \
                             const CUtensorMap& tmA1, const CUtensorMap& tmB1,                 \
                             const CUtensorMap& tmAk, const CUtensorMap& tmBk,                 \
                             const Params& p, int grid, cudaStream_t stream)                   \
    {                                                                                          \
        static unsigned long long attr_done = 0; /* one bit per device ordinal < 64 */         \
        int dev = 0;                                                                           \
        cudaError_t e = cudaGetDevice(&dev);                                                   \
        if (e != cudaSuccess) return e;                                                        \
        auto kern = forge_wgrad_kernel<IT, OP, ST, GROUPED, MANUAL>;                           \
        const unsigned long long bit = 1ull << (dev & 63);                                     \
        if (!(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & bit)) {                          \
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                     SmemCta::alloc(kMaxExperts));                             \
            if (e != cudaSuccess) return e;                                                    \
            __atomic_fetch_or(&attr_done, bit, __ATOMIC_ACQ_REL);                              \
        }                                                                                      \
        kern<<<grid, EpiFor<GROUPED>::threads, SmemCta::alloc(p.E), stream>>>(                 \
            tmA, tmB, tmA1, tmB1, tmAk, tmBk, p);                                              \
        return cudaGetLastError();                                                             \
    }                                                                                          \
    }

#define FORGE_INSTANTIATE(IT, OP, ST, G, MAN)                                                  \
    template cudaError_t forge::launch_wgrad<IT, OP, ST, G, MAN>(                              \
        const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,        \
        const CUtensorMap&, const CUtensorMap&, const forge::Params&, int, cudaStream_t);
