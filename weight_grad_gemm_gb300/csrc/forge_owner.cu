// forge_owner.cu -- the owner's optimizer step behind a reduce-scatter.
//
// With the token dimension split across ranks (data parallelism), each rank
// contracts only its own tokens, so its dW is a partial sum; a reduce-scatter
// then delivers every output tile, summed over the ranks, to the one rank
// that owns it, and that rank alone applies the optimizer step (FORGE
// assessment PR, tessera#565, "Math verified, not asserted", P3: under a
// reduce-scatter the owner of each tile is unambiguous, so the fused update
// runs once per tile).  This kernel is that owner-side step: it reads the
// summed fp32 gradient shard and updates the owner's W, m, v (or W and the
// momentum buffer) in place with exactly the arithmetic of the fused kernel's
// epilogue (step4), so feeding it the fused kernel's own dW reproduces the
// fused call bit for bit.  Unlike the fused path it reads a gradient from
// HBM: the partial gradients exist because the collective needs them.
//
// HBM-bound: every parameter is read and written once (fp32 state: 4 B of
// gradient + 12 B read and 12 B written), in 16-byte vectors, several in
// flight per thread, over a grid of whole waves.
#include <cuda_runtime.h>

#include <cstdint>

#include "forge_device.h"
#include "forge_kernel.cuh"

namespace forge {
namespace {

constexpr int kOwnerThreads = 256;
constexpr int kOwnerBlocksPerSm = 8;  // 2048 threads: a full SM
constexpr int kOwnerUnroll = 2;       // four-element vectors in flight per thread

template <int OP, int ST>
__device__ __forceinline__ void owner_load4(const float* G, const Params& p, int64_t i, float* g,
                                            float* w, float* a, float* b)
{
    StateIO<ST_F32>::ld4(G, i, g);
    StateIO<ST_F32>::ld4(p.W, i, w);
    StateIO<ST>::ld4(p.s1, i, a);
    if constexpr (OP == OP_ADAMW) StateIO<ST>::ld4(p.s2, i, b);
}

template <int OP, int ST>
__device__ __forceinline__ void owner_store4(const Params& p, int64_t i, const float* w,
                                             const float* a, const float* b)
{
    StateIO<ST_F32>::st4(p.W, i, w);
    StateIO<ST>::st4(p.s1, i, a);
    if constexpr (OP == OP_ADAMW) StateIO<ST>::st4(p.s2, i, b);
}

// One thread per element (the scalar path; also a vector path's tail).  The
// element rides in lane 0 of a four-lane step4 whose other lanes repeat it.
template <int OP, int ST>
__device__ __forceinline__ void owner_one(const float* G, const Params& p, int64_t i)
{
    float g[4], w[4], a[4], b[4];
    g[0] = G[i];
    w[0] = StateIO<ST_F32>::ld(p.W, i);
    a[0] = StateIO<ST>::ld(p.s1, i);
    b[0] = OP == OP_ADAMW ? StateIO<ST>::ld(p.s2, i) : 0.0f;
#pragma unroll
    for (int j = 1; j < 4; ++j) {
        g[j] = g[0];
        w[j] = w[0];
        a[j] = a[0];
        b[j] = b[0];
    }
    step4<OP>(p, g, w, a, b);
    StateIO<ST_F32>::st(p.W, i, w[0]);
    StateIO<ST>::st(p.s1, i, a[0]);
    if constexpr (OP == OP_ADAMW) StateIO<ST>::st(p.s2, i, b[0]);
}

template <int OP, int ST, bool VEC>
__global__ void __launch_bounds__(kOwnerThreads) forge_owner_kernel(const float* __restrict__ G,
                                                                    const Params p, int64_t n)
{
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i0 = 0;
    if constexpr (VEC) {
        const int64_t n4 = n / 4;
        for (int64_t j0 = tid; j0 < n4; j0 += kOwnerUnroll * stride) {
            float g[kOwnerUnroll][4], w[kOwnerUnroll][4], a[kOwnerUnroll][4], b[kOwnerUnroll][4];
#pragma unroll
            for (int u = 0; u < kOwnerUnroll; ++u)
                if (j0 + u * stride < n4)
                    owner_load4<OP, ST>(G, p, 4 * (j0 + u * stride), g[u], w[u], a[u], b[u]);
#pragma unroll
            for (int u = 0; u < kOwnerUnroll; ++u) {
                if (j0 + u * stride >= n4) continue;
                step4<OP>(p, g[u], w[u], a[u], b[u]);
                owner_store4<OP, ST>(p, 4 * (j0 + u * stride), w[u], a[u], b[u]);
            }
        }
        i0 = 4 * n4;
    }
    for (int64_t i = i0 + tid; i < n; i += stride) owner_one<OP, ST>(G, p, i);
}

template <int OP, int ST>
cudaError_t launch(const float* G, const Params& p, int64_t n, bool vec, int sms,
                   cudaStream_t stream)
{
    const int64_t per_block = static_cast<int64_t>(kOwnerThreads) * (vec ? 4 * kOwnerUnroll : 1);
    const int64_t want = (n + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(kOwnerBlocksPerSm) * sms;
    const int blocks = static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
    if (vec)
        forge_owner_kernel<OP, ST, true><<<blocks, kOwnerThreads, 0, stream>>>(G, p, n);
    else
        forge_owner_kernel<OP, ST, false><<<blocks, kOwnerThreads, 0, stream>>>(G, p, n);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_owner(int op, int st, const float* G, const Params& p, int64_t n, bool vec,
                         int sms, cudaStream_t stream)
{
    if (op == OP_ADAMW)
        return st == ST_F32 ? launch<OP_ADAMW, ST_F32>(G, p, n, vec, sms, stream)
                            : launch<OP_ADAMW, ST_BF16>(G, p, n, vec, sms, stream);
    return st == ST_F32 ? launch<OP_SGDM, ST_F32>(G, p, n, vec, sms, stream)
                        : launch<OP_SGDM, ST_BF16>(G, p, n, vec, sms, stream);
}

}  // namespace forge
