// forge_quant.cu -- per-tensor e4m3 quantisation with an amax scale, the step
// in front of an fp8 call: s = amax |x| / 448 (1 when amax is 0) and every
// code is the e4m3 value nearest to x / s (ties to even).
//
// Two HBM-bound passes, because no code can be written before amax is known,
// and no scratch memory: the first pass reduces |x| to one partial maximum
// per block and parks the partials in the codes buffer itself (an aligned
// window of it, which the codes overwrite later); one block folds them into
// amax and writes s to the caller's scale; the second pass reads s and
// converts every element with the hardware's round-to-nearest-even,
// saturating fp32 -> e4m3 conversion.  Stream order keeps the three launches
// apart, so no block overwrites a partial another block still needs.  No
// atomics.  Inputs of fewer than 8 elements take one single-block launch
// that does both passes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "forge.h"
#include "forge_device.h"

namespace {

constexpr int kThreads = 512;
constexpr int kBlocksPerSm = 4;
constexpr int kUnroll = 4;  // independent vector loads in flight per thread

// four consecutive inputs widened to float (fp32: one 16-byte load; bf16:
// one 8-byte load)
__device__ __forceinline__ void load4(const float* x, int64_t i, float (&v)[4])
{
    const float4 t = __ldcs(reinterpret_cast<const float4*>(x + i));
    v[0] = t.x;
    v[1] = t.y;
    v[2] = t.z;
    v[3] = t.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* x, int64_t i, float (&v)[4])
{
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(x + i));
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xFFFF0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xFFFF0000u);
}
__device__ __forceinline__ float load1(const float* x, int64_t i) { return x[i]; }
__device__ __forceinline__ float load1(const __nv_bfloat16* x, int64_t i)
{
    return __bfloat162float(x[i]);
}

// Maximum over the block (NaN operands are skipped by fmaxf); every thread
// receives the result.
__device__ __forceinline__ float block_max(float v, float* sh)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5;
    __syncthreads();  // sh may still be read from an earlier call
    if ((threadIdx.x & 31) == 0) sh[w] = v;
    __syncthreads();
    v = 0.0f;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) v = fmaxf(v, sh[i]);
    return v;
}

// Two fp32 values to e4m3 (round to nearest even, saturating): lo lands in
// the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads) forge_amax_kernel(const T* __restrict__ x, int64_t n,
                                                              float* __restrict__ part)
{
    __shared__ float sh[32];
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    float m = 0.0f;
    int64_t i0 = 0;
    if constexpr (VEC) {
        const int64_t n4 = n / 4;
        for (int64_t j0 = tid; j0 < n4; j0 += kUnroll * stride) {
            float v[kUnroll][4];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (j0 + u * stride < n4) load4(x, 4 * (j0 + u * stride), v[u]);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (j0 + u * stride < n4)
                    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[u][0]), fabsf(v[u][1])),
                                       fmaxf(fabsf(v[u][2]), fabsf(v[u][3]))));
        }
        i0 = 4 * n4;
    }
    for (int64_t i = i0 + tid; i < n; i += stride) m = fmaxf(m, fabsf(load1(x, i)));
    m = block_max(m, sh);
    if (threadIdx.x == 0) part[blockIdx.x] = m;
}

// s from amax, as the recipe divides it: in fp32, and 1 for an all-zero input
__device__ __forceinline__ float scale_of(float amax)
{
    return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

// One block: amax over the partials, then s into *scale.
__global__ void __launch_bounds__(kThreads) forge_amax_fold_kernel(const float* __restrict__ part,
                                                                   int nparts,
                                                                   float* __restrict__ scale)
{
    __shared__ float sh[32];
    float m = 0.0f;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) m = fmaxf(m, part[i]);
    m = block_max(m, sh);
    if (threadIdx.x == 0) *scale = scale_of(m);
}

// One block, both passes, for inputs too short to hold the partials.
template <typename T>
__global__ void __launch_bounds__(kThreads) forge_quant_small_kernel(const T* __restrict__ x,
                                                                     int64_t n,
                                                                     uint8_t* __restrict__ q,
                                                                     float* __restrict__ scale)
{
    __shared__ float sh[32];
    float m = 0.0f;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, fabsf(load1(x, i)));
    const float s = scale_of(block_max(m, sh));
    if (threadIdx.x == 0) *scale = s;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x)
        q[i] = static_cast<uint8_t>(e4m3x2(__fdiv_rn(load1(x, i), s), 0.0f) & 0xFFu);
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads) forge_quant_kernel(const T* __restrict__ x, int64_t n,
                                                               uint8_t* __restrict__ q,
                                                               const float* __restrict__ scale)
{
    const float s = *scale;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i0 = 0;
    if constexpr (VEC) {
        const int64_t n4 = n / 4;
        for (int64_t j0 = tid; j0 < n4; j0 += kUnroll * stride) {
            float v[kUnroll][4];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (j0 + u * stride < n4) load4(x, 4 * (j0 + u * stride), v[u]);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t j = j0 + u * stride;
                if (j >= n4) continue;
                const uint32_t c = e4m3x2(__fdiv_rn(v[u][0], s), __fdiv_rn(v[u][1], s)) |
                                   (e4m3x2(__fdiv_rn(v[u][2], s), __fdiv_rn(v[u][3], s)) << 16);
                __stcs(reinterpret_cast<unsigned int*>(q + 4 * j), c);
            }
        }
        i0 = 4 * n4;
    }
    for (int64_t i = i0 + tid; i < n; i += stride)
        q[i] = static_cast<uint8_t>(e4m3x2(__fdiv_rn(load1(x, i), s), 0.0f) & 0xFFu);
}

bool aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

template <typename T>
cudaError_t quantize(const T* x, int64_t n, uint8_t* q, float* scale, int sms,
                     cudaStream_t stream)
{
    // partials window: the first 4-byte aligned byte of q onwards
    const int64_t pad = static_cast<int64_t>((4 - reinterpret_cast<uintptr_t>(q) % 4) % 4);
    if (n < pad + 4 * 2) {
        forge_quant_small_kernel<T><<<1, kThreads, 0, stream>>>(x, n, q, scale);
        return cudaGetLastError();
    }
    const bool vec = aligned(x, 4 * sizeof(T)) && aligned(q, 4);
    const int64_t units = vec ? n / 4 + (n % 4) : n;
    int64_t want = (units + static_cast<int64_t>(kThreads) * kUnroll - 1) /
                   (static_cast<int64_t>(kThreads) * kUnroll);
    const int64_t cap = std::min<int64_t>(static_cast<int64_t>(kBlocksPerSm) * sms, (n - pad) / 4);
    const int blocks = static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
    float* part = reinterpret_cast<float*>(q + pad);
    if (vec)
        forge_amax_kernel<T, true><<<blocks, kThreads, 0, stream>>>(x, n, part);
    else
        forge_amax_kernel<T, false><<<blocks, kThreads, 0, stream>>>(x, n, part);
    forge_amax_fold_kernel<<<1, kThreads, 0, stream>>>(part, blocks, scale);
    if (vec)
        forge_quant_kernel<T, true><<<blocks, kThreads, 0, stream>>>(x, n, q, scale);
    else
        forge_quant_kernel<T, false><<<blocks, kThreads, 0, stream>>>(x, n, q, scale);
    return cudaGetLastError();
}

}  // namespace

extern "C" forge_status forge_quantize_e4m3(const void* x, forge_dtype x_dtype, int64_t n,
                                            uint8_t* codes, float* scale, forge_stream_t stream)
{
    if (n < 0 || !scale || (n > 0 && (!x || !codes))) return FORGE_ERR_INVALID_ARG;
    if (x_dtype != FORGE_F32 && x_dtype != FORGE_BF16) return FORGE_ERR_UNSUPPORTED_DTYPE;
    if (!aligned(scale, 4) || (x && !aligned(x, x_dtype == FORGE_F32 ? 4 : 2)))
        return FORGE_ERR_MISALIGNED;
    int sms = 0;
    forge_status st = forge::device_sms(&sms);
    if (st != FORGE_OK) return st;
    const void* ptrs[] = {n > 0 ? x : nullptr, n > 0 ? codes : nullptr, scale};
    if ((st = forge::device_resident(ptrs, 3)) != FORGE_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e =
        x_dtype == FORGE_F32
            ? quantize(static_cast<const float*>(x), n, codes, scale, sms, s)
            : quantize(static_cast<const __nv_bfloat16*>(x), n, codes, scale, sms, s);
    return e == cudaSuccess ? FORGE_OK : FORGE_ERR_CUDA;
}
