// forge_dgrad.cu -- the input gradient dX = dY W^T, and the backward step that
// orders it before the in-place weight update.
//
// "Math verified, not asserted", P1: the fused update overwrites W in place,
// so dX must have read W first (FORGE's in-place dX-before-update hazard).
// forge_backward_adamw issues both on one stream in that order, so the caller
// no longer has to.
//
// The contraction here runs over d_out (M): dX[k][n] = sum_m dY[k][m] W[n][m].
// Both operands keep the contraction index contiguous (dY rows, W rows), so
// both are K-major for the tensor core: TMA boxes of 64 bf16 of d_out (one
// 128-byte swizzle row) x 128 token rows (A) or x 256 weight rows (B).  One
// CTA per SM, persistent over 128 (tokens) x 256 (d_in) output tiles ordered
// token-fastest, so a wave of tiles shares W's rows in L2 while dY streams;
// warp 0 is the TMA producer, lane 0 of warp 1 the MMA issuer, warps 4-11 the
// epilogue (TMEM -> fp32 -> bf16, nearest even, 32-byte row segments per
// lane).  The accumulator is double-buffered in TMEM (2 x 256 columns).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "forge.h"
#include "forge_device.h"
#include "forge_kernel.cuh"

namespace forge {
namespace dgrad {

constexpr int BT = 128;  // tokens per tile: UMMA M, TMEM lanes
constexpr int BN = 256;  // d_in per tile: UMMA N, TMEM columns per accumulator
constexpr int BK = 64;   // d_out per stage: one 128-byte swizzle row of bf16
constexpr int UK = 16;   // d_out per MMA instruction (kind::f16)
constexpr int kStages = 4;
constexpr int kStageA = BT * BK * 2;  // 16 KB
constexpr int kStageB = BN * BK * 2;  // 32 KB
constexpr int kStageBytes = kStageA + kStageB;
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 8;
constexpr int kSmemBar = kStages * kStageBytes;
constexpr int kSmemBytes = kSmemBar + 256;
constexpr int kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = ptx::make_idesc(1, 1, false, false, BT, BN);  // bf16, K-major

struct DParams {
    int64_t K, N, M;
    int32_t tiles_t, tiles_n;
    __nv_bfloat16* dX;
    int32_t vec_ok;  // N % 8 == 0 and dX 16-byte aligned: 16-byte stores
    Params w;        // timeout_ns and status for the bounded waits
};

// 16 accumulator columns of one token row -> bf16 (nearest even) at
// dX[row][col0 ..], 32 bytes per lane; columns past N and rows past K are
// skipped.
__device__ __forceinline__ void store_row_chunk(const DParams& p, int64_t row, int64_t col0,
                                                const uint32_t (&r)[16])
{
    if (row >= p.K || col0 >= p.N) return;
    __nv_bfloat16* dst = p.dX + row * p.N + col0;
    if (p.vec_ok && col0 + 16 <= p.N) {
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const __nv_bfloat162 h =
                __floats2bfloat162_rn(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            w[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (col0 + j < p.N) dst[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    forge_dgrad_kernel(const __grid_constant__ CUtensorMap tmA,  // dY [K, M]
                       const __grid_constant__ CUtensorMap tmB,  // W  [N, M]
                       const DParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSmemBar);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&tfull[b], 1);
            ptx::mbar_init(&tempty[b], kEpiWarps);
        }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int32_t total = p.tiles_t * p.tiles_n;
    const int32_t nk = static_cast<int32_t>((p.M + BK - 1) / BK);

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_mask = 0, last_parity = 0;
            bool ok = true;
            for (int32_t t = blockIdx.x; ok && t < total; t += gridDim.x) {
                const int32_t t0 = (t % p.tiles_t) * BT;
                const int32_t n0 = (t / p.tiles_t) * BN;
                for (int32_t kb = 0; kb < nk; ++kb) {
                    if (!wait_bounded(&empty[s], ph ^ 1u, abort_flag, p.w)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&full[s], kStageBytes);
                    uint8_t* sa = smem + s * kStageBytes;
                    ptx::tma_load_2d(sa, &tmA, &full[s], kb * BK, t0);
                    ptx::tma_load_2d(sa + kStageA, &tmB, &full[s], kb * BK, n0);
                    issued_mask |= 1u << s;
                    last_parity = (last_parity & ~(1u << s)) | (ph << s);
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // wait (bounded) for this thread's copies still in flight
                const uint64_t tw = ptx::globaltimer_ns();
                for (int q = 0; q < kStages; ++q) {
                    if (!(issued_mask & (1u << q))) continue;
                    const uint32_t a = ptx::smem_addr(&full[q]);
                    while (!ptx::mbar_try_wait(a, (last_parity >> q) & 1u)) {
                        if (static_cast<int64_t>(ptx::globaltimer_ns() - tw) > p.w.timeout_ns)
                            break;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer (lane 0)
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t ct = 0;
            bool ok = true;
            bool issued_any = false;
            for (int32_t t = blockIdx.x; ok && t < total; t += gridDim.x) {
                const uint32_t b = ct & 1u;
                ok = wait_bounded(&tempty[b], ((ct >> 1) & 1u) ^ 1u, abort_flag, p.w);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * BN;
                for (int32_t kb = 0; kb < nk; ++kb) {
                    ok = wait_bounded(&full[s], ph, abort_flag, p.w);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_addr(smem + s * kStageBytes);
                    const uint32_t sb = sa + kStageA;
#pragma unroll
                    for (int ks = 0; ks < BK / UK; ++ks) {
                        // K-major, 128-byte swizzle: 8-row groups 1024 bytes apart;
                        // the k sub-block is a 32-byte step inside the swizzle row
                        const uint64_t ad = ptx::smem_desc_sw128(sa + ks * UK * 2, 16, 1024);
                        const uint64_t bd = ptx::smem_desc_sw128(sb + ks * UK * 2, 16, 1024);
                        ptx::umma_f16(d_tmem, ad, bd, kIdesc, (kb | ks) != 0 ? 1u : 0u);
                    }
                    ptx::umma_commit(&empty[s]);
                    issued_any = true;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::umma_commit(&tfull[b]);
                ++ct;
            }
            if (!ok && issued_any) {
                ptx::umma_commit(drain);
                const uint32_t a = ptx::smem_addr(drain);
                const uint64_t tw = ptx::globaltimer_ns();
                while (!ptx::mbar_try_wait(a, 0)) {
                    if (static_cast<int64_t>(ptx::globaltimer_ns() - tw) > p.w.timeout_ns) break;
                }
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------------------------------------------- epilogue
        // Warp (q, half): TMEM lanes 32q.. (tokens) x columns 128 half .. (d_in),
        // in 16-column chunks; each lane stores its own row's 32 bytes.
        const int q = warp & 3;
        const int half = (warp - kEpiWarp0) >> 2;
        uint32_t ct = 0;
        for (int32_t t = blockIdx.x; t < total; t += gridDim.x) {
            const uint32_t b = ct & 1u;
            if (!warp_wait(&tfull[b], (ct >> 1) & 1u, abort_flag, p.w, lane)) break;
            ptx::tc_fence_after();
            const int64_t row = static_cast<int64_t>(t % p.tiles_t) * BT + 32 * q + lane;
            const int64_t cbase = static_cast<int64_t>(t / p.tiles_t) * BN + 128 * half;
            const uint32_t tcol =
                tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * BN + 128 * half;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t r[16];
                ptx::tmem_ld_32x32b_x16(tcol + 16 * c, r);
                ptx::tmem_ld_wait();
                if (c == 7) {  // accumulator fully read
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&tempty[b]);
                }
                store_row_chunk(p, row, cbase + 16 * c, r);
            }
            ++ct;
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// CTA-pair form: a pair owns 256 tokens x 256 d_in.  CTA r loads token rows
// t0 + 128 r (A) and weight rows n0 + 128 r (B); the even CTA issues
// tcgen05.mma.cta_group::2 (256 x 256 x 16), which leaves each CTA's 128
// token rows x 256 columns in its own TMEM, and both CTAs run the same
// epilogue on their rows.  A stage is 32 KB per CTA, six stages.
constexpr int kPairStages = 6;
constexpr int kPairStageA = BT * BK * 2;          // this CTA's 128 token rows
constexpr int kPairStageB = (BN / 2) * BK * 2;    // this CTA's 128 weight rows
constexpr int kPairStageBytes = kPairStageA + kPairStageB;
constexpr int kPairSmemBar = kPairStages * kPairStageBytes;
constexpr int kPairSmemAlloc = kPairSmemBar + 256 + 1024;
constexpr uint32_t kPairIdesc = ptx::make_idesc(1, 1, false, false, 2 * BT, BN);

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    forge_dgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA,  // dY, boxes of 128 rows
                            const __grid_constant__ CUtensorMap tmB,  // W, boxes of 128 rows
                            const DParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPairSmemBar);
    uint64_t* empty = full + kPairStages;
    uint64_t* tfull = empty + kPairStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();  // 0 or 1
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&tfull[b], 1);
            ptx::mbar_init(&tempty[b], 2 * kEpiWarps);
        }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(tmem_slot, kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int32_t total = p.tiles_t * p.tiles_n;  // pair tiles
    const int32_t nk = static_cast<int32_t>((p.M + BK - 1) / BK);
    const int32_t first = static_cast<int32_t>(blockIdx.x >> 1);
    const int32_t step = static_cast<int32_t>(gridDim.x >> 1);

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer (both CTAs)
        if (lane == 0) {
            const uint32_t full0 = ptx::mapa_shared(ptx::smem_addr(&full[0]), 0);
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_mask = 0, last_parity = 0;
            bool ok = true;
            for (int32_t t = first; ok && t < total; t += step) {
                const int32_t t0 = (t % p.tiles_t) * (2 * BT) + static_cast<int32_t>(rank) * BT;
                const int32_t n0 = (t / p.tiles_t) * BN + static_cast<int32_t>(rank) * (BN / 2);
                for (int32_t kb = 0; kb < nk; ++kb) {
                    if (!wait_bounded(&empty[s], ph ^ 1u, abort_flag, p.w)) {
                        ok = false;
                        break;
                    }
                    if (leader) ptx::mbar_arrive_expect_tx(&full[s], 2 * kPairStageBytes);
                    uint8_t* sa = smem + s * kPairStageBytes;
                    const uint32_t bar = full0 + s * 8;
                    ptx::tma_load_2d_pair(sa, &tmA, bar, kb * BK, t0);
                    ptx::tma_load_2d_pair(sa + kPairStageA, &tmB, bar, kb * BK, n0);
                    issued_mask |= 1u << s;
                    last_parity = (last_parity & ~(1u << s)) | (ph << s);
                    if (++s == kPairStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok && leader) {
                // the pair's copies all complete on the even CTA's barriers
                const uint64_t tw = ptx::globaltimer_ns();
                for (int q = 0; q < kPairStages; ++q) {
                    if (!(issued_mask & (1u << q))) continue;
                    const uint32_t a = ptx::smem_addr(&full[q]);
                    while (!ptx::mbar_try_wait(a, (last_parity >> q) & 1u)) {
                        if (static_cast<int64_t>(ptx::globaltimer_ns() - tw) > p.w.timeout_ns)
                            break;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- pair MMA issuer (even CTA, lane 0)
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t ct = 0;
            bool ok = true;
            bool issued_any = false;
            for (int32_t t = first; ok && t < total; t += step) {
                const uint32_t b = ct & 1u;
                ok = wait_bounded(&tempty[b], ((ct >> 1) & 1u) ^ 1u, abort_flag, p.w);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * BN;
                for (int32_t kb = 0; kb < nk; ++kb) {
                    ok = wait_bounded(&full[s], ph, abort_flag, p.w);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_addr(smem + s * kPairStageBytes);
                    const uint32_t sb = sa + kPairStageA;
#pragma unroll
                    for (int ks = 0; ks < BK / UK; ++ks) {
                        const uint64_t ad = ptx::smem_desc_sw128(sa + ks * UK * 2, 16, 1024);
                        const uint64_t bd = ptx::smem_desc_sw128(sb + ks * UK * 2, 16, 1024);
                        ptx::umma_f16_pair(d_tmem, ad, bd, kPairIdesc, (kb | ks) != 0 ? 1u : 0u);
                    }
                    ptx::umma_commit_pair(&empty[s], 0x3);  // the stage of both CTAs is free
                    issued_any = true;
                    if (++s == kPairStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::umma_commit_pair(&tfull[b], 0x3);  // both accumulators ready
                ++ct;
            }
            if (!ok && issued_any) {
                ptx::umma_commit_pair(drain, 0x1);
                const uint32_t a = ptx::smem_addr(drain);
                const uint64_t tw = ptx::globaltimer_ns();
                while (!ptx::mbar_try_wait(a, 0)) {
                    if (static_cast<int64_t>(ptx::globaltimer_ns() - tw) > p.w.timeout_ns) break;
                }
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int q = warp & 3;
        const int half = (warp - kEpiWarp0) >> 2;
        const uint32_t tempty0 = ptx::mapa_shared(ptx::smem_addr(&tempty[0]), 0);
        uint32_t ct = 0;
        for (int32_t t = first; t < total; t += step) {
            const uint32_t b = ct & 1u;
            if (!warp_wait(&tfull[b], (ct >> 1) & 1u, abort_flag, p.w, lane)) break;
            ptx::tc_fence_after();
            const int64_t row = static_cast<int64_t>(t % p.tiles_t) * (2 * BT) +
                                static_cast<int64_t>(rank) * BT + 32 * q + lane;
            const int64_t cbase = static_cast<int64_t>(t / p.tiles_t) * BN + 128 * half;
            const uint32_t tcol =
                tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * BN + 128 * half;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t r[16];
                ptx::tmem_ld_32x32b_x16(tcol + 16 * c, r);
                ptx::tmem_ld_wait();
                if (c == 7) {  // accumulator fully read: tell the pair's MMA issuer
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (leader)
                            ptx::mbar_arrive(&tempty[b]);
                        else
                            ptx::mbar_arrive_cluster(tempty0 + 8 * b);
                    }
                }
                store_row_chunk(p, row, cbase + 16 * c, r);
            }
            ++ct;
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        }
    }

    ptx::tc_fence_before();
    ptx::cluster_sync();  // no CTA leaves while the other may still signal it
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// fp32 -> bf16, nearest even: the bf16 copy of W [rows, cols] the input
// gradient reads when the caller has none, written with rows ld elements
// apart (ld >= cols; the padding is left unwritten).
__global__ void __launch_bounds__(256) forge_round_bf16_kernel(const float* __restrict__ src,
                                                               __nv_bfloat16* __restrict__ dst,
                                                               int64_t rows, int64_t cols,
                                                               int64_t ld)
{
    const int64_t n = rows * cols;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        const int64_t r = ld == cols ? 0 : i / cols;
        dst[i + r * (ld - cols)] = __float2bfloat16_rn(__ldcs(src + i));
    }
}

bool aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// CTA pairs unless the call has a single 128-token tile (or FORGE_DGRAD_KERNEL
// = single, read on every call, asks for the one-CTA kernel).
bool use_pairs(int64_t K)
{
    const char* e = std::getenv("FORGE_DGRAD_KERNEL");
    if (e && std::strcmp(e, "single") == 0) return false;
    if (e && std::strcmp(e, "pair") == 0) return true;
    return K > BT;
}

// Row stride in bytes TMA needs for M bf16 columns: M * 2 rounded up to 16.
int64_t padded_row(int64_t M) { return (M * 2 + 15) / 16 * 16; }

// Whether a [*, M] bf16 operand at base must be staged before TMA reads it.
bool needs_stage(const void* base, int64_t M) { return !aligned(base, 16) || (M * 2) % 16 != 0; }

// ldA, ldB: the row strides in bytes of dY and Wb (multiples of 16, bases
// 16-byte aligned).
cudaError_t launch(const void* dY, const void* Wb, void* dX, int64_t M, int64_t N, int64_t K,
                   int64_t ldA, int64_t ldB, int sms, cudaStream_t stream)
{
    const bool pairs = use_pairs(K);
    CUtensorMap ta, tb;
    if (encode_bf16_kmajor(&ta, dY, M, K, BT, ldA) != cudaSuccess ||
        encode_bf16_kmajor(&tb, Wb, M, N, pairs ? BN / 2 : BN, ldB) != cudaSuccess)
        return cudaErrorInvalidValue;
    DParams p{};
    p.K = K;
    p.N = N;
    p.M = M;
    p.tiles_t = static_cast<int32_t>((K + (pairs ? 2 * BT : BT) - 1) / (pairs ? 2 * BT : BT));
    p.tiles_n = static_cast<int32_t>((N + BN - 1) / BN);
    p.dX = static_cast<__nv_bfloat16*>(dX);
    p.vec_ok = (N % 8 == 0) && aligned(dX, 16);
    p.w.timeout_ns = wait_timeout();
    p.w.status = device_status_word();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int64_t total = static_cast<int64_t>(p.tiles_t) * p.tiles_n;
    if (!pairs) {
        static unsigned long long attr_done = 0;  // one bit per device ordinal < 64
        const unsigned long long bit = 1ull << (dev & 63);
        if (!(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & bit)) {
            e = cudaFuncSetAttribute(forge_dgrad_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
            if (e != cudaSuccess) return e;
            __atomic_fetch_or(&attr_done, bit, __ATOMIC_ACQ_REL);
        }
        const int grid = static_cast<int>(total < sms ? total : sms);
        forge_dgrad_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(ta, tb, p);
        return cudaGetLastError();
    }
    // the grid: as many pairs as can be resident at once, at most one per tile
    static int max_clusters[64] = {0};
    int& mc = max_clusters[dev & 63];
    if (__atomic_load_n(&mc, __ATOMIC_ACQUIRE) == 0) {
        e = cudaFuncSetAttribute(forge_dgrad_pair_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmemAlloc);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kPairSmemAlloc;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, forge_dgrad_pair_kernel, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        __atomic_store_n(&mc, n, __ATOMIC_RELEASE);
    }
    const int64_t nc = total < mc ? total : mc;
    forge_dgrad_pair_kernel<<<static_cast<int>(2 * nc), kThreads, kPairSmemAlloc, stream>>>(ta, tb,
                                                                                          p);
    return cudaGetLastError();
}

// Host checks of the input-gradient call.  Wb may be NULL only where the
// caller lets the library round W itself (wb_optional).
forge_status check(const void* dY, const void* Wb, const void* dX, int64_t M, int64_t N,
                   int64_t K, forge_dtype in_dtype, bool wb_optional)
{
    if (M < 1 || N < 1 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return FORGE_ERR_INVALID_ARG;
    if (K > 0 && (!dY || !dX)) return FORGE_ERR_INVALID_ARG;
    if (!Wb && !wb_optional) return FORGE_ERR_INVALID_ARG;
    if (in_dtype != FORGE_BF16) return FORGE_ERR_UNSUPPORTED_DTYPE;
    // bases aligned to the element; rows TMA cannot address are staged
    if ((Wb && !aligned(Wb, 2)) || (dY && !aligned(dY, 2)) || (dX && !aligned(dX, 2)))
        return FORGE_ERR_MISALIGNED;
    return FORGE_OK;
}

// dX = dY Wb^T with any row width: dY and Wb rows TMA cannot address (a base
// or a row of M * 2 bytes not a multiple of 16) are staged into rows padded
// to 16 bytes in one stream-ordered scratch allocation from the library's
// pool, freed on `stream` after the launch.  With Wb == NULL the bf16 copy is
// W (fp32 [N, M]) rounded to nearest even into that scratch.
cudaError_t run(const void* dY, const void* Wb, const float* W, void* dX, int64_t M, int64_t N,
                int64_t K, int sms, cudaStream_t stream)
{
    const int64_t pad = padded_row(M);
    const bool stage_a = needs_stage(dY, M);
    const bool stage_b = !Wb || needs_stage(Wb, M);
    const int64_t bytes = (stage_a ? pad * K : 0) + (stage_b ? pad * N : 0);
    void* scratch = nullptr;
    if (bytes > 0) {
        const cudaError_t e = scratch_alloc(&scratch, static_cast<size_t>(bytes), stream);
        if (e != cudaSuccess) return e;
    }
    uint8_t* sp = static_cast<uint8_t*>(scratch);
    const void* opA = dY;
    const void* opB = Wb;
    int64_t ldA = M * 2, ldB = M * 2;
    cudaError_t e = cudaSuccess;
    if (stage_a) {
        e = stage_padded_rows(dY, sp, K, M * 2, pad, stream);
        opA = sp;
        ldA = pad;
        sp += pad * K;
    }
    if (e == cudaSuccess && stage_b) {
        if (!Wb) {
            const int64_t n = N * M;
            const int64_t want = (n + 255) / 256;
            const int blocks = static_cast<int>(want < 8LL * sms ? want : 8LL * sms);
            forge_round_bf16_kernel<<<blocks, 256, 0, stream>>>(
                W, reinterpret_cast<__nv_bfloat16*>(sp), N, M, pad / 2);
            e = cudaGetLastError();
        } else {
            e = stage_padded_rows(Wb, sp, N, M * 2, pad, stream);
        }
        opB = sp;
        ldB = pad;
    }
    if (e == cudaSuccess) e = launch(opA, opB, dX, M, N, K, ldA, ldB, sms, stream);
    if (scratch) {
        const cudaError_t fe = scratch_free(scratch, stream);
        if (e == cudaSuccess) e = fe;
    }
    return e;
}

}  // namespace dgrad
}  // namespace forge

using namespace forge;

extern "C" forge_status forge_dgrad(const void* dY, const void* Wb, void* dX, int64_t M,
                                    int64_t N, int64_t K, forge_dtype in_dtype,
                                    forge_stream_t stream)
{
    forge_status st = dgrad::check(dY, Wb, dX, M, N, K, in_dtype, false);
    if (st != FORGE_OK) return st;
    int sms = 0;
    if ((st = device_sms(&sms)) != FORGE_OK) return st;
    if (K == 0) return FORGE_OK;
    const void* ptrs[] = {dY, Wb, dX};
    if ((st = device_resident(ptrs, 3)) != FORGE_OK) return st;
    const cudaError_t e =
        dgrad::run(dY, Wb, nullptr, dX, M, N, K, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) cudaGetLastError();
    return e == cudaSuccess ? FORGE_OK : FORGE_ERR_CUDA;
}

extern "C" forge_status forge_backward_adamw(const void* X, const void* dY, float* W, void* m,
                                             void* v, const void* Wb, void* dX, int64_t M,
                                             int64_t N, int64_t K, forge_dtype in_dtype,
                                             forge_dtype state_dtype, float lr, float beta1,
                                             float beta2, float eps, float wd, int64_t step,
                                             forge_stream_t stream)
{
    // every check of both halves runs before the first launch
    forge_status st = dgrad::check(dY, Wb, dX, M, N, K, in_dtype, true);
    if (st != FORGE_OK) return st;
    if ((st = adamw_checks(X, dY, W, m, v, M, N, K, in_dtype, state_dtype, lr, beta1, beta2, eps,
                           wd, step)) != FORGE_OK)
        return st;
    int sms = 0;
    if ((st = device_sms(&sms)) != FORGE_OK) return st;
    {
        const void* ptrs[] = {K > 0 ? X : nullptr, K > 0 ? dY : nullptr, W, m, v,
                              K > 0 ? Wb : nullptr, K > 0 ? dX : nullptr};
        if ((st = device_resident(ptrs, 7)) != FORGE_OK) return st;
    }
    // dX from the weights as they are before this step's update (the
    // caller's bf16 copy, or W rounded now) ...
    if (K > 0 &&
        dgrad::run(dY, Wb, W, dX, M, N, K, sms, reinterpret_cast<cudaStream_t>(stream)) !=
            cudaSuccess) {
        cudaGetLastError();
        return FORGE_ERR_CUDA;
    }
    // ... then the fused dW + AdamW that overwrites W, later on the same stream
    return forge_wgrad_adamw(X, dY, W, m, v, M, N, K, in_dtype, state_dtype, lr, beta1, beta2, eps,
                             wd, step, nullptr, stream);
}
