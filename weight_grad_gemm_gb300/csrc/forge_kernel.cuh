// forge_kernel.cuh -- the fused weight-gradient GEMM + optimizer kernel.
//
// dW = X^T dY with the optimizer step applied in the tiled epilogue, so the
// gradient lives only in tensor memory and registers (FORGE assessment PR,
// tessera#565, opening paragraph; "What's already in tree and easy to miss":
// dRhs = matmul(lhs, dy, transposeA=true) and K kept whole per output tile).
//
// Mapping onto the tensor core.  One output tile is 128 (d_out, m) x 256
// (d_in, n).  The UMMA computes D[m][n] = sum_k dY[k][m] X[k][n], i.e. the
// A operand is dY and the B operand is X, both token-major, so both are
// "MN-major" (the contraction index k is the strided one).  D lives in TMEM
// with one lane per m and one 32-bit column per n; the epilogue thread that
// owns lane m therefore touches W[n][m] for consecutive n, and a warp's 32
// lanes cover 32 consecutive m: every global access of the epilogue is a
// fully coalesced 128-byte (fp32) or 64-byte (bf16) row segment.
//
// Roles (384 or 640 threads, one CTA per SM, persistent over a static tile list):
//   warp 0      TMA producer: K-blocks of dY and X into a 4-stage ring
//   warp 1      TMEM allocator; lane 0 alone issues tcgen05.mma into one of
//               two 128x256 fp32 accumulators (512 TMEM columns)
//   warps 2-3   cp.async loader for operands TMA cannot address
//   warps 4-    epilogue: tcgen05.ld the accumulator, apply AdamW / SGD-m /
//               plain store, write W and the state back; two warpgroups
//               (dense calls) or four (grouped calls) split the 256 columns
// Each output tile is computed by exactly one CTA over the whole K in a
// fixed order: no split-K and no atomics, so results are bitwise
// reproducible and independent of the schedule (P1).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "forge_ptx.cuh"

namespace forge {

enum InType : int { IN_BF16 = 0, IN_E4M3 = 1 };
enum OpKind : int { OP_ADAMW = 0, OP_SGDM = 1, OP_DW = 2 };
enum StateType : int { ST_F32 = 0, ST_BF16 = 1 };

// device status word values (match forge_status)
constexpr int kDevOk = 0;
constexpr int kDevInvalidArg = -1;
constexpr int kDevTimeout = -6;

constexpr int kEpiWarp0 = 4;  // warps 0-3: producer, MMA issuer, cp.async loader
constexpr int BM = 128;  // m (d_out) per tile = UMMA M = TMEM lanes
constexpr int BN = 256;  // n (d_in) per tile  = UMMA N = TMEM columns per accumulator
constexpr int kStages = 4;
constexpr int kStageA = 16384;  // BK rows x 128 m x elemsize
constexpr int kStageB = 32768;  // BK rows x 256 n x elemsize
constexpr int kStageBytes = kStageA + kStageB;
constexpr int kTmemCols = 512;  // two 256-column accumulators
constexpr int kMaxExperts = 1024;
constexpr int kMaxProblems = 8;  // multi-problem calls: problems sharing X per launch

// Epilogue geometry for EW epilogue warps.  Warp (q, grp) owns TMEM lane
// quarter q and warp_cols accumulator columns, walked in chunks of
// chunk_cols (n) x 32 (m); after a transpose within each quad of lanes a lane
// holds four consecutive m for chunk_n consecutive n.  Sixteen warps with 8-column
// chunks keep more state loads in flight per SM (the epilogue-bound grouped
// calls); eight warps with 16-column chunks leave more issue slots to the
// producer and the MMA issuer (the MMA-bound dense calls).
template <int EW>
struct Epi {
    static_assert(EW == 8 || EW == 16, "two or four warpgroups");
    static constexpr int warps = EW;
    static constexpr int threads = (kEpiWarp0 + EW) * 32;
    static constexpr int groups = EW / 4;  // column groups per TMEM lane quarter
    static constexpr int warp_cols = BN / groups;
    static constexpr int chunk_cols = EW == 16 ? 8 : 16;
    static constexpr int chunk_n = chunk_cols / 4;
    static constexpr int chunks = warp_cols / chunk_cols;
};
template <bool GROUPED>
using EpiFor = Epi<GROUPED ? 16 : 8>;

// Shared memory of a kernel whose operand ring takes RING bytes: the ring,
// the mbarriers, then the grouped schedule (expert offsets and order), sized
// per launch for the call's E experts.  Shared memory and L1 share 256 KB per
// SM, and the carve-out is taken in steps (..., 164, 196, 228 KB).  The
// epilogue's state loads occupy L1 while in flight: at the 228 KB step (a
// 28 KB L1) a decay-only stream of W, m, v measured 4.5 TB/s, at the 196 KB
// step (60 KB) 6.1 TB/s.  Both kernels' rings (six 32 KB stages per CTA of a
// pair, four 48 KB stages for a single CTA) fit the 196 KB step with their
// barriers and the table of up to kCarveoutExperts experts, the 1 KB the
// runtime keeps per block included; calls with more experts take the next.
template <int RING>
struct SmemLayout {
    static constexpr int bar = RING;
    static constexpr int sched = bar + 256;
    // dynamic shared memory for a call over `experts` experts, with slack
    // for the 1024-byte alignment of the ring
    static constexpr int alloc(int experts)
    {
        return ((sched + 4 * (2 * experts + 2) + 127) & ~127) + 1024;
    }
};
constexpr int kCarveout196 = 196 * 1024;
constexpr int kSmemPerCtaMax = 227 * 1024;  // dynamic shared memory one CTA may take
constexpr int kCarveoutExperts = 128;
using SmemCta = SmemLayout<kStages * kStageBytes>;
static_assert(SmemCta::alloc(kCarveoutExperts) + 1024 <= kCarveout196, "196 KB step");

template <int IT>
struct InTraits;
template <>
struct InTraits<IN_BF16> {
    static constexpr int esize = 2;
    static constexpr int BK = 64;       // k rows per stage
    static constexpr int box_mn = 64;   // elements per 128-byte swizzle row
    static constexpr int umma_k = 16;   // k per tcgen05.mma
    static constexpr uint32_t fmt = 1;  // bf16 (kind::f16)
};
template <>
struct InTraits<IN_E4M3> {
    static constexpr int esize = 1;
    static constexpr int BK = 128;
    static constexpr int box_mn = 128;
    static constexpr int umma_k = 32;
    static constexpr uint32_t fmt = 0;  // e4m3 (kind::f8f6f4)
};

struct Params {
    int64_t M, N, K;         // dense sizes (K unused when grouped)
    int64_t T_max;           // grouped: rows of the packed X / dY
    const int32_t* offsets;  // grouped: [E+1] on the device
    int32_t E;               // 1 when dense
    int32_t tiles_m, tiles_n;
    int32_t raster_band;  // d_out tiles per raster band, 1 <= raster_band <= tiles_m
    int32_t has_maps;  // 0 when there are no token rows at all (maps left unencoded)
    int32_t vec_ok;    // M % 4 == 0 and W / state / dW aligned for 4-element vectors
    // Operands whose rows TMA cannot address (row stride or base not a
    // multiple of 16 bytes), when they are not staged into a padded copy,
    // are copied by the cp.async loader:
    int32_t manual_a, manual_b;  // dY / X loaded by cp.async
    int32_t gran_a, gran_b;      // cp.async width in bytes (4 or 8)
    const uint8_t* gA;           // dY base
    const uint8_t* gB;           // X base
    float* W;
    void* s1;  // m (AdamW) or momentum (SGD)
    void* s2;  // v (AdamW)
    float* dW;
    const float* scales;  // {sX, sdY} for e4m3, else null
    // AdamW
    float decay;         // 1 - lr * wd
    float b1, omb1, b2, omb2;
    float step_size;     // lr / (1 - b1^t)
    float inv_sqrt_bc2;  // 1 / sqrt(1 - b2^t)
    float eps;
    // SGD momentum
    float lr, mu, wd;
    int64_t timeout_ns;
    int* status;  // device status word
    // Multi-problem calls (P > 0): problems j = 0 .. P-1 share X, N and K and
    // each has its own dY [K, M_of[j]] and W, m, v [N, M_of[j]]; problem j's
    // tiles are [tile_begin[j], tile_begin[j + 1]) of the list, d_out fastest
    // over tiles_m_of[j] tile rows.  Entries past P hold tile_begin = INT32_MAX.
    int32_t P;
    int32_t tile_begin[kMaxProblems + 1];
    int32_t tiles_m_of[kMaxProblems];
    int64_t M_of[kMaxProblems];
    float* W_of[kMaxProblems];
    void* s1_of[kMaxProblems];
    void* s2_of[kMaxProblems];
};

// The dY tensor maps of a multi-problem call, one per problem.
struct MultiMaps {
    CUtensorMap a[kMaxProblems];
};

// Problem j's entry of a per-problem array of Params, by compile-time
// indices only (select chain), so the parameter array is never indexed at
// run time.
template <class T, int LEN>
__device__ __forceinline__ T pick(const T (&arr)[LEN], int32_t j)
{
    T r = arr[0];
#pragma unroll
    for (int i = 1; i < LEN; ++i)
        if (j == i) r = arr[i];
    return r;
}

struct Tile {
    int32_t m0, n0;
    int64_t k_begin, k_end;  // token rows [k_begin, k_end) of X / dY
    int64_t pbase;           // element offset of this tile's expert block in W / m / v
    int32_t prob;            // multi-problem calls: the tile's problem
};

// Static tile list.  Dense: tiles ordered m-fastest so the CTAs of one wave
// share X column blocks in L2.  Grouped: experts sorted by token count,
// heaviest first (stable), each contributing tiles_m * tiles_n tiles.
struct Sched {
    int32_t tiles_m, tiles_n, per_expert, total;
    int32_t m_step;        // d_out rows per tile: 128 (one CTA) or 256 (CTA pair)
    int32_t m_off;         // this CTA's first row within the tile (128 for the odd CTA of a pair)
    int32_t first, step;   // this CTA's share of the tile list: first, first + step, ...
    int32_t count;         // tiles in this CTA's share
    int32_t alternate;     // walk the share front, back, front, ... (grouped)
    int32_t band;          // d_out tiles per raster band (tiles_m: plain m-fastest order)

    // The i-th tile this CTA processes.  With `alternate`, a share of the
    // heavy-first grouped list is walked from both ends, so heavy tiles
    // (MMA-bound) and light ones (epilogue-bound, down to decay-only tiles of
    // experts without tokens) alternate and overlap through the two
    // accumulators.
    __device__ __forceinline__ int32_t nth(int32_t i) const
    {
        const int32_t j = alternate ? ((i & 1) ? count - 1 - (i >> 1) : (i >> 1)) : i;
        return first + j * step;
    }

    __device__ __forceinline__ void set_share(int32_t f, int32_t s, int32_t alt)
    {
        first = f;
        step = s;
        count = f < total ? (total - f + s - 1) / s : 0;
        alternate = alt;
    }
    const int32_t* offs;   // smem copy of offsets (grouped) or null
    const int32_t* order;  // smem expert order (grouped) or null
    const Params* multi;   // the launch's parameters for a multi-problem call, else null
    int64_t K, MN;

    __device__ __forceinline__ Tile get(int32_t t) const
    {
        Tile r;
        r.prob = 0;
        if (multi) {
            // problem j holds tiles [tile_begin[j], tile_begin[j + 1])
            const Params& q = *multi;
            int32_t j = 0;
#pragma unroll
            for (int i = 1; i < kMaxProblems; ++i) j += t >= q.tile_begin[i] ? 1 : 0;
            const int32_t local = t - pick(q.tile_begin, j);
            const int32_t tm = pick(q.tiles_m_of, j);
            // the problem's tiles in raster bands, as below
            const int32_t bw = band < tm ? band : tm;
            const int32_t per_band = bw * tiles_n;
            const int32_t g = local / per_band;
            const int32_t within = local - g * per_band;
            const int32_t rows_left = tm - g * bw;
            const int32_t gsz = rows_left < bw ? rows_left : bw;
            r.m0 = (g * bw + within % gsz) * m_step + m_off;
            r.n0 = ((g & 1) ? tiles_n - 1 - within / gsz : within / gsz) * BN;
            r.k_begin = 0;
            r.k_end = K;
            r.pbase = 0;
            r.prob = j;
            return r;
        }
        int32_t j = t / per_expert;
        int32_t local = t - j * per_expert;
        // Raster: bands of `band` d_out tiles; within a band, d_out fastest,
        // then across all d_in tiles, odd bands from the last d_in tile back
        // to the first.  A wave of tiles then touches only the band's dY
        // columns, which stay in L2 while the band lasts, and a band starts
        // on the X columns the previous band ended on, still in L2.
        const int32_t per_band = band * tiles_n;
        const int32_t g = local / per_band;
        const int32_t within = local - g * per_band;
        const int32_t rows_left = tiles_m - g * band;
        const int32_t gsz = rows_left < band ? rows_left : band;
        int32_t mt = g * band + within % gsz;
        int32_t nt = within / gsz;
        if (g & 1) nt = tiles_n - 1 - nt;  // serpentine: odd bands walk d_in backwards
        r.m0 = mt * m_step + m_off;
        r.n0 = nt * BN;
        if (order) {
            int32_t e = order[j];
            r.k_begin = offs[e];
            r.k_end = offs[e + 1];
            r.pbase = static_cast<int64_t>(e) * MN;
        } else {
            r.k_begin = 0;
            r.k_end = K;
            r.pbase = 0;
        }
        return r;
    }
};

// Bounded wait on an mbarrier phase.  Gives up after `timeout_ns` of
// wall-clock time or when another role of this CTA has given up, records
// FORGE_ERR_TIMEOUT in the device status word and returns false.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, const Params& p)
{
    const uint32_t a = ptx::smem_addr(bar);
    if (ptx::mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(a, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (static_cast<int64_t>(ptx::globaltimer_ns() - t0) > p.timeout_ns) {
                *abort_flag = 1;
                *reinterpret_cast<volatile int*>(p.status) = kDevTimeout;
                return false;
            }
        }
    }
}

// Lane 0 waits (bounded); the outcome is broadcast to the whole warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          const Params& p, int lane)
{
    int ok = 0;
    if (lane == 0) ok = wait_bounded(bar, parity, abort_flag, p) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// ------------------------------------------------------------------ epilogue

template <int ST>
struct StateIO;
template <>
struct StateIO<ST_F32> {
    static __device__ __forceinline__ float ld(const void* base, int64_t i)
    {
        return __ldcs(static_cast<const float*>(base) + i);
    }
    static __device__ __forceinline__ void st(void* base, int64_t i, float x)
    {
        __stcs(static_cast<float*>(base) + i, x);
    }
    // four consecutive elements starting at i (i % 4 == 0, 16-byte aligned)
    static __device__ __forceinline__ void ld4(const void* base, int64_t i, float* o)
    {
        const float4 v =
            __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i));
        o[0] = v.x;
        o[1] = v.y;
        o[2] = v.z;
        o[3] = v.w;
    }
    static __device__ __forceinline__ void st4(void* base, int64_t i, const float* x)
    {
        __stcs(reinterpret_cast<float4*>(static_cast<float*>(base) + i),
               make_float4(x[0], x[1], x[2], x[3]));
    }
};
template <>
struct StateIO<ST_BF16> {
    static __device__ __forceinline__ float ld(const void* base, int64_t i)
    {
        unsigned short u = __ldcs(static_cast<const unsigned short*>(base) + i);
        return __uint_as_float(static_cast<uint32_t>(u) << 16);
    }
    static __device__ __forceinline__ void st(void* base, int64_t i, float x)
    {
        __stcs(static_cast<unsigned short*>(base) + i,
               __bfloat16_as_ushort(__float2bfloat16_rn(x)));
    }
    // four consecutive bf16 (8 bytes, 8-byte aligned); bf16 widens exactly
    static __device__ __forceinline__ void ld4(const void* base, int64_t i, float* o)
    {
        const uint2 u =
            __ldcs(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(base) + i));
        o[0] = __uint_as_float(u.x << 16);
        o[1] = __uint_as_float(u.x & 0xFFFF0000u);
        o[2] = __uint_as_float(u.y << 16);
        o[3] = __uint_as_float(u.y & 0xFFFF0000u);
    }
    static __device__ __forceinline__ void st4(void* base, int64_t i, const float* x)
    {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]);  // round to nearest even
        const __nv_bfloat162 hi = __floats2bfloat162_rn(x[2], x[3]);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&lo);
        u.y = *reinterpret_cast<const uint32_t*>(&hi);
        __stcs(reinterpret_cast<uint2*>(static_cast<unsigned short*>(base) + i), u);
    }
};

// One lane's share of a (4 CN) (n) x 32 (m) accumulator chunk: CN n rows of
// four consecutive m each; element [jj * 4 + i] is (n = CN ns + jj, m = 4 mg + i).
template <int CN>
struct Chunk {
    float g[4 * CN];
    float w[4 * CN];
    float a[4 * CN];  // m (AdamW) or momentum (SGD)
    float b[4 * CN];  // v (AdamW)
};

// The optimizer step on four consecutive parameters of one row.
template <int OP>
__device__ __forceinline__ void step4(const Params& p, const float* g, float* w, float* a,
                                      float* b)
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (OP == OP_SGDM) {
            // g' = g + wd W;  buf' = mu buf + g';  W' = W - lr buf'
            const float g1 = fmaf(p.wd, w[i], g[i]);
            a[i] = fmaf(p.mu, a[i], g1);
            w[i] = fmaf(-p.lr, a[i], w[i]);
        } else if constexpr (OP == OP_ADAMW) {
            // m' = b1 m + (1-b1) g;  v' = b2 v + (1-b2) g^2
            // W' = W (1 - lr wd) - (lr / bc1) m' / (sqrt(v') / sqrt(bc2) + eps)
            const float gi = g[i];
            a[i] = fmaf(p.b1, a[i], p.omb1 * gi);
            b[i] = fmaf(p.b2, b[i], p.omb2 * (gi * gi));
            const float den = fmaf(ptx::sqrt_approx(b[i]), p.inv_sqrt_bc2, p.eps);
            w[i] = fmaf(-p.step_size * a[i], ptx::rcp_approx(den), w[i] * p.decay);
        }
    }
}

// ------------------------------------------------------------------ epilogue role

// Epilogue warps of one CTA (EC::warps of them, from warp kEpiWarp0).  Warp
// (q, grp) owns TMEM lanes 32q..32q+31 (m) and columns EC::warp_cols grp ..
// EC::warp_cols (grp + 1) - 1 (n) of the accumulator, walked in chunks.  Each
// chunk goes TMEM -> registers (lane = m) -> a transpose within each quad of
// lanes (shuffles, no shared memory) that leaves lane 4 mg + ns holding
// m = 4 mg .. 4 mg + 3 for n = chunk_n ns .. chunk_n ns + chunk_n - 1, so every
// global access is a 16-byte (fp32) or 8-byte (bf16) vector and a warp
// instruction covers four 128-byte (or 64-byte) row segments.  The state loads of chunk c+1 are in flight while
// chunk c is updated and stored.  `release_acc(b)` hands accumulator buffer b
// back to the MMA issuer once it has been read.
// One chunk of TMEM columns (the overload matches the chunk width).
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[8])
{
    ptx::tmem_ld_32x32b_x8(taddr, r);
}
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[16])
{
    ptx::tmem_ld_32x32b_x16(taddr, r);
}

// Lane 4 mg + i holds row m = 4 mg + i of a chunk: x[CN s + jj] is column
// n = CN s + jj (s, i = 0..3).  Afterwards lane 4 mg + s holds column
// n = CN s + jj of the four rows 4 mg + i in x[CN i + jj]: the 4 x 4
// transpose of (lane within the quad) and s, for each jj, in two butterfly
// exchanges, each swapping one bit of the lane index with the same bit of s.
template <int CN>
__device__ __forceinline__ void quad_transpose(float (&x)[4 * CN], int lane)
{
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const bool up = (lane >> b) & 1;
#pragma unroll
        for (int jj = 0; jj < CN; ++jj)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                if (s & (1 << b)) continue;
                const int lo = CN * s + jj;             // bit b of s clear
                const int hi = CN * (s | (1 << b)) + jj;  // bit b of s set
                // the element whose lane bit and s bit differ changes sides
                const float recv = __shfl_xor_sync(0xffffffffu, up ? x[lo] : x[hi], 1 << b);
                if (up)
                    x[lo] = recv;
                else
                    x[hi] = recv;
            }
    }
}

template <int IT, int OP, int ST, class EC, bool MULTI = false, class ReleaseAcc>
__device__ __forceinline__ void epilogue_role(const Params& p, const Sched& sc,
                                              uint64_t* tfull, uint32_t tmem_base,
                                              volatile int* abort_flag, int warp, int lane,
                                              ReleaseAcc release_acc)
{
    const int ew = warp - kEpiWarp0;
    const int q = warp & 3;     // TMEM lane quarter this warp may access
    const int grp = ew >> 2;    // which EC::warp_cols of the 256 columns
    constexpr int kWarpCols = EC::warp_cols;
    constexpr int kChunkCols = EC::chunk_cols;
    constexpr int kChunkN = EC::chunk_n;
    constexpr int kChunks = EC::chunks;
    using Chunk = forge::Chunk<kChunkN>;
    const int mg = lane >> 2;  // m group: lanes 4 mg .. 4 mg + 3 read TMEM rows 4 mg ..
    const int ns = lane & 3;   // n group within the chunk after the quad transpose
    const int64_t N = p.N;
    float gscale = 1.0f;
    if constexpr (IT == IN_E4M3) gscale = p.scales[0] * p.scales[1];
    uint32_t ct = 0;
    // Two cursors over this CTA's share: the next tile with tokens (whose
    // accumulators are read in the order the MMAs fill them) and the next
    // decay-only tile (an expert without tokens: no accumulator).  With bf16
    // state, while both remain, a warp streams a decay-only tile whenever the
    // next accumulator is not ready yet, so the state of empty experts fills
    // the time the epilogue would otherwise spend waiting on the MMAs (the
    // MoE layer's routings with empty experts ran up to 7% faster).  With
    // fp32 state the same policy was 12-15% slower on those routings: the
    // extra state traffic beside the MMAs costs more than the idle time it
    // fills, so fp32 state keeps the share's own order.  Which tile a warp
    // takes changes only the timing: every tile's update is the same.
    constexpr bool kFillWithDecay = ST == ST_BF16;
    auto next_kind = [&](int32_t from, bool tokens) {
        int32_t i = from;
        for (; i < sc.count; ++i) {
            const Tile x = sc.get(sc.nth(i));
            if ((x.k_end > x.k_begin) == tokens) break;
        }
        return i;
    };
    int32_t it_tok = next_kind(0, true);
    int32_t it_dec = next_kind(0, false);
    while (it_tok < sc.count || it_dec < sc.count) {
        bool take_tok = it_dec >= sc.count;
        if (!kFillWithDecay && !take_tok && it_tok < sc.count) take_tok = it_tok < it_dec;
        else if (!take_tok && it_tok < sc.count) {
            int ready = 0;
            if (lane == 0)
                ready = ptx::mbar_test_wait(ptx::smem_addr(&tfull[ct & 1u]), (ct >> 1) & 1u) ? 1 : 0;
            take_tok = __shfl_sync(0xffffffffu, ready, 0) != 0;
        }
        const int32_t it = take_tok ? it_tok : it_dec;
        if (take_tok)
            it_tok = next_kind(it_tok + 1, true);
        else
            it_dec = next_kind(it_dec + 1, false);
        const int32_t t = sc.nth(it);
        const Tile tl = sc.get(t);
        // the tile's d_out and state (per problem in a multi-problem call)
        const int64_t M = MULTI ? pick(p.M_of, tl.prob) : p.M;
        float* const Wst = MULTI ? pick(p.W_of, tl.prob) : p.W;
        void* const S1 = MULTI ? pick(p.s1_of, tl.prob) : p.s1;
        void* const S2 = MULTI ? pick(p.s2_of, tl.prob) : p.s2;
        const bool has_acc = tl.k_end > tl.k_begin;
        const uint32_t b = ct & 1u;
        if (has_acc) {
            // warp-uniform outcome: the TMEM loads below are warp-collective
            if (!warp_wait(&tfull[b], (ct >> 1) & 1u, abort_flag, p, lane)) break;
            ptx::tc_fence_after();
        }
        const int64_t mrow = tl.m0 + 32 * q + 4 * mg;  // this lane's first m
        const int mvalid = mrow >= M ? 0 : (mrow + 4 <= M ? 4 : static_cast<int>(M - mrow));
        const bool vec = p.vec_ok && mvalid == 4;
        const int64_t n_first = tl.n0 + kWarpCols * grp;
        const int64_t left = N - n_first;
        const int nchunks =
            left <= 0 ? 0
                      : (left >= kWarpCols ? kChunks
                                           : static_cast<int>((left + kChunkCols - 1) / kChunkCols));
        const uint32_t tcol =
            tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * BN + kWarpCols * grp;

        auto release = [&]() {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) release_acc(b);
        };

        // The gradient of chunk c: TMEM -> registers (lane = m row) -> a 4 x 4
        // transpose within each quad of lanes -> this lane's 4 m x chunk_n n
        // (zeros for a tile without tokens).
        auto grad = [&](int c, Chunk& ch) {
            if (has_acc) {
                uint32_t r[kChunkCols];
                tmem_ld_chunk(tcol + kChunkCols * c, r);
                ptx::tmem_ld_wait();
                if (c == nchunks - 1) release();  // accumulator fully read
                float x[kChunkCols];
#pragma unroll
                for (int j = 0; j < kChunkCols; ++j) x[j] = __uint_as_float(r[j]) * gscale;
                quad_transpose<kChunkN>(x, lane);
#pragma unroll
                for (int jj = 0; jj < kChunkN; ++jj)
#pragma unroll
                    for (int i = 0; i < 4; ++i) ch.g[jj * 4 + i] = x[kChunkN * i + jj];
            } else {
#pragma unroll
                for (int j = 0; j < 4 * kChunkN; ++j) ch.g[j] = 0.0f;
            }
        };
        // The state loads of chunk c.
        auto state = [&](int c, Chunk& ch) {
            if constexpr (OP != OP_DW) {
#pragma unroll
                for (int jj = 0; jj < kChunkN; ++jj) {
                    const int64_t n = n_first + kChunkCols * c + kChunkN * ns + jj;
                    if (n >= N || mvalid == 0) continue;
                    const int64_t idx = tl.pbase + n * M + mrow;
                    float* w = ch.w + 4 * jj;
                    float* a = ch.a + 4 * jj;
                    float* bb = ch.b + 4 * jj;
                    if (vec) {
                        StateIO<ST_F32>::ld4(Wst, idx, w);
                        StateIO<ST>::ld4(S1, idx, a);
                        if constexpr (OP == OP_ADAMW) StateIO<ST>::ld4(S2, idx, bb);
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (i < mvalid) {
                                w[i] = StateIO<ST_F32>::ld(Wst, idx + i);
                                a[i] = StateIO<ST>::ld(S1, idx + i);
                                if constexpr (OP == OP_ADAMW) bb[i] = StateIO<ST>::ld(S2, idx + i);
                            }
                    }
                }
            }
        };

        auto process = [&](int c, Chunk& ch) {
#pragma unroll
            for (int jj = 0; jj < kChunkN; ++jj) {
                const int64_t n = n_first + kChunkCols * c + kChunkN * ns + jj;
                if (n >= N || mvalid == 0) continue;
                const int64_t idx = tl.pbase + n * M + mrow;
                float* g = ch.g + 4 * jj;
                if constexpr (OP == OP_DW) {
                    if (vec) {
                        StateIO<ST_F32>::st4(p.dW, idx, g);
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (i < mvalid) StateIO<ST_F32>::st(p.dW, idx + i, g[i]);
                    }
                } else {
                    float* w = ch.w + 4 * jj;
                    float* a = ch.a + 4 * jj;
                    float* bb = ch.b + 4 * jj;
                    step4<OP>(p, g, w, a, bb);
                    if (vec) {
                        StateIO<ST_F32>::st4(Wst, idx, w);
                        StateIO<ST>::st4(S1, idx, a);
                        if constexpr (OP == OP_ADAMW) StateIO<ST>::st4(S2, idx, bb);
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (i < mvalid) {
                                StateIO<ST_F32>::st(Wst, idx + i, w[i]);
                                StateIO<ST>::st(S1, idx + i, a[i]);
                                if constexpr (OP == OP_ADAMW) StateIO<ST>::st(S2, idx + i, bb[i]);
                            }
                    }
                }
            }
        };

        if (nchunks == 0) {
            if (has_acc) release();
        } else {
            // A chunk's gradient is read just before its update rather than
            // with its state loads: one chunk's gradient fewer live, which
            // keeps the sixteen-warp epilogue (96 registers) free of spills
            // and measured slightly faster with eight warps too.
            constexpr bool kLateGrad = true;
            auto fetch = [&](int c, Chunk& ch) {
                if constexpr (!kLateGrad) grad(c, ch);
                state(c, ch);
            };
            auto update = [&](int c, Chunk& ch) {
                if constexpr (kLateGrad) grad(c, ch);
                process(c, ch);
            };
            Chunk A, B;
            fetch(0, A);
#pragma unroll 1
            for (int c = 0; c < nchunks; c += 2) {
                if (c + 1 < nchunks) fetch(c + 1, B);
                update(c, A);
                if (c + 1 < nchunks) {
                    if (c + 2 < nchunks) fetch(c + 2, A);
                    update(c + 1, B);
                }
            }
        }
        if (has_acc) ++ct;
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
    }
}

// ------------------------------------------------------------------ grouped set-up

// Copies the expert offsets into shared memory, validates them and ranks the
// experts by token count (descending, ties by index) without atomics.  Every
// thread of the CTA calls it; it returns false for the whole CTA (after the
// first CTA records FORGE_ERR_INVALID_ARG) when the offsets are invalid.
__device__ __forceinline__ bool grouped_setup(const Params& p, int32_t* s_offs, int32_t* s_order,
                                              volatile int* s_bad)
{
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_offs[i] = p.offsets[i];
    if (threadIdx.x == 0) *s_bad = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        const int32_t a = s_offs[e], b = s_offs[e + 1];
        if (a < 0 || b < a || static_cast<int64_t>(b) > p.T_max) *s_bad = 1;
    }
    __syncthreads();
    if (*s_bad) {
        if (threadIdx.x == 0 && blockIdx.x == 0)
            *reinterpret_cast<volatile int*>(p.status) = kDevInvalidArg;
        return false;
    }
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        const int32_t ke = s_offs[e + 1] - s_offs[e];
        int32_t rank = 0;
        for (int f = 0; f < p.E; ++f) {
            const int32_t kf = s_offs[f + 1] - s_offs[f];
            rank += (kf > ke) || (kf == ke && f < e);
        }
        s_order[rank] = e;
    }
    return true;
}

// An expert's last k-block (grouped calls): rows [ky, ky + BK) of NBOX
// 128-byte column blocks from column mn0, of which the rows before kend
// belong to the expert.  Rows at or past kend must read as zeros in both
// operands, so that another expert's tokens never enter the product (not
// even as 0 x inf).  The whole MMA k-steps of UK rows come as k-step-high
// boxes, box(byte offset, column, row); the incomplete k-step four rows at a
// time through a one-row-box map, gather(byte offset, column, rows[4]), rows
// at or past kend given the out-of-range index oob (TMA writes zeros); the
// k-steps after it as boxes starting at oob, past the tensor's last row
// (zero filled).  The stage receives BK rows of bytes, as a full k-block.
// Gathering the whole block four rows at a time took 16 copies per column
// block and stalled the MMA issuer about 2.6 us on every tile.
template <int BK, int UK, int NBOX, int BOX_MN, int BOX_BYTES, class Box, class Gather>
__device__ __forceinline__ void partial_block(int32_t mn0, int32_t ky, int32_t kend, int32_t oob,
                                              Box&& box, Gather&& gather)
{
    static_assert(BK % UK == 0 && UK % 4 == 0, "k-steps of whole four-row gathers");
    const int32_t valid = kend - ky;
    const int32_t whole = valid / UK;
    const int32_t steps = (valid + UK - 1) / UK;
#pragma unroll 1
    for (int32_t j = 0; j < BK / UK; ++j) {
        if (j == whole && whole < steps) continue;  // gathered below
        const int32_t y = j < whole ? ky + j * UK : oob;
#pragma unroll
        for (int i = 0; i < NBOX; ++i) box(i * BOX_BYTES + j * UK * 128, mn0 + i * BOX_MN, y);
    }
    if (whole < steps) {
#pragma unroll 1
        for (int32_t r = whole * UK; r < steps * UK; r += 4) {
            int32_t y[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) y[j] = ky + r + j < kend ? ky + r + j : oob;
#pragma unroll
            for (int i = 0; i < NBOX; ++i) gather(i * BOX_BYTES + r * 128, mn0 + i * BOX_MN, y);
        }
    }
}

// ------------------------------------------------------------------ cp.async loader

constexpr int kLoaderWarp0 = 2;  // warps 2 and 3
constexpr int kLoaderThreads = 64;

// Copies one operand's k-block [k0, k0 + BK) x [mn0, mn0 + TILE_MN) into the
// same 128-byte-swizzled layout TMA would produce: column block `box` (128
// bytes of the contiguous dimension) at box * box_bytes, k row r at r * 128,
// 16-byte chunk c of the row at (c ^ (r & 7)) * 16.  Rows at or past k_lim
// and columns at or past mn_lim are zero-filled.  GRAN is the copy width in
// bytes (8 or 4); every division below is by a compile-time constant.
template <int IT, int TILE_MN, int GRAN>
__device__ __forceinline__ void load_block_cp_async(uint8_t* stage, const uint8_t* g, int64_t ld,
                                                    int64_t mn0, int64_t mn_lim, int64_t k0,
                                                    int64_t k_lim, int tid)
{
    using TR = InTraits<IT>;
    constexpr int BK = TR::BK;
    constexpr int es = TR::esize;
    constexpr int box_bytes = TR::box_mn * es * BK;
    constexpr int kUnitsPerRow = TILE_MN * es / GRAN;
    constexpr int kTotal = BK * kUnitsPerRow;
    static_assert(kTotal % kLoaderThreads == 0, "whole passes");
#pragma unroll 4
    for (int u = tid; u < kTotal; u += kLoaderThreads) {
        const int r = u / kUnitsPerRow;
        const int cb = (u - r * kUnitsPerRow) * GRAN;  // byte offset in the tile row
        uint8_t* d = stage + (cb >> 7) * box_bytes + r * 128 +
                     ((((cb & 127) >> 4) ^ (r & 7)) << 4) + (cb & 15);
        const int64_t k = k0 + r;
        const int64_t col = mn0 + cb / es;
        int src_bytes = 0;
        const uint8_t* src = g;
        if (k < k_lim && col < mn_lim) {
            const int64_t avail = (mn_lim - col) * es;
            src_bytes = avail >= GRAN ? GRAN : static_cast<int>(avail);
            src = g + (k * ld + col) * es;
        }
        ptx::cp_async(d, src, GRAN, src_bytes);
    }
}

template <int IT, int TILE_MN>
__device__ __forceinline__ void load_block_cp_async(uint8_t* stage, const uint8_t* g, int64_t ld,
                                                    int64_t mn0, int64_t mn_lim, int64_t k0,
                                                    int64_t k_lim, int gran, int tid)
{
    if (gran == 8)
        load_block_cp_async<IT, TILE_MN, 8>(stage, g, ld, mn0, mn_lim, k0, k_lim, tid);
    else
        load_block_cp_async<IT, TILE_MN, 4>(stage, g, ld, mn0, mn_lim, k0, k_lim, tid);
}

// ------------------------------------------------------------------ kernel

template <int IT, int OP, int ST, bool GROUPED, bool MANUAL>
__global__ void __launch_bounds__(EpiFor<GROUPED>::threads, 1)
    forge_wgrad_kernel(const __grid_constant__ CUtensorMap tmA,   // dY
                       const __grid_constant__ CUtensorMap tmB,   // X
                       const __grid_constant__ CUtensorMap tmA1,  // dY, one-row boxes (grouped)
                       const __grid_constant__ CUtensorMap tmB1,  // X, one-row boxes (grouped)
                       const __grid_constant__ CUtensorMap tmAk,  // dY, one-k-step boxes (grouped)
                       const __grid_constant__ CUtensorMap tmBk,  // X, one-k-step boxes (grouped)
                       const Params p)
{
    using TR = InTraits<IT>;
    constexpr int BK = TR::BK;
    constexpr int kBoxBytes = TR::box_mn * TR::esize * BK;  // one 128-byte-wide column block
    constexpr int kABoxes = BM / TR::box_mn;
    constexpr int kBBoxes = BN / TR::box_mn;
    constexpr int kKSteps = BK / TR::umma_k;
    constexpr uint32_t kKStepBytes = TR::umma_k * 128;  // umma_k rows of 128 bytes
    constexpr uint32_t kIdesc = ptx::make_idesc(TR::fmt, TR::fmt, true, true, BM, BN);
    static_assert(kABoxes * kBoxBytes == kStageA && kBBoxes * kBoxBytes == kStageB, "stage size");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SmemCta::bar);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int32_t* s_offs = reinterpret_cast<int32_t*>(smem + SmemCta::sched);
    int32_t* s_order = s_offs + (p.E + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // TMA producer's arrive (+ one arrive per cp.async loader thread)
            ptx::mbar_init(&full[s], 1 + (MANUAL ? kLoaderThreads : 0));
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&tfull[b], 1);
            ptx::mbar_init(&tempty[b], EpiFor<GROUPED>::warps);
        }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_mbarrier_init();
    }

    if constexpr (GROUPED) {
        if (!grouped_setup(p, s_offs, s_order, abort_flag + 1)) return;  // nothing allocated yet
    }

    if (warp == 0 && lane == 0 && p.has_maps) {
        if (!p.manual_a) ptx::prefetch_tensormap(&tmA);
        if (!p.manual_b) ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    Sched sc;
    sc.tiles_m = p.tiles_m;
    sc.tiles_n = p.tiles_n;
    sc.m_step = BM;
    sc.m_off = 0;
    sc.band = p.raster_band;
    sc.per_expert = p.tiles_m * p.tiles_n;
    sc.total = sc.per_expert * p.E;
    sc.set_share(blockIdx.x, gridDim.x, GROUPED ? 1 : 0);
    sc.offs = GROUPED ? s_offs : nullptr;
    sc.order = GROUPED ? s_order : nullptr;
    sc.multi = nullptr;
    sc.K = p.K;
    sc.MN = p.M * p.N;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            // dY (the smaller operand, reused by every wave of tiles) is kept
            // in L2; X column blocks are consumed within one wave.
            const uint64_t pol = ptx::policy_evict_last();
            const bool tma_a = !(MANUAL && p.manual_a);
            const bool tma_b = !(MANUAL && p.manual_b);
            const uint32_t tx_bytes = (tma_a ? kStageA : 0) + (tma_b ? kStageB : 0);
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_mask = 0, last_parity = 0;
            bool ok = true;
            for (int32_t it = 0; ok && it < sc.count; ++it) {
                const int32_t t = sc.nth(it);
                const Tile tl = sc.get(t);
                for (int64_t k = tl.k_begin; k < tl.k_end; k += BK) {
                    if (!wait_bounded(&empty[s], ph ^ 1u, abort_flag, p)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&full[s], tx_bytes);
                    uint8_t* sa = smem + s * kStageBytes;
                    uint8_t* sb = sa + kStageA;
                    const int32_t ky = static_cast<int32_t>(k);
                    const bool partial = GROUPED && tl.k_end - k < BK;
                    const int32_t kend = static_cast<int32_t>(tl.k_end);
                    const int32_t oob = static_cast<int32_t>(p.T_max);
                    if (tma_a) {
                        if (partial) {
                            partial_block<BK, TR::umma_k, kABoxes, TR::box_mn, kBoxBytes>(
                                tl.m0, ky, kend, oob,
                                [&](int off, int32_t x, int32_t y) {
                                    ptx::tma_load_2d(sa + off, &tmAk, &full[s], x, y);
                                },
                                [&](int off, int32_t x, const int32_t* y) {
                                    ptx::tma_gather4_2d(sa + off, &tmA1, &full[s], x, y[0], y[1],
                                                        y[2], y[3]);
                                });
                        } else {
#pragma unroll
                            for (int i = 0; i < kABoxes; ++i)
                                ptx::tma_load_2d_hint(sa + i * kBoxBytes, &tmA, &full[s],
                                                      tl.m0 + i * TR::box_mn, ky, pol);
                        }
                    }
                    if (tma_b) {
                        if (partial) {
                            partial_block<BK, TR::umma_k, kBBoxes, TR::box_mn, kBoxBytes>(
                                tl.n0, ky, kend, oob,
                                [&](int off, int32_t x, int32_t y) {
                                    ptx::tma_load_2d(sb + off, &tmBk, &full[s], x, y);
                                },
                                [&](int off, int32_t x, const int32_t* y) {
                                    ptx::tma_gather4_2d(sb + off, &tmB1, &full[s], x, y[0], y[1],
                                                        y[2], y[3]);
                                });
                        } else {
#pragma unroll
                            for (int i = 0; i < kBBoxes; ++i)
                                ptx::tma_load_2d(sb + i * kBoxBytes, &tmB, &full[s],
                                                 tl.n0 + i * TR::box_mn, ky);
                        }
                    }
                    issued_mask |= 1u << s;
                    last_parity = (last_parity & ~(1u << s)) | (ph << s);
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Wait (bounded) for this thread's copies still in flight.
                const uint64_t t0 = ptx::globaltimer_ns();
                for (int q = 0; q < kStages; ++q) {
                    if (!(issued_mask & (1u << q))) continue;
                    const uint32_t a = ptx::smem_addr(&full[q]);
                    while (!ptx::mbar_try_wait(a, (last_parity >> q) & 1u)) {
                        if (static_cast<int64_t>(ptx::globaltimer_ns() - t0) > p.timeout_ns)
                            break;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- UMMA issuer
        // Lane 0 alone waits on the barriers and issues the MMAs: a
        // warp-wide loop would add a warp synchronisation to every stage and
        // keep the issuer from running ahead of the tensor pipe.
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t ct = 0;  // accumulator tiles issued by this CTA
            bool ok = true;
            bool issued_any = false;
            for (int32_t it = 0; ok && it < sc.count; ++it) {
                const int32_t t = sc.nth(it);
                const Tile tl = sc.get(t);
                if (tl.k_end <= tl.k_begin) continue;  // no tokens: epilogue-only tile
                const uint32_t b = ct & 1u;
                const uint32_t aph = (ct >> 1) & 1u;
                ok = wait_bounded(&tempty[b], aph ^ 1u, abort_flag, p);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * BN;
                uint32_t first = 1;
                for (int64_t k = tl.k_begin; k < tl.k_end; k += BK) {
                    ok = wait_bounded(&full[s], ph, abort_flag, p);
                    if (!ok) break;
                    const uint32_t sa = ptx::smem_addr(smem + s * kStageBytes);
                    const uint32_t sb = sa + kStageA;
#pragma unroll
                    for (int ks = 0; ks < kKSteps; ++ks) {
                        const uint64_t ad =
                            ptx::smem_desc_sw128(sa + ks * kKStepBytes, kBoxBytes, 1024);
                        const uint64_t bd =
                            ptx::smem_desc_sw128(sb + ks * kKStepBytes, kBoxBytes, 1024);
                        if constexpr (IT == IN_BF16)
                            ptx::umma_f16(d_tmem, ad, bd, kIdesc, first ? 0u : 1u);
                        else
                            ptx::umma_f8(d_tmem, ad, bd, kIdesc, first ? 0u : 1u);
                        first = 0;
                    }
                    ptx::umma_commit(&empty[s]);  // stage free once these MMAs are done
                    issued_any = true;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::umma_commit(&tfull[b]);  // accumulator ready
                ++ct;
            }
            if (!ok && issued_any) {
                // Wait (bounded) until every MMA this thread issued is done.
                ptx::umma_commit(drain);
                const uint32_t a = ptx::smem_addr(drain);
                const uint64_t t0 = ptx::globaltimer_ns();
                while (!ptx::mbar_try_wait(a, 0)) {
                    if (static_cast<int64_t>(ptx::globaltimer_ns() - t0) > p.timeout_ns) break;
                }
            }
        }
    } else if (MANUAL && (warp == kLoaderWarp0 || warp == kLoaderWarp0 + 1)) {
        // ---------------------------------------------------- cp.async loader
        // Fills the operands TMA cannot address.  Each thread keeps up to
        // kLag stages of its copies in flight; a stage is announced (proxy
        // fence, then an arrive on its full barrier) once its copies are
        // complete: when more than kLag are outstanding, and all of them
        // whenever the next slot is not free yet, so no announcement waits
        // on the MMA.
        constexpr int kLag = kStages - 1;
        const int tid = threadIdx.x - kLoaderWarp0 * 32;
        int s = 0;
        uint32_t ph = 0;
        int npend = 0;  // stages issued but not yet announced, oldest first
        bool ok = true;
        for (int32_t it = 0; ok && it < sc.count; ++it) {
            const int32_t t = sc.nth(it);
            const Tile tl = sc.get(t);
            for (int64_t k = tl.k_begin; k < tl.k_end; k += BK) {
                // Announce every pending stage before blocking on a busy slot.
                if (npend > 0 && !ptx::mbar_test_wait(ptx::smem_addr(&empty[s]), ph ^ 1u)) {
                    ptx::cp_async_wait<0>();
                    ptx::fence_proxy_async_smem();
                    for (; npend > 0; --npend)
                        ptx::mbar_arrive(&full[(s - npend + kStages) % kStages]);
                }
                ok = warp_wait(&empty[s], ph ^ 1u, abort_flag, p, lane);
                if (!ok) break;
                uint8_t* sa = smem + s * kStageBytes;
                if (p.manual_a)
                    load_block_cp_async<IT, BM>(sa, p.gA, p.M, tl.m0, p.M, k, tl.k_end, p.gran_a,
                                                tid);
                if (p.manual_b)
                    load_block_cp_async<IT, BN>(sa + kStageA, p.gB, p.N, tl.n0, p.N, k, tl.k_end,
                                                p.gran_b, tid);
                ptx::cp_async_commit();
                if (++npend > kLag) {
                    ptx::cp_async_wait<kLag>();
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(&full[(s - kLag + kStages) % kStages]);
                    --npend;
                }
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        ptx::cp_async_wait<0>();
        if (ok) {
            ptx::fence_proxy_async_smem();
            for (; npend > 0; --npend) ptx::mbar_arrive(&full[(s - npend + kStages) % kStages]);
        }
    } else if (warp >= kEpiWarp0) {
        epilogue_role<IT, OP, ST, EpiFor<GROUPED>>(
            p, sc, tfull, tmem_base, abort_flag, warp, lane,
            [&](uint32_t b) { ptx::mbar_arrive(&tempty[b]); });
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------ CTA-pair kernel

// CTA-pair form (dense, and grouped with one expert per tile).  A pair owns a
// 256 (m) x 256 (n) tile: CTA r of
// the pair loads the 128 rows m0 + 128 r .. of dY and the 128 columns
// n0 + 128 r .. of X, and the even CTA issues tcgen05.mma.cta_group::2, which
// reads the A half of each CTA and both B halves and leaves each CTA's 128 x
// 256 fp32 result in its own TMEM.  A stage is therefore 32 KB per CTA
// instead of 48 KB, so six stages fit where four did and each SM pulls a
// third fewer operand bytes through L2 per MMA.  Each CTA runs the same
// epilogue on its own 128 rows.  Every operand byte a CTA receives comes
// from this GPU's memory through a plain (non-multicast) TMA load.
//
// Synchronisation:
//   full[s]   (even CTA)  its producer expects the 64 KB landing in the pair;
//                         every load into the pair completes on it
//   empty[s]  (each CTA)  the pair's MMA commit arrives in both CTAs
//   tfull[b]  (each CTA)  the pair's MMA commit, when accumulator b is complete
//   tempty[b] (even CTA)  all epilogue warps of the pair arrive (the odd
//                         CTA's remotely) once accumulator b has been read
constexpr int kPairStageA = 16384;  // this CTA's 128 rows of dY x BK
constexpr int kPairStageB = 16384;  // this CTA's 128 columns of X x BK
constexpr int kPairStageBytes = kPairStageA + kPairStageB;
#ifndef FORGE_GROUPED_PAIR_STAGES
#define FORGE_GROUPED_PAIR_STAGES 6
#endif
// Operand stages per CTA: dense and multi-problem calls six (the 196 KB
// carve-out step, a 60 KB L1); grouped calls FORGE_GROUPED_PAIR_STAGES
// (compile time).  The ring and L1 share the SM's 256 KB: the ring covers the
// operand loads' latency, L1 holds the epilogue's state loads in flight.
template <bool GROUPED>
struct PairRing {
    static constexpr int stages = GROUPED ? FORGE_GROUPED_PAIR_STAGES : 6;
    using Smem = SmemLayout<stages * kPairStageBytes>;
};
static_assert(PairRing<false>::Smem::alloc(kCarveoutExperts) + 1024 <= kCarveout196,
              "196 KB step");
static_assert(PairRing<true>::stages >= 4 &&
                  PairRing<true>::Smem::alloc(8) + 1024 <= kSmemPerCtaMax,
              "grouped ring and an eight-expert table within one CTA's shared memory");

template <int IT, int OP, int ST, bool GROUPED, bool MULTI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(EpiFor<GROUPED>::threads, 1)
    forge_wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA,   // dY
                            const __grid_constant__ CUtensorMap tmB,   // X
                            const __grid_constant__ CUtensorMap tmA1,  // dY, one-row boxes (grouped)
                            const __grid_constant__ CUtensorMap tmB1,  // X, one-row boxes (grouped)
                            const __grid_constant__ CUtensorMap tmAk,  // dY, one-k-step boxes (grouped)
                            const __grid_constant__ CUtensorMap tmBk,  // X, one-k-step boxes (grouped)
                            const __grid_constant__ MultiMaps mm,      // dY of each problem (multi)
                            const __grid_constant__ Params p)
{
    static_assert(!MULTI || !GROUPED, "multi-problem calls are dense");
    static_assert(InTraits<IT>::BK == 4 * InTraits<IT>::umma_k,
                  "the one-k-step maps hold a quarter of a k-block");
    using TR = InTraits<IT>;
    constexpr int BK = TR::BK;
    constexpr int kBoxBytes = TR::box_mn * TR::esize * BK;
    constexpr int kABoxes = BM / TR::box_mn;
    constexpr int kBBoxes = (BN / 2) / TR::box_mn;
    constexpr int kKSteps = BK / TR::umma_k;
    constexpr uint32_t kKStepBytes = TR::umma_k * 128;
    constexpr uint32_t kIdesc = ptx::make_idesc(TR::fmt, TR::fmt, true, true, 2 * BM, BN);
    static_assert(kABoxes * kBoxBytes == kPairStageA && kBBoxes * kBoxBytes == kPairStageB,
                  "stage size");

    constexpr int kPairStages = PairRing<GROUPED>::stages;
    using SmemPair = typename PairRing<GROUPED>::Smem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SmemPair::bar);
    uint64_t* empty = full + kPairStages;
    uint64_t* tfull = empty + kPairStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int32_t* s_offs = reinterpret_cast<int32_t*>(smem + SmemPair::sched);
    int32_t* s_order = s_offs + (p.E + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = ptx::cluster_ctarank();  // position in the pair
    const bool leader = crank == 0;                 // the pair's even CTA
    constexpr uint16_t kPairMask = 0x3;             // both CTAs of the pair

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&tfull[b], 1);
            ptx::mbar_init(&tempty[b], 2 * EpiFor<GROUPED>::warps);
        }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_mbarrier_init();
    }
    if constexpr (GROUPED) {
        // both CTAs of a pair read the same offsets, so they return together
        if (!grouped_setup(p, s_offs, s_order, abort_flag + 1)) return;
    }
    if (warp == 0 && lane == 0 && p.has_maps) {
        if constexpr (MULTI) {
            for (int j = 0; j < p.P; ++j) ptx::prefetch_tensormap(&mm.a[j]);
        } else {
            ptx::prefetch_tensormap(&tmA);
        }
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(tmem_slot, kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();  // all barriers of the cluster initialised, TMEM allocated
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    Sched sc;
    sc.tiles_m = p.tiles_m;  // 256-row tiles
    sc.tiles_n = p.tiles_n;
    sc.m_step = 2 * BM;
    sc.m_off = static_cast<int32_t>(crank) * BM;
    sc.band = p.raster_band;
    sc.per_expert = p.tiles_m * p.tiles_n;
    sc.total = MULTI ? pick(p.tile_begin, p.P) : sc.per_expert * p.E;
    sc.set_share(blockIdx.x / 2, gridDim.x / 2, GROUPED ? 1 : 0);
    sc.offs = GROUPED ? s_offs : nullptr;
    sc.order = GROUPED ? s_order : nullptr;
    sc.multi = MULTI ? &p : nullptr;
    sc.K = p.K;
    sc.MN = p.M * p.N;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer (both CTAs)
        if (lane == 0) {
            const uint64_t pol = ptx::policy_evict_last();
            const uint32_t full0 = ptx::mapa_shared(ptx::smem_addr(&full[0]), 0);
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_mask = 0, last_parity = 0;
            bool ok = true;
            for (int32_t it = 0; ok && it < sc.count; ++it) {
                const int32_t t = sc.nth(it);
                const Tile tl = sc.get(t);
                for (int64_t k = tl.k_begin; k < tl.k_end; k += BK) {
                    if (!wait_bounded(&empty[s], ph ^ 1u, abort_flag, p)) {
                        ok = false;
                        break;
                    }
                    if (leader) ptx::mbar_arrive_expect_tx(&full[s], 2 * kPairStageBytes);
                    uint8_t* sa = smem + s * kPairStageBytes;
                    uint8_t* sb = sa + kPairStageA;
                    const uint32_t bar = full0 + s * 8;
                    const int32_t ky = static_cast<int32_t>(k);
                    const int32_t nb = tl.n0 + static_cast<int32_t>(crank) * (BN / 2);
                    if (GROUPED && tl.k_end - k < BK) {
                        // the expert's last k-block: rows past its end read as zeros
                        const int32_t kend = static_cast<int32_t>(tl.k_end);
                        const int32_t oob = static_cast<int32_t>(p.T_max);
                        partial_block<BK, TR::umma_k, kABoxes, TR::box_mn, kBoxBytes>(
                            tl.m0, ky, kend, oob,
                            [&](int off, int32_t x, int32_t y) {
                                ptx::tma_load_2d_pair(sa + off, &tmAk, bar, x, y);
                            },
                            [&](int off, int32_t x, const int32_t* y) {
                                ptx::tma_gather4_2d_pair(sa + off, &tmA1, bar, x, y[0], y[1],
                                                         y[2], y[3]);
                            });
                        partial_block<BK, TR::umma_k, kBBoxes, TR::box_mn, kBoxBytes>(
                            nb, ky, kend, oob,
                            [&](int off, int32_t x, int32_t y) {
                                ptx::tma_load_2d_pair(sb + off, &tmBk, bar, x, y);
                            },
                            [&](int off, int32_t x, const int32_t* y) {
                                ptx::tma_gather4_2d_pair(sb + off, &tmB1, bar, x, y[0], y[1],
                                                         y[2], y[3]);
                            });
                    } else {
                        // dY's map: the call's, or the tile's problem's
                        const CUtensorMap* mapA = &tmA;
                        if constexpr (MULTI) {
#pragma unroll
                            for (int j = 0; j < kMaxProblems; ++j)
                                if (tl.prob == j) mapA = &mm.a[j];
                        }
#pragma unroll
                        for (int i = 0; i < kABoxes; ++i)
                            ptx::tma_load_2d_pair_hint(sa + i * kBoxBytes, mapA, bar,
                                                       tl.m0 + i * TR::box_mn, ky, pol);
#pragma unroll
                        for (int i = 0; i < kBBoxes; ++i)
                            ptx::tma_load_2d_pair(sb + i * kBoxBytes, &tmB, bar,
                                                  nb + i * TR::box_mn, ky);
                    }
                    issued_mask |= 1u << s;
                    last_parity = (last_parity & ~(1u << s)) | (ph << s);
                    if (++s == kPairStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok && leader) {
                // Wait (bounded) for the pair's copies still in flight: they
                // all complete on the even CTA's full barriers.
                const uint64_t t0 = ptx::globaltimer_ns();
                for (int q = 0; q < kPairStages; ++q) {
                    if (!(issued_mask & (1u << q))) continue;
                    const uint32_t a = ptx::smem_addr(&full[q]);
                    while (!ptx::mbar_try_wait(a, (last_parity >> q) & 1u)) {
                        if (static_cast<int64_t>(ptx::globaltimer_ns() - t0) > p.timeout_ns) break;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- pair MMA issuer (even CTA)
        // Lane 0 alone waits and issues (no warp synchronisation per stage).
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t ct = 0;
            bool ok = true;
            bool issued_any = false;
            for (int32_t it = 0; ok && it < sc.count; ++it) {
                const int32_t t = sc.nth(it);
                const Tile tl = sc.get(t);
                if (tl.k_end <= tl.k_begin) continue;
                const uint32_t b = ct & 1u;
                const uint32_t aph = (ct >> 1) & 1u;
                ok = wait_bounded(&tempty[b], aph ^ 1u, abort_flag, p);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * BN;
                uint32_t first = 1;
                for (int64_t k = tl.k_begin; k < tl.k_end; k += BK) {
                    ok = wait_bounded(&full[s], ph, abort_flag, p);
                    if (!ok) break;
                    const uint32_t sa = ptx::smem_addr(smem + s * kPairStageBytes);
                    const uint32_t sb = sa + kPairStageA;
#pragma unroll
                    for (int ks = 0; ks < kKSteps; ++ks) {
                        const uint64_t ad =
                            ptx::smem_desc_sw128(sa + ks * kKStepBytes, kBoxBytes, 1024);
                        const uint64_t bd =
                            ptx::smem_desc_sw128(sb + ks * kKStepBytes, kBoxBytes, 1024);
                        if constexpr (IT == IN_BF16)
                            ptx::umma_f16_pair(d_tmem, ad, bd, kIdesc, first ? 0u : 1u);
                        else
                            ptx::umma_f8_pair(d_tmem, ad, bd, kIdesc, first ? 0u : 1u);
                        first = 0;
                    }
                    // stage s of both CTAs is free once these MMAs are done
                    ptx::umma_commit_pair(&empty[s], kPairMask);
                    issued_any = true;
                    if (++s == kPairStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::umma_commit_pair(&tfull[b], kPairMask);  // both accumulators ready
                ++ct;
            }
            if (!ok && issued_any) {
                ptx::umma_commit_pair(drain, static_cast<uint16_t>(1u << crank));
                const uint32_t a = ptx::smem_addr(drain);
                const uint64_t t0 = ptx::globaltimer_ns();
                while (!ptx::mbar_try_wait(a, 0)) {
                    if (static_cast<int64_t>(ptx::globaltimer_ns() - t0) > p.timeout_ns) break;
                }
            }
        }
    } else if (warp >= kEpiWarp0) {
        const uint32_t tempty0 = ptx::mapa_shared(ptx::smem_addr(&tempty[0]), 0);
        epilogue_role<IT, OP, ST, EpiFor<GROUPED>, MULTI>(
            p, sc, tfull, tmem_base, abort_flag, warp, lane, [&](uint32_t b) {
                                      if (leader)
                                          ptx::mbar_arrive(&tempty[b]);
                                      else
                                          ptx::mbar_arrive_cluster(tempty0 + 8 * b);
                                  });
    }

    ptx::tc_fence_before();
    ptx::cluster_sync();  // no CTA leaves while another may still signal it
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

}  // namespace forge
