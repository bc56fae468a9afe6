// forge_api.cu -- the C ABI of libforge.so: argument validation, device
// checks, TMA descriptor encoding, tile-grid sizing and kernel dispatch.
//
// The checks on the arguments' values run before the first CUDA call, so
// such calls fail with a status code even on a machine without a GPU; the
// device, residency and alignment checks follow, all before any launch.  The
// device memory the library owns for the life of the process is the status
// word below (once per device) and, once forge_wgrad_adamw_noalloc has run on
// a device, its fixed staging buffer; the one per-call allocation is the
// staging copy of an operand whose rows TMA cannot address (stream-ordered,
// from the library's memory pool, freed on the same stream after the kernel).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "forge.h"
#include "forge_device.h"
#include "forge_launch.cuh"
#include "forge_static_stage.h"

namespace {

using namespace forge;

constexpr int kMaxDevices = 64;
constexpr int32_t kDefaultRasterBand = 8;  // d_out tiles per raster band (dense and grouped calls)

// Device status word: 0, or the first device-side error since the last read.
__device__ int g_forge_status = 0;

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int ordinal = -1;
    int sms = 0;
    int* status = nullptr;  // device address of g_forge_status on this device
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int64_t wait_timeout_ns()
{
    static const int64_t v = [] {
        const char* s = std::getenv("FORGE_WAIT_TIMEOUT_MS");
        long long ms = s ? std::atoll(s) : 10000;
        if (ms <= 0) ms = 10000;
        return static_cast<int64_t>(ms) * 1000000;
    }();
    return v;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool finite_nonneg(float x) { return std::isfinite(x) && x >= 0.0f; }

int elem_size(forge_dtype t) { return t == FORGE_BF16 ? 2 : (t == FORGE_E4M3 ? 1 : 4); }

// Resolves the current device and caches its properties.  The first call on
// a device also resolves the address of the status word there.
forge_status current_device(DeviceInfo** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return FORGE_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return FORGE_ERR_UNSUPPORTED_DEVICE;
        }
        d.supported = (major == 10 && minor == 3);
        d.ordinal = dev;
        d.sms = sms;
        if (d.supported) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_forge_status) != cudaSuccess) {
                cudaGetLastError();
                return FORGE_ERR_CUDA;
            }
            d.status = static_cast<int*>(addr);
        }
        d.ready = true;
    }
    if (!d.supported) return FORGE_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return FORGE_OK;
}

// 2-D token-major operand [rows, inner] with a row stride of ld_bytes (a
// multiple of 16) -> TMA map with 128-byte swizzled boxes of (128 bytes of
// the inner dimension) x (k rows per stage / row_split).  row_split = 0 asks
// for one-row boxes, the form tile::gather4 copies use.
// Resolves cuTensorMapEncodeTiled through the runtime once per process.
bool ensure_encode()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return g_encode != nullptr;
}

forge_status encode_operand(CUtensorMap* map, const void* base, forge_dtype dt, int64_t inner,
                            int64_t rows, int64_t ld_bytes, int row_split = 1)
{
    if (!ensure_encode()) return FORGE_ERR_CUDA;
    const int es = elem_size(dt);
    const cuuint32_t box_inner = 128 / es;
    const cuuint32_t box_rows =
        row_split == 0 ? 1
                       : (dt == FORGE_BF16 ? InTraits<IN_BF16>::BK : InTraits<IN_E4M3>::BK) /
                             row_split;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_bytes)};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType t =
        dt == FORGE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = g_encode(map, t, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FORGE_OK : FORGE_ERR_CUDA;
}

// Failure-detection self-test: wait on a barrier no one arrives at.
__global__ void forge_wait_selftest_kernel(int64_t timeout_ns, int* status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        Params p{};
        p.timeout_ns = timeout_ns;
        p.status = status;
        (void)wait_bounded(&bar, 0, &abort_flag, p);
    }
}

forge_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FORGE_OK : FORGE_ERR_CUDA; }

// Every pointer a call dereferences must be device memory (cudaMalloc, a
// memory pool, a virtual-memory mapping) of the current device: TMA and the
// epilogue address it directly, and host memory or a peer GPU's memory would
// be reached over the wrong link or not at all.  Null entries are skipped.
forge_status check_resident(int ordinal, const void* const* ptrs, int n)
{
    for (int i = 0; i < n; ++i) {
        if (!ptrs[i]) continue;
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, ptrs[i]) != cudaSuccess) {
            cudaGetLastError();
            return FORGE_ERR_INVALID_ARG;
        }
        if (a.type != cudaMemoryTypeDevice || a.device != ordinal) return FORGE_ERR_INVALID_ARG;
    }
    return FORGE_OK;
}

// ------------------------------------------------------------------ operand staging

// Rows whose base or length is not a multiple of 4 bytes (odd bf16 widths,
// e4m3 widths not divisible by 4): each thread builds one 4-byte word of a
// destination row from the one or two aligned source words that hold its
// bytes (a funnel shift).  A source word is read only if it holds at least
// one byte of the tensor, so no read leaves the memory pages the tensor
// touches.  Bytes of the last word past the row's end land in the
// destination row's padding, which the tensor map never reads.
__global__ void __launch_bounds__(256) forge_stage_bytes_kernel(const uint8_t* __restrict__ src,
                                                                uint32_t* __restrict__ dst,
                                                                int64_t rows, int64_t row_bytes,
                                                                int64_t dst_row_words)
{
    // flattened over the destination words of all rows, four in flight per
    // thread: word i is word i % words of row i / words
    const int64_t words = (row_bytes + 3) / 4;
    const int64_t total = rows * words;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < total;
         i0 += 4 * stride) {
        uint32_t v[4];
        int64_t at[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t i = i0 + j * stride;
            at[j] = -1;
            if (i >= total) continue;
            const int64_t r = i / words;
            const int64_t w = i - r * words;
            const int64_t nv = row_bytes - 4 * w < 4 ? row_bytes - 4 * w : 4;
            const uintptr_t first = reinterpret_cast<uintptr_t>(src + r * row_bytes + 4 * w);
            const uintptr_t lo_word = first & ~static_cast<uintptr_t>(3);
            const uintptr_t hi_word = (first + nv - 1) & ~static_cast<uintptr_t>(3);
            const uint32_t* a = reinterpret_cast<const uint32_t*>(lo_word);
            const uint32_t lo = __ldcs(a);
            const uint32_t hi = hi_word != lo_word ? __ldcs(a + 1) : 0u;
            v[j] = __funnelshift_r(lo, hi, static_cast<uint32_t>(8 * (first & 3)));
            at[j] = r * dst_row_words + w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (at[j] >= 0) dst[at[j]] = v[j];
    }
}

// Rows of 8- or 4-byte granularity (base and length), flattened over the
// destination's 16-byte chunks: thread i of the grid builds chunk i (row
// i / chunks_per_row) from the 16 / sizeof(U) source units it covers and
// stores it as one 16-byte vector, four chunks in flight per thread, so a
// row boundary costs no extra memory round trip.  Units past a row's end
// are not read; the chunk's bytes there land in the row's padding.
template <typename U>
__global__ void __launch_bounds__(256) forge_stage_chunks_kernel(const U* __restrict__ src,
                                                                 uint4* __restrict__ dst,
                                                                 int64_t rows, int64_t units,
                                                                 int64_t dst_chunks)
{
    constexpr int kPer = 16 / sizeof(U);  // source units per destination chunk
    const int64_t per_row = (units + kPer - 1) / kPer;
    const int64_t total = rows * per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < total;
         i0 += 4 * stride) {
        uint4 v[4];
        int64_t at[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t i = i0 + j * stride;
            at[j] = -1;
            if (i >= total) continue;
            const int64_t r = i / per_row;
            const int64_t c = i - r * per_row;
            const U* sp = src + r * units + c * kPer;
            U t[kPer];
#pragma unroll
            for (int k = 0; k < kPer; ++k) t[k] = c * kPer + k < units ? __ldcs(sp + k) : U{};
            v[j] = *reinterpret_cast<const uint4*>(t);
            at[j] = r * dst_chunks + c;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (at[j] >= 0) dst[at[j]] = v[j];
    }
}

// Stages [rows, row_bytes] (base and stride aligned to `gran` = 8, 4, 2 or 1
// bytes) into dst (256-byte aligned) with a row stride of dst_row_bytes (a
// multiple of 16).
cudaError_t stage_rows(const void* src, void* dst, int64_t rows, int64_t row_bytes,
                       int64_t dst_row_bytes, int gran, int sms, cudaStream_t stream)
{
    if (gran < 4) {
        const int64_t words = rows * ((row_bytes + 3) / 4);
        const int64_t want = (words + 4LL * 256 - 1) / (4LL * 256);
        const int wblocks = static_cast<int>(want < 8LL * sms ? want : 8LL * sms);
        forge_stage_bytes_kernel<<<wblocks, 256, 0, stream>>>(static_cast<const uint8_t*>(src),
                                                              static_cast<uint32_t*>(dst), rows,
                                                              row_bytes, dst_row_bytes / 4);
    } else {
        const int64_t chunks = rows * ((row_bytes + 15) / 16);
        const int64_t want = (chunks + 4LL * 256 - 1) / (4LL * 256);
        const int cblocks = static_cast<int>(want < 8LL * sms ? want : 8LL * sms);
        if (gran == 8)
            forge_stage_chunks_kernel<uint2><<<cblocks, 256, 0, stream>>>(
                static_cast<const uint2*>(src), static_cast<uint4*>(dst), rows, row_bytes / 8,
                dst_row_bytes / 16);
        else
            forge_stage_chunks_kernel<uint32_t><<<cblocks, 256, 0, stream>>>(
                static_cast<const uint32_t*>(src), static_cast<uint4*>(dst), rows,
                row_bytes / 4, dst_row_bytes / 16);
    }
    return cudaGetLastError();
}

// Operands whose rows TMA cannot address are either staged into a padded
// copy (default) or fetched by the kernel's cp.async loader.
// FORGE_MISALIGNED = loader | stage (read on every call) overrides; rows
// that are not a multiple of 4 bytes are staged either way (cp.async copies
// 4, 8 or 16 bytes).
bool stage_misaligned()
{
    const char* e = std::getenv("FORGE_MISALIGNED");
    return !(e && std::strcmp(e, "loader") == 0);
}

// The four operand maps of one call: dY and X with whole k-block boxes, and
// (grouped calls) the same tensors with one-row boxes for gathered blocks.
// The problem table's maps of a call that is not a multi-problem call.
const MultiMaps kNoProblemMaps = {};

struct Maps {
    CUtensorMap a, b;    // boxes of one k-block (BK token rows)
    CUtensorMap a1, b1;  // grouped: one-row boxes (four-row gathers)
    CUtensorMap ak, bk;  // grouped: boxes of one MMA k-step (an expert's last k-block)
};

template <int IT, bool MAN>
cudaError_t dispatch_op(int op, int st, bool grouped, const Maps& m, const Params& p, int grid,
                        cudaStream_t s)
{
#define FORGE_L(OPV, STV, G) \
    launch_wgrad<IT, OPV, STV, G, MAN>(m.a, m.b, m.a1, m.b1, m.ak, m.bk, p, grid, s)
    if (grouped)
        return st == ST_F32 ? FORGE_L(OP_ADAMW, ST_F32, true) : FORGE_L(OP_ADAMW, ST_BF16, true);
    switch (op) {
    case OP_ADAMW:
        return st == ST_F32 ? FORGE_L(OP_ADAMW, ST_F32, false) : FORGE_L(OP_ADAMW, ST_BF16, false);
    case OP_SGDM:
        return st == ST_F32 ? FORGE_L(OP_SGDM, ST_F32, false) : FORGE_L(OP_SGDM, ST_BF16, false);
    default:
        return FORGE_L(OP_DW, ST_F32, false);
    }
#undef FORGE_L
}

template <int IT>
cudaError_t dispatch_pair(int op, int st, bool grouped, const Maps& m, const Params& p,
                          int64_t grid, cudaStream_t s)
{
#define FORGE_L(OPV, STV, G)                                                   \
    launch_wgrad_pair<IT, OPV, STV, G, false>(m.a, m.b, m.a1, m.b1, m.ak, m.bk, \
                                              kNoProblemMaps, p, grid, s)
    if (grouped)
        return st == ST_F32 ? FORGE_L(OP_ADAMW, ST_F32, true) : FORGE_L(OP_ADAMW, ST_BF16, true);
    switch (op) {
    case OP_ADAMW:
        return st == ST_F32 ? FORGE_L(OP_ADAMW, ST_F32, false) : FORGE_L(OP_ADAMW, ST_BF16, false);
    case OP_SGDM:
        return st == ST_F32 ? FORGE_L(OP_SGDM, ST_F32, false) : FORGE_L(OP_SGDM, ST_BF16, false);
    default:
        return FORGE_L(OP_DW, ST_F32, false);
    }
#undef FORGE_L
}

// Kernel form: 0 = one CTA per 128 x 256 tile; 1 = CTA pairs on 256 x 256
// tiles.  Pairs serve calls whose operands TMA can address and whose d_out
// exceeds 128, dense or grouped.  FORGE_KERNEL = single | pair (read on every
// call) overrides the automatic choice where that form applies.
int kernel_form(const Params& p, bool manual)
{
    if (manual) return 0;
    const char* e = std::getenv("FORGE_KERNEL");
    if (e && std::strcmp(e, "single") == 0) return 0;
    if (e && std::strcmp(e, "pair") == 0) return 1;
    return p.M > BM ? 1 : 0;
}

// d_out tiles per raster band.  FORGE_RASTER_BAND (read on every call)
// overrides `default_band`; 0 or a value >= tiles_m means plain d_out-fastest.
// A wave of tiles in a band of 8 d_out tiles reads fewer dY column blocks,
// which then stay in L2 for the band's later waves: the fp8 workload (K 32768,
// 32 tile rows, 8 MB blocks) ran 3.5% faster than in plain order, the grouped
// MoE layer 1.9%, the MLP down-projection 0.3%; bands of 4 were slower again.
// The multi-problem attention launch measured no gain and keeps plain order.
int32_t raster_band(int32_t tiles_m, int32_t default_band)
{
    int32_t band = default_band;
    if (const char* e = std::getenv("FORGE_RASTER_BAND")) band = std::atoi(e);
    if (band <= 0 || band > tiles_m) band = tiles_m;
    return band;
}

// How an operand [rows, ld] of elemsize es reaches shared memory: 0 = TMA
// (16-byte aligned base and row stride), 8 or 4 = staged or fetched by
// cp.async of that width (base and row stride aligned to it), 2 or 1 =
// staged (base aligned to the element), -1 = a base not aligned to its
// element size.
int operand_path(const void* base, int64_t ld, int es)
{
    const int64_t row = ld * es;
    if (aligned(base, 16) && row % 16 == 0) return 0;
    if (aligned(base, 8) && row % 8 == 0) return 8;
    if (aligned(base, 4) && row % 4 == 0) return 4;
    if (aligned(base, static_cast<uintptr_t>(es))) return es;
    return -1;
}

// Where a staging copy lives: a stream-ordered allocation from the library's
// memory pool, or the fixed per-device buffer of the no-allocation entry.
enum class StageFrom { Pool, Static };

// Shared tail of every entry point, after the argument checks.
//   rows: K (dense) or T_max (grouped) -- the rows of X and dY.
forge_status run(const void* X, const void* dY, int64_t rows, forge_dtype in_dtype, int op,
                 forge_dtype state_dtype, bool grouped, Params p, cudaStream_t stream,
                 StageFrom stage_from = StageFrom::Pool)
{
    DeviceInfo* dev = nullptr;
    forge_status st = current_device(&dev);
    if (st != FORGE_OK) return st;
    {
        const void* ptrs[] = {rows > 0 ? X : nullptr, rows > 0 ? dY : nullptr, p.W, p.s1,
                              p.s2, p.dW, p.scales, p.offsets};
        if ((st = check_resident(dev->ordinal, ptrs, 8)) != FORGE_OK) return st;
    }

    // the tile list of the smallest tiles must be indexable in 32 bits
    if (((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN) * p.E > INT32_MAX)
        return FORGE_ERR_INVALID_ARG;

    const int es = elem_size(in_dtype);
    if (rows > 0) {
        const int path_a = operand_path(dY, p.M, es);
        const int path_b = operand_path(X, p.N, es);
        if (path_a < 0 || path_b < 0) return FORGE_ERR_MISALIGNED;
        p.manual_a = path_a > 0;
        p.manual_b = path_b > 0;
        p.gran_a = path_a;
        p.gran_b = path_b;
        p.gA = static_cast<const uint8_t*>(dY);
        p.gB = static_cast<const uint8_t*>(X);
    }
    const uintptr_t sa = state_dtype == FORGE_BF16 ? 2 : 4;
    if (!aligned(p.W, 4) || (p.s1 && !aligned(p.s1, sa)) || (p.s2 && !aligned(p.s2, sa)) ||
        (p.dW && !aligned(p.dW, 4)))
        return FORGE_ERR_MISALIGNED;

    // 4-element vector access in the epilogue: rows of whole vectors and
    // vector-aligned bases (16 bytes for fp32, 8 bytes for bf16 state)
    const uintptr_t va = state_dtype == FORGE_BF16 ? 8 : 16;
    p.vec_ok = (p.M % 4 == 0) && aligned(p.W, 16) && (!p.s1 || aligned(p.s1, va)) &&
                       (!p.s2 || aligned(p.s2, va)) && (!p.dW || aligned(p.dW, 16))
                   ? 1
                   : 0;

    // Operands TMA cannot address: a padded staging copy with 16-byte rows
    // (one HBM-bound pass, then the TMA kernels), unless the caller asks for
    // the in-kernel loader or the allocation fails; rows that are not a
    // multiple of 4 bytes are always staged (the loader cannot copy them).
    const void* opA = dY;
    const void* opB = X;
    int64_t ldA = p.M * es, ldB = p.N * es;
    void* scratch = nullptr;  // pool allocation to return after the kernel
    const bool want_stage = stage_misaligned();
    const bool stage_a = rows > 0 && p.manual_a && (want_stage || p.gran_a < 4);
    const bool stage_b = rows > 0 && p.manual_b && (want_stage || p.gran_b < 4);
    const bool must_stage = (stage_a && p.gran_a < 4) || (stage_b && p.gran_b < 4);
    if (stage_a || stage_b) {
        const int64_t pa = stage_a ? (ldA + 15) / 16 * 16 : 0;
        const int64_t pb = stage_b ? (ldB + 15) / 16 * 16 : 0;
        const int64_t need = (pa + pb) * rows;
        void* stage = nullptr;
        if (stage_from == StageFrom::Static) {
            // fixed buffer: refuse what does not fit, before any launch
            if (need > static_cast<int64_t>(static_stage_capacity()))
                return FORGE_ERR_SCRATCH_TOO_SMALL;
            if (static_stage_address(dev->ordinal, &stage) != cudaSuccess) {
                cudaGetLastError();
                return FORGE_ERR_CUDA;
            }
        } else if (scratch_alloc(&scratch, static_cast<size_t>(need), stream) == cudaSuccess) {
            stage = scratch;
        } else {
            cudaGetLastError();
            scratch = nullptr;
            if (must_stage) return FORGE_ERR_CUDA;  // no loader fallback for such rows
        }
        if (stage) {
            uint8_t* sp = static_cast<uint8_t*>(stage);
            cudaError_t ce = cudaSuccess;
            if (stage_a) {
                ce = stage_rows(dY, sp, rows, ldA, pa, p.gran_a, dev->sms, stream);
                opA = sp;
                ldA = pa;
                p.manual_a = 0;
                sp += pa * rows;
            }
            if (ce == cudaSuccess && stage_b) {
                ce = stage_rows(X, sp, rows, ldB, pb, p.gran_b, dev->sms, stream);
                opB = sp;
                ldB = pb;
                p.manual_b = 0;
            }
            if (ce != cudaSuccess) {
                if (scratch) scratch_free(scratch, stream);
                return FORGE_ERR_CUDA;
            }
        }
    }

    const bool man = p.manual_a || p.manual_b;
    const int form = kernel_form(p, man);
    Maps maps;
    std::memset(&maps, 0, sizeof maps);
    p.has_maps = rows > 0 ? 1 : 0;
    if (rows > 0) {
        st = FORGE_OK;
        if (!p.manual_a) st = encode_operand(&maps.a, opA, in_dtype, p.M, rows, ldA);
        if (st == FORGE_OK && !p.manual_b)
            st = encode_operand(&maps.b, opB, in_dtype, p.N, rows, ldB);
        if (st == FORGE_OK && grouped && !p.manual_a)
            st = encode_operand(&maps.a1, opA, in_dtype, p.M, rows, ldA, 0);
        if (st == FORGE_OK && grouped && !p.manual_b)
            st = encode_operand(&maps.b1, opB, in_dtype, p.N, rows, ldB, 0);
        // one MMA k-step (16 bf16 or 32 e4m3 rows) = a quarter of a k-block
        if (st == FORGE_OK && grouped && !p.manual_a)
            st = encode_operand(&maps.ak, opA, in_dtype, p.M, rows, ldA, 4);
        if (st == FORGE_OK && grouped && !p.manual_b)
            st = encode_operand(&maps.bk, opB, in_dtype, p.N, rows, ldB, 4);
        if (st != FORGE_OK) {
            if (scratch) scratch_free(scratch, stream);
            return st;
        }
    }
    const int64_t tile_m = form == 1 ? 2 * BM : BM;
    const int64_t tiles_m = (p.M + tile_m - 1) / tile_m;
    const int64_t tiles_n = (p.N + BN - 1) / BN;
    const int64_t total = tiles_m * tiles_n * p.E;  // at least 1, within the bound checked above
    p.tiles_m = static_cast<int32_t>(tiles_m);
    p.tiles_n = static_cast<int32_t>(tiles_n);
    p.raster_band = raster_band(p.tiles_m, kDefaultRasterBand);
    p.timeout_ns = wait_timeout_ns();
    p.status = dev->status;

    const int ist = state_dtype == FORGE_BF16 ? ST_BF16 : ST_F32;
    cudaError_t e;
    if (form == 1) {
        // the launcher sizes the grid from the resident-cluster limit
        e = in_dtype == FORGE_BF16
                ? dispatch_pair<IN_BF16>(op, ist, grouped, maps, p, total, stream)
                : dispatch_pair<IN_E4M3>(op, ist, grouped, maps, p, total, stream);
    } else {
        const int grid = static_cast<int>(total < dev->sms ? total : dev->sms);
        if (in_dtype == FORGE_BF16)
            e = man ? dispatch_op<IN_BF16, true>(op, ist, grouped, maps, p, grid, stream)
                    : dispatch_op<IN_BF16, false>(op, ist, grouped, maps, p, grid, stream);
        else
            e = man ? dispatch_op<IN_E4M3, true>(op, ist, grouped, maps, p, grid, stream)
                    : dispatch_op<IN_E4M3, false>(op, ist, grouped, maps, p, grid, stream);
    }
    // the staging copy is released after the kernel, in stream order
    if (scratch) {
        const cudaError_t fe = scratch_free(scratch, stream);
        if (e == cudaSuccess) e = fe;
    }
    return from_cuda(e);
}

// A multi-problem call: P problems share X [K, N]; problem j has dY_j
// [K, M_j] and W_j, m_j, v_j [N, M_j].  One launch of the CTA-pair kernel
// walks all problems' tiles (problem by problem, d_out fastest), so small
// problems fill the SMs that a lone call of theirs would leave idle and the
// launch has one tail instead of P.  bf16 inputs, AdamW.  Operands whose rows
// TMA cannot address are staged into one pool allocation first.
forge_status run_multi(const void* X, int64_t N, int64_t K, int32_t P, const void* const* dY,
                       forge_dtype state_dtype, Params p, cudaStream_t stream)
{
    DeviceInfo* dev = nullptr;
    forge_status st = current_device(&dev);
    if (st != FORGE_OK) return st;
    {
        const void* ptrs[1 + 4 * kMaxProblems] = {K > 0 ? X : nullptr};
        for (int j = 0; j < P; ++j) {
            ptrs[1 + 4 * j] = K > 0 ? dY[j] : nullptr;
            ptrs[2 + 4 * j] = p.W_of[j];
            ptrs[3 + 4 * j] = p.s1_of[j];
            ptrs[4 + 4 * j] = p.s2_of[j];
        }
        if ((st = check_resident(dev->ordinal, ptrs, 1 + 4 * P)) != FORGE_OK) return st;
    }
    constexpr int es = 2;  // bf16
    const int64_t tiles_n = (N + BN - 1) / BN;
    int64_t total = 0;
    for (int j = 0; j < P; ++j) {
        const int64_t tm = (p.M_of[j] + 2 * BM - 1) / (2 * BM);
        p.tile_begin[j] = static_cast<int32_t>(total);
        p.tiles_m_of[j] = static_cast<int32_t>(tm);
        total += tm * tiles_n;
        if (total > INT32_MAX) return FORGE_ERR_INVALID_ARG;
    }
    for (int j = P; j <= kMaxProblems; ++j)
        p.tile_begin[j] = j == P ? static_cast<int32_t>(total) : INT32_MAX;

    const uintptr_t sa = state_dtype == FORGE_BF16 ? 2 : 4;
    const uintptr_t va = state_dtype == FORGE_BF16 ? 8 : 16;
    bool vec = true;
    for (int j = 0; j < P; ++j) {
        if (!aligned(p.W_of[j], 4) || !aligned(p.s1_of[j], sa) || !aligned(p.s2_of[j], sa))
            return FORGE_ERR_MISALIGNED;
        vec = vec && p.M_of[j] % 4 == 0 && aligned(p.W_of[j], 16) && aligned(p.s1_of[j], va) &&
              aligned(p.s2_of[j], va);
    }
    p.vec_ok = vec ? 1 : 0;

    // operands TMA cannot address: padded copies with 16-byte rows
    const void* opX = X;
    int64_t ldX = N * es;
    const void* opD[kMaxProblems] = {};
    int64_t ldD[kMaxProblems] = {};
    int gran[kMaxProblems + 1] = {};
    int64_t need = 0;
    if (K > 0) {
        gran[kMaxProblems] = operand_path(X, N, es);
        if (gran[kMaxProblems] < 0) return FORGE_ERR_MISALIGNED;
        if (gran[kMaxProblems] > 0) need += (ldX + 15) / 16 * 16 * K;
        for (int j = 0; j < P; ++j) {
            opD[j] = dY[j];
            ldD[j] = p.M_of[j] * es;
            gran[j] = operand_path(dY[j], p.M_of[j], es);
            if (gran[j] < 0) return FORGE_ERR_MISALIGNED;
            if (gran[j] > 0) need += (ldD[j] + 15) / 16 * 16 * K;
        }
    }
    void* scratch = nullptr;
    if (need > 0) {
        if (scratch_alloc(&scratch, static_cast<size_t>(need), stream) != cudaSuccess) {
            cudaGetLastError();
            return FORGE_ERR_CUDA;
        }
        uint8_t* sp = static_cast<uint8_t*>(scratch);
        cudaError_t ce = cudaSuccess;
        if (gran[kMaxProblems] > 0) {
            const int64_t pad = (ldX + 15) / 16 * 16;
            ce = stage_rows(X, sp, K, ldX, pad, gran[kMaxProblems], dev->sms, stream);
            opX = sp;
            ldX = pad;
            sp += pad * K;
        }
        for (int j = 0; j < P && ce == cudaSuccess; ++j) {
            if (gran[j] == 0) continue;
            const int64_t pad = (ldD[j] + 15) / 16 * 16;
            ce = stage_rows(dY[j], sp, K, ldD[j], pad, gran[j], dev->sms, stream);
            opD[j] = sp;
            ldD[j] = pad;
            sp += pad * K;
        }
        if (ce != cudaSuccess) {
            scratch_free(scratch, stream);
            return FORGE_ERR_CUDA;
        }
    }

    Maps maps;
    std::memset(&maps, 0, sizeof maps);
    MultiMaps mm;
    std::memset(&mm, 0, sizeof mm);
    p.has_maps = K > 0 ? 1 : 0;
    if (K > 0) {
        st = encode_operand(&maps.b, opX, FORGE_BF16, N, K, ldX);
        for (int j = 0; j < P && st == FORGE_OK; ++j)
            st = encode_operand(&mm.a[j], opD[j], FORGE_BF16, p.M_of[j], K, ldD[j]);
        if (st != FORGE_OK) {
            if (scratch) scratch_free(scratch, stream);
            return st;
        }
    }
    p.N = N;
    p.K = K;
    p.E = 1;
    p.P = P;
    p.M = p.M_of[0];
    p.W = p.W_of[0];
    p.s1 = p.s1_of[0];
    p.s2 = p.s2_of[0];
    p.tiles_m = p.tiles_m_of[0];
    p.tiles_n = static_cast<int32_t>(tiles_n);
    int32_t tm_max = 1;
    for (int j = 0; j < P; ++j) tm_max = std::max(tm_max, p.tiles_m_of[j]);
    p.raster_band = raster_band(tm_max, 0);
    p.timeout_ns = wait_timeout_ns();
    p.status = dev->status;
    cudaError_t e =
        state_dtype == FORGE_BF16
            ? launch_wgrad_pair<IN_BF16, OP_ADAMW, ST_BF16, false, true>(
                  maps.a, maps.b, maps.a1, maps.b1, maps.ak, maps.bk, mm, p, total, stream)
            : launch_wgrad_pair<IN_BF16, OP_ADAMW, ST_F32, false, true>(
                  maps.a, maps.b, maps.a1, maps.b1, maps.ak, maps.bk, mm, p, total, stream);
    if (scratch) {
        const cudaError_t fe = scratch_free(scratch, stream);
        if (e == cudaSuccess) e = fe;
    }
    return from_cuda(e);
}

forge_status check_sizes(int64_t M, int64_t N, int64_t K)
{
    if (M < 1 || N < 1 || K < 0) return FORGE_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FORGE_ERR_INVALID_ARG;
    return FORGE_OK;
}

forge_status check_inputs(const void* X, const void* dY, int64_t K, forge_dtype in_dtype,
                          const float* scales)
{
    if (K > 0 && (!X || !dY)) return FORGE_ERR_INVALID_ARG;
    if (in_dtype != FORGE_BF16 && in_dtype != FORGE_E4M3) return FORGE_ERR_UNSUPPORTED_DTYPE;
    if (in_dtype == FORGE_E4M3 && !scales) return FORGE_ERR_INVALID_ARG;
    if (in_dtype == FORGE_BF16 && scales) return FORGE_ERR_INVALID_ARG;
    return FORGE_OK;
}

forge_status check_adam(float lr, float beta1, float beta2, float eps, float wd, int64_t step)
{
    if (step < 1) return FORGE_ERR_INVALID_ARG;
    if (!finite_nonneg(lr) || !finite_nonneg(eps) || !finite_nonneg(wd)) return FORGE_ERR_INVALID_ARG;
    if (!(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f))
        return FORGE_ERR_INVALID_ARG;
    return FORGE_OK;
}

void fill_adam(Params& p, float lr, float beta1, float beta2, float eps, float wd, int64_t step)
{
    // Bias corrections in double, as torch computes them on the host.
    const double bc1 = 1.0 - std::pow(static_cast<double>(beta1), static_cast<double>(step));
    const double bc2 = 1.0 - std::pow(static_cast<double>(beta2), static_cast<double>(step));
    p.decay = static_cast<float>(1.0 - static_cast<double>(lr) * wd);
    p.b1 = beta1;
    p.omb1 = static_cast<float>(1.0 - static_cast<double>(beta1));
    p.b2 = beta2;
    p.omb2 = static_cast<float>(1.0 - static_cast<double>(beta2));
    p.step_size = static_cast<float>(lr / bc1);
    p.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
    p.eps = eps;
}

}  // namespace

forge_status forge::device_sms(int* sms)
{
    DeviceInfo* dev = nullptr;
    const forge_status st = current_device(&dev);
    if (st == FORGE_OK) *sms = dev->sms;
    return st;
}

forge_status forge::device_resident(const void* const* ptrs, int n)
{
    DeviceInfo* dev = nullptr;
    const forge_status st = current_device(&dev);
    return st == FORGE_OK ? check_resident(dev->ordinal, ptrs, n) : st;
}

namespace {
std::mutex g_pool_mu;
cudaMemPool_t g_pool[kMaxDevices] = {};
}  // namespace

cudaError_t forge::scratch_alloc(void** ptr, size_t bytes, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaMemPool_t pool;
    {
        std::lock_guard<std::mutex> lk(g_pool_mu);
        if (!g_pool[dev]) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            cudaMemPool_t np;
            if ((e = cudaMemPoolCreate(&np, &props)) != cudaSuccess) return e;
            uint64_t keep = ~0ull;
            if ((e = cudaMemPoolSetAttribute(np, cudaMemPoolAttrReleaseThreshold, &keep)) !=
                cudaSuccess) {
                cudaMemPoolDestroy(np);
                return e;
            }
            g_pool[dev] = np;
        }
        pool = g_pool[dev];
    }
    return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

cudaError_t forge::scratch_free(void* ptr, cudaStream_t stream) { return cudaFreeAsync(ptr, stream); }

int* forge::device_status_word()
{
    DeviceInfo* dev = nullptr;
    return current_device(&dev) == FORGE_OK ? dev->status : nullptr;
}

int64_t forge::wait_timeout() { return wait_timeout_ns(); }

cudaError_t forge::encode_bf16_kmajor(CUtensorMap* map, const void* base, int64_t inner,
                                      int64_t rows, uint32_t box_rows, int64_t ld_bytes)
{
    if (!ensure_encode()) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_bytes)};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r =
        g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t forge::stage_padded_rows(const void* src, void* dst, int64_t rows, int64_t row_bytes,
                                     int64_t dst_row_bytes, cudaStream_t stream)
{
    DeviceInfo* dev = nullptr;
    if (current_device(&dev) != FORGE_OK) return cudaErrorInvalidDevice;
    const int gran = aligned(src, 8) && row_bytes % 8 == 0   ? 8
                     : aligned(src, 4) && row_bytes % 4 == 0 ? 4
                                                             : 1;
    return stage_rows(src, dst, rows, row_bytes, dst_row_bytes, gran, dev->sms, stream);
}

forge_status forge::adamw_checks(const void* X, const void* dY, const float* W, const void* m,
                                 const void* v, int64_t M, int64_t N, int64_t K,
                                 forge_dtype in_dtype, forge_dtype state_dtype, float lr,
                                 float beta1, float beta2, float eps, float wd, int64_t step)
{
    if (!W || !m || !v) return FORGE_ERR_INVALID_ARG;
    forge_status s;
    if ((s = check_sizes(M, N, K)) != FORGE_OK) return s;
    if ((s = check_inputs(X, dY, K, in_dtype, nullptr)) != FORGE_OK) return s;
    if (state_dtype != FORGE_F32 && state_dtype != FORGE_BF16) return FORGE_ERR_UNSUPPORTED_DTYPE;
    if ((s = check_adam(lr, beta1, beta2, eps, wd, step)) != FORGE_OK) return s;
    const uintptr_t sa = state_dtype == FORGE_BF16 ? 2 : 4;
    if (!aligned(W, 4) || !aligned(m, sa) || !aligned(v, sa)) return FORGE_ERR_MISALIGNED;
    if (K > 0 && operand_path(X, N, elem_size(in_dtype)) < 0) return FORGE_ERR_MISALIGNED;
    return FORGE_OK;
}

namespace {

// The owner-side step behind a reduce-scatter: checks, then one HBM-bound
// elementwise launch over the shard (forge_owner.cu).
forge_status run_owner(int op, const float* G, float* W, void* s1, void* s2, int64_t n,
                       forge_dtype state_dtype, Params& p, cudaStream_t stream)
{
    DeviceInfo* dev = nullptr;
    forge_status st = current_device(&dev);
    if (st != FORGE_OK) return st;
    if (n == 0) return FORGE_OK;
    const void* ptrs[] = {G, W, s1, s2};
    if ((st = check_resident(dev->ordinal, ptrs, 4)) != FORGE_OK) return st;
    const uintptr_t sa = state_dtype == FORGE_BF16 ? 2 : 4;
    const uintptr_t va = state_dtype == FORGE_BF16 ? 8 : 16;
    if (!aligned(G, 4) || !aligned(W, 4) || !aligned(s1, sa) || (s2 && !aligned(s2, sa)))
        return FORGE_ERR_MISALIGNED;
    const bool vec = aligned(G, 16) && aligned(W, 16) && aligned(s1, va) && (!s2 || aligned(s2, va));
    p.W = W;
    p.s1 = s1;
    p.s2 = s2;
    return from_cuda(launch_owner(op, state_dtype == FORGE_BF16 ? ST_BF16 : ST_F32, G, p, n, vec,
                                  dev->sms, stream));
}

}  // namespace

extern "C" {

forge_status forge_wgrad_adamw(const void* X, const void* dY, float* W, void* m, void* v,
                               int64_t M, int64_t N, int64_t K, forge_dtype in_dtype,
                               forge_dtype state_dtype, float lr, float beta1, float beta2,
                               float eps, float wd, int64_t step, const float* scales,
                               forge_stream_t stream)
{
    if (!W || !m || !v) return FORGE_ERR_INVALID_ARG;
    forge_status s;
    if ((s = check_sizes(M, N, K)) != FORGE_OK) return s;
    if ((s = check_inputs(X, dY, K, in_dtype, scales)) != FORGE_OK) return s;
    if (state_dtype != FORGE_F32 && state_dtype != FORGE_BF16) return FORGE_ERR_UNSUPPORTED_DTYPE;
    if ((s = check_adam(lr, beta1, beta2, eps, wd, step)) != FORGE_OK) return s;
    Params p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.E = 1;
    p.W = W;
    p.s1 = m;
    p.s2 = v;
    p.scales = scales;
    fill_adam(p, lr, beta1, beta2, eps, wd, step);
    return run(X, dY, K, in_dtype, OP_ADAMW, state_dtype, false, p,
               reinterpret_cast<cudaStream_t>(stream));
}

forge_status forge_wgrad_adamw_multi(const void* X, int64_t N, int64_t K, int32_t P,
                                     const void* const* dY, const int64_t* M, float* const* W,
                                     void* const* m, void* const* v, forge_dtype in_dtype,
                                     forge_dtype state_dtype, float lr, float beta1, float beta2,
                                     float eps, float wd, int64_t step, forge_stream_t stream)
{
    if (P < 1 || P > kMaxProblems || !M || !W || !m || !v || (K > 0 && (!X || !dY)))
        return FORGE_ERR_INVALID_ARG;
    if (in_dtype != FORGE_BF16) return FORGE_ERR_UNSUPPORTED_DTYPE;
    if (state_dtype != FORGE_F32 && state_dtype != FORGE_BF16) return FORGE_ERR_UNSUPPORTED_DTYPE;
    forge_status s;
    if ((s = check_adam(lr, beta1, beta2, eps, wd, step)) != FORGE_OK) return s;
    Params p{};
    for (int j = 0; j < P; ++j) {
        if ((s = check_sizes(M[j], N, K)) != FORGE_OK) return s;
        if (!W[j] || !m[j] || !v[j] || (K > 0 && !dY[j])) return FORGE_ERR_INVALID_ARG;
        p.M_of[j] = M[j];
        p.W_of[j] = W[j];
        p.s1_of[j] = m[j];
        p.s2_of[j] = v[j];
    }
    fill_adam(p, lr, beta1, beta2, eps, wd, step);
    return run_multi(X, N, K, P, dY, state_dtype, p, reinterpret_cast<cudaStream_t>(stream));
}

forge_status forge_wgrad_adamw_noalloc(const void* X, const void* dY, float* W, void* m, void* v,
                                       int64_t M, int64_t N, int64_t K, forge_dtype in_dtype,
                                       forge_dtype state_dtype, float lr, float beta1,
                                       float beta2, float eps, float wd, int64_t step,
                                       const float* scales, forge_stream_t stream)
{
    if (!W || !m || !v) return FORGE_ERR_INVALID_ARG;
    forge_status s;
    if ((s = check_sizes(M, N, K)) != FORGE_OK) return s;
    if ((s = check_inputs(X, dY, K, in_dtype, scales)) != FORGE_OK) return s;
    if (state_dtype != FORGE_F32 && state_dtype != FORGE_BF16) return FORGE_ERR_UNSUPPORTED_DTYPE;
    if ((s = check_adam(lr, beta1, beta2, eps, wd, step)) != FORGE_OK) return s;
    Params p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.E = 1;
    p.W = W;
    p.s1 = m;
    p.s2 = v;
    p.scales = scales;
    fill_adam(p, lr, beta1, beta2, eps, wd, step);
    return run(X, dY, K, in_dtype, OP_ADAMW, state_dtype, false, p,
               reinterpret_cast<cudaStream_t>(stream), StageFrom::Static);
}

forge_status forge_wgrad_sgdm(const void* X, const void* dY, float* W, void* mom, int64_t M,
                              int64_t N, int64_t K, forge_dtype in_dtype, forge_dtype state_dtype,
                              float lr, float momentum, float wd, const float* scales,
                              forge_stream_t stream)
{
    if (!W || !mom) return FORGE_ERR_INVALID_ARG;
    forge_status s;
    if ((s = check_sizes(M, N, K)) != FORGE_OK) return s;
    if ((s = check_inputs(X, dY, K, in_dtype, scales)) != FORGE_OK) return s;
    if (state_dtype != FORGE_F32 && state_dtype != FORGE_BF16) return FORGE_ERR_UNSUPPORTED_DTYPE;
    if (!finite_nonneg(lr) || !finite_nonneg(momentum) || !finite_nonneg(wd))
        return FORGE_ERR_INVALID_ARG;
    Params p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.E = 1;
    p.W = W;
    p.s1 = mom;
    p.scales = scales;
    p.lr = lr;
    p.mu = momentum;
    p.wd = wd;
    return run(X, dY, K, in_dtype, OP_SGDM, state_dtype, false, p,
               reinterpret_cast<cudaStream_t>(stream));
}

forge_status forge_wgrad_only(const void* X, const void* dY, float* dW, int64_t M, int64_t N,
                              int64_t K, forge_dtype in_dtype, const float* scales,
                              forge_stream_t stream)
{
    if (!dW) return FORGE_ERR_INVALID_ARG;
    forge_status s;
    if ((s = check_sizes(M, N, K)) != FORGE_OK) return s;
    if ((s = check_inputs(X, dY, K, in_dtype, scales)) != FORGE_OK) return s;
    Params p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.E = 1;
    p.W = dW;  // only for the alignment check; the kernel writes p.dW
    p.dW = dW;
    p.scales = scales;
    return run(X, dY, K, in_dtype, OP_DW, FORGE_F32, false, p,
               reinterpret_cast<cudaStream_t>(stream));
}

forge_status forge_grouped_wgrad_adamw(const void* X, const void* dY, float* W, void* m, void* v,
                                       const int32_t* offsets, int32_t E, int64_t T_max,
                                       int64_t M, int64_t N, forge_dtype in_dtype,
                                       forge_dtype state_dtype, float lr, float beta1, float beta2,
                                       float eps, float wd, int64_t step, const float* scales,
                                       forge_stream_t stream)
{
    if (!W || !m || !v || !offsets) return FORGE_ERR_INVALID_ARG;
    if (E < 1 || E > kMaxExperts) return FORGE_ERR_INVALID_ARG;
    forge_status s;
    if ((s = check_sizes(M, N, T_max)) != FORGE_OK) return s;
    if ((s = check_inputs(X, dY, T_max, in_dtype, scales)) != FORGE_OK) return s;
    if (state_dtype != FORGE_F32 && state_dtype != FORGE_BF16) return FORGE_ERR_UNSUPPORTED_DTYPE;
    if ((s = check_adam(lr, beta1, beta2, eps, wd, step)) != FORGE_OK) return s;
    if (!aligned(offsets, 4)) return FORGE_ERR_MISALIGNED;
    Params p{};
    p.M = M;
    p.N = N;
    p.K = 0;
    p.T_max = T_max;
    p.offsets = offsets;
    p.E = E;
    p.W = W;
    p.s1 = m;
    p.s2 = v;
    p.scales = scales;
    fill_adam(p, lr, beta1, beta2, eps, wd, step);
    return run(X, dY, T_max, in_dtype, OP_ADAMW, state_dtype, true, p,
               reinterpret_cast<cudaStream_t>(stream));
}

forge_status forge_owner_adamw(const float* G, float* W, void* m, void* v, int64_t n,
                               forge_dtype state_dtype, float lr, float beta1, float beta2,
                               float eps, float wd, int64_t step, forge_stream_t stream)
{
    if (n < 0 || (n > 0 && (!G || !W || !m || !v))) return FORGE_ERR_INVALID_ARG;
    if (state_dtype != FORGE_F32 && state_dtype != FORGE_BF16) return FORGE_ERR_UNSUPPORTED_DTYPE;
    forge_status s;
    if ((s = check_adam(lr, beta1, beta2, eps, wd, step)) != FORGE_OK) return s;
    Params p{};
    fill_adam(p, lr, beta1, beta2, eps, wd, step);
    return run_owner(OP_ADAMW, G, W, m, v, n, state_dtype, p,
                     reinterpret_cast<cudaStream_t>(stream));
}

forge_status forge_owner_sgdm(const float* G, float* W, void* mom, int64_t n,
                              forge_dtype state_dtype, float lr, float momentum, float wd,
                              forge_stream_t stream)
{
    if (n < 0 || (n > 0 && (!G || !W || !mom))) return FORGE_ERR_INVALID_ARG;
    if (state_dtype != FORGE_F32 && state_dtype != FORGE_BF16) return FORGE_ERR_UNSUPPORTED_DTYPE;
    if (!finite_nonneg(lr) || !finite_nonneg(momentum) || !finite_nonneg(wd))
        return FORGE_ERR_INVALID_ARG;
    Params p{};
    p.lr = lr;
    p.mu = momentum;
    p.wd = wd;
    return run_owner(OP_SGDM, G, W, mom, nullptr, n, state_dtype, p,
                     reinterpret_cast<cudaStream_t>(stream));
}

const char* forge_status_string(forge_status status)
{
    switch (status) {
    case FORGE_OK: return "ok";
    case FORGE_ERR_INVALID_ARG: return "invalid argument";
    case FORGE_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case FORGE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case FORGE_ERR_MISALIGNED: return "misaligned pointer or row stride";
    case FORGE_ERR_CUDA: return "CUDA error";
    case FORGE_ERR_TIMEOUT: return "device-side wait timed out";
    case FORGE_ERR_SCRATCH_TOO_SMALL: return "operand staging needs more than the fixed scratch buffer";
    }
    return "unknown status";
}

forge_status forge_get_device_status(void)
{
    DeviceInfo* dev = nullptr;
    forge_status st = current_device(&dev);
    if (st != FORGE_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return FORGE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_forge_status, sizeof v) != cudaSuccess) return FORGE_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_forge_status, &zero, sizeof zero) != cudaSuccess) return FORGE_ERR_CUDA;
    return static_cast<forge_status>(v);
}

forge_status forge_selftest_wait_timeout(uint32_t timeout_us, forge_stream_t stream)
{
    if (timeout_us == 0 || timeout_us > 10000000u) return FORGE_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    forge_status st = current_device(&dev);
    if (st != FORGE_OK) return st;
    forge_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<int64_t>(timeout_us) * 1000, dev->status);
    return from_cuda(cudaGetLastError());
}

int32_t forge_version(void) { return 100; }

}  // extern "C"
