/*
 * forge.h -- C ABI of libforge.so: the weight-gradient GEMM dW = X^T dY with
 * the optimizer step fused into its tiled epilogue, for NVIDIA GB300
 * (compute capability 10.3, sm_103a).
 *
 * What the operations are (FORGE assessment PR, tessera#565, "docs(audit):
 * FORGE assessment + residency-aware epilogue-fusion track"):
 *   - The weight gradient of a linear layer is dW = X^T dY ("What's already
 *     in tree and easy to miss": dRhs = matmul(lhs, dy, transposeA=true)).
 *   - The optimizer step runs in the GEMM's tiled epilogue, so the gradient
 *     never reaches device memory (opening paragraph).  Each output tile is
 *     owned by one CTA and keeps the whole token dimension K (the full_k
 *     legality condition of FORGE Prop. 1, same section), so there is no
 *     split-K and no atomic accumulation; results are bitwise reproducible
 *     ("Math verified, not asserted", P1).
 *   - The fp32 accumulator feeds the optimizer state without truncation to
 *     bf16 (P6; the "truncf" item of "What's already in tree").
 *   - AdamW and SGD with momentum are the optimizers ("Claim hygiene on the
 *     source").  AdamW follows torch.optim.AdamW: W <- W (1 - lr wd);
 *     m <- b1 m + (1-b1) g; v <- b2 v + (1-b2) g^2;
 *     W <- W - lr (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps).
 *     SGD follows torch.optim.SGD (dampening 0, no Nesterov):
 *     g' = g + wd W; buf <- mu buf + g'; W <- W - lr buf.
 *   - Gradient clipping is not offered: exact global-norm clipping cannot be
 *     fused ("Math verified, not asserted", P2).
 *   - A routed (expert) weight whose expert received no tokens still takes
 *     the step with g = 0, i.e. m and v decay by b1, b2 and W by its weight
 *     decay (P5).
 *
 * Layouts (all row-major, element strides 1, no padding):
 *   X  [K, N]   activations, token-major (K tokens, N = d_in)
 *   dY [K, M]   output gradients, token-major (M = d_out)
 *   W, m, v, buf, dW  [N, M]   ([E, N, M] for the grouped call)
 *   dW[n][m] = sum_k X[k][n] * dY[k][m]  (times sX * sdY for e4m3 inputs)
 * An nn.Linear weight [d_out, d_in] is the transpose of W; pass it as its
 * [d_in, d_out] row-major view.
 *
 * Ownership and ordering: every pointer is caller-owned device memory of
 * the current device (cudaMalloc, a memory pool or a virtual-memory mapping;
 * host memory, managed memory and a peer GPU's memory are refused) and the
 * library keeps no pointer after the call returns.  Calls whose operands TMA
 * can address allocate nothing.  Two cases take stream-ordered scratch from
 * a memory pool the library creates per device (allocated and freed on
 * `stream`; the pool keeps what it has reserved, at most the largest scratch
 * in use at once, until the process ends):
 *   - an operand (X or dY; for dX, dY or Wb) whose base is not 16-byte
 *     aligned or whose row stride is not a multiple of 16 bytes (any odd
 *     bf16 width, any e4m3 width not divisible by 16) is first copied into
 *     rows padded to 16 bytes (one extra read and write of that operand).
 *     If that allocation fails, or the environment variable
 *     FORGE_MISALIGNED is "loader", an X or dY of the weight-gradient calls
 *     whose rows are a multiple of 4 bytes is fetched by the kernel itself
 *     with cp.async instead; other rows need the copy, and a failed
 *     allocation returns FORGE_ERR_CUDA.  forge_wgrad_adamw_noalloc stages
 *     into a fixed buffer instead;
 *   - forge_backward_adamw without a bf16 weight copy (see there).
 * W, m, v, buf are updated in place.  Calls are asynchronous and ordered on
 * `stream`, and can be captured in a CUDA graph once a first call has run
 * on the device; the return value reports only host-side validation and
 * launch errors.  Errors detected on the device (a bounded wait that
 * ran out) are recorded in a device status word read by
 * forge_get_device_status().  The library resolves the device addresses of
 * its own device variables (that status word, the no-allocation staging
 * buffer) once per device ordinal and keeps them; they belong to the device's
 * primary context, so calls after cudaDeviceReset, or from a context other
 * than the primary one, are not supported.
 *
 * Environment (each read on every call unless noted; none is needed):
 *   FORGE_MISALIGNED = stage | loader  how X, dY rows TMA cannot address
 *                      reach the kernel (default stage, see above)
 *   FORGE_KERNEL = single | pair       the weight-gradient kernel form:
 *                      one CTA per 128 x 256 tile, or CTA pairs on 256 x 256
 *                      tiles (default: pairs when d_out > 128)
 *   FORGE_RASTER_BAND = n              d_out tiles per raster band of the
 *                      tile walk (default 8; 0 = whole rows); the results
 *                      do not depend on it
 *   FORGE_DGRAD_KERNEL = single | pair the dX kernel form (default: pairs
 *                      unless K fits one 128-token tile)
 *   FORGE_WAIT_TIMEOUT_MS = ms         limit of every device-side wait
 *                      (read once per process; default 10000)
 *
 * Caller preconditions (not checked):
 *   - X and dY do not overlap W, m, v, buf or dW.
 *   - dX = dY W^T has already consumed the old W (the in-place
 *     "dX-before-update" hazard, "Math verified, not asserted", P1).
 *   - W's whole gradient for this step is X^T dY: no tied or shared use
 *     (the single-use guard of P1).
 *
 * Host-side checks run before any launch, in this order: null pointers
 * (X and dY may be NULL only when K == 0), sizes (M >= 1, N >= 1, K >= 0,
 * E >= 1, step >= 1), dtypes, then the device (compute capability 10.3),
 * then residency (every pointer the call reads or writes is device memory
 * of the current device, else FORGE_ERR_INVALID_ARG), then alignment (X, dY:
 * bases aligned to their element size, rows of any length; W, dW: 4-byte
 * bases; m, v, buf: bases aligned to their element size; see
 * FORGE_ERR_MISALIGNED).  The checks up to the dtypes need no GPU.
 */
#ifndef FORGE_H
#define FORGE_H

#include <stdint.h>

#if defined(__GNUC__)
#define FORGE_API __attribute__((visibility("default")))
#else
#define FORGE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers (same underlying type). */
typedef struct CUstream_st* forge_stream_t;

typedef enum {
    FORGE_OK = 0,
    FORGE_ERR_INVALID_ARG = -1,       /* null pointer, bad size or hyperparameter, or a
                                         pointer that is not device memory of the
                                         current device */
    FORGE_ERR_UNSUPPORTED_DTYPE = -2, /* dtype outside the supported set */
    FORGE_ERR_UNSUPPORTED_DEVICE = -3,/* no device, or compute capability != 10.3 */
    FORGE_ERR_MISALIGNED = -4,        /* a base pointer not aligned to its element size */
    FORGE_ERR_CUDA = -5,              /* a CUDA runtime / driver call failed */
    FORGE_ERR_TIMEOUT = -6,           /* a device-side bounded wait ran out */
    FORGE_ERR_SCRATCH_TOO_SMALL = -7  /* forge_wgrad_adamw_noalloc: staging exceeds its buffer */
} forge_status;

typedef enum {
    FORGE_BF16 = 0, /* bfloat16 */
    FORGE_E4M3 = 1, /* OCP fp8 E4M3 ("fn": no infinities, max 448) */
    FORGE_F32 = 2   /* IEEE binary32 */
} forge_dtype;

/*
 * Fused dW = X^T dY and one AdamW step on W, m, v.
 *   X, dY        device, [K, N] and [K, M] of in_dtype (FORGE_BF16 or
 *                FORGE_E4M3).  K may be 0: the step then runs with g = 0.
 *   W            device fp32 [N, M], updated in place.
 *   m, v         device [N, M] of state_dtype (FORGE_F32 or FORGE_BF16),
 *                updated in place.  With bf16 state, W is updated from the
 *                unrounded fp32 m, v and then m, v are stored rounded to
 *                nearest even.
 *   lr, beta1, beta2, eps, wd   AdamW hyperparameters (0 < beta < 1,
 *                lr >= 0, eps >= 0, wd >= 0).
 *   step         1-based step count after incrementing (as torch's AdamW).
 *   scales       device fp32 [2] = {sX, sdY} for FORGE_E4M3 inputs (the
 *                gradient is sX * sdY * X^T dY); must be NULL for bf16.
 * Row strides: N * elemsize(in_dtype) and M * elemsize(in_dtype) bytes, of
 * any length (rows TMA cannot address are staged, see above).
 */
FORGE_API forge_status forge_wgrad_adamw(const void* X, const void* dY, float* W, void* m, void* v,
                               int64_t M, int64_t N, int64_t K, forge_dtype in_dtype,
                               forge_dtype state_dtype, float lr, float beta1, float beta2,
                               float eps, float wd, int64_t step, const float* scales,
                               forge_stream_t stream);

/*
 * forge_wgrad_adamw without any device allocation.  The FORGE pages have no
 * counterpart to this call: it is a library variant of forge_wgrad_adamw for
 * callers that must not allocate device memory during a step.  Arguments,
 * layouts, checks and results are those of forge_wgrad_adamw (the results
 * are bitwise identical); only the staging copy of an operand whose base or
 * row stride is not 16-byte aligned differs: it goes into a fixed 256 MiB
 * buffer per device, a file-scope device array inside the library, instead
 * of a stream-ordered allocation.
 *   - Oversize: a call whose staging copy needs more than the buffer
 *     ((rows of X, dY) x (row bytes rounded up to 16), summed over the
 *     operands that need staging) returns FORGE_ERR_SCRATCH_TOO_SMALL before
 *     any launch and changes nothing.  Aligned operands need no staging.
 *   - Races: the buffer is shared by every call of this function on the
 *     device.  Calls that stage must be ordered (one stream, or streams
 *     synchronised with each other); two overlapping calls on unordered
 *     streams overwrite each other's staging copy.  forge_wgrad_adamw and
 *     the other entry points never touch the buffer.
 *   - State: each call writes every byte of the buffer that its kernel then
 *     reads (the padding after each staged row lies outside the tensor maps),
 *     so nothing carries over from an earlier call.
 *   - First-call setup: the first call on a device resolves the buffer's
 *     address (cudaGetSymbolAddress) and caches it for that device ordinal.
 *     Under lazy module loading (the CUDA default) this first call loads the
 *     library module holding the buffer and reserves its 256 MiB there for
 *     the life of the process; with CUDA_MODULE_LOADING=EAGER every device
 *     reserves it as soon as the process creates its context there, whether
 *     or not this function is ever called.  Make that first call outside
 *     stream capture; later calls are capturable.  The cached address
 *     belongs to the device's primary context: calls after cudaDeviceReset,
 *     or from another context on the device, are not supported.
 *   - FORGE_MISALIGNED=loader selects the kernel's own cp.async loader here
 *     too for rows that are a multiple of 4 bytes (no staging, no buffer);
 *     other rows are still staged into the buffer.
 */
FORGE_API forge_status forge_wgrad_adamw_noalloc(const void* X, const void* dY, float* W, void* m,
                                                 void* v, int64_t M, int64_t N, int64_t K,
                                                 forge_dtype in_dtype, forge_dtype state_dtype,
                                                 float lr, float beta1, float beta2, float eps,
                                                 float wd, int64_t step, const float* scales,
                                                 forge_stream_t stream);

/*
 * Several AdamW weight-gradient steps that share X, in one launch: for each
 * problem j < P, dW_j = X^T dY_j and one AdamW step on W_j, m_j, v_j, exactly
 * as forge_wgrad_adamw(X, dY[j], W[j], m[j], v[j], M[j], N, K, ...) would
 * compute it (bitwise wherever that call runs on CTA pairs, M[j] > 128: the
 * same 256 x 256 tiles in the same K order).  For layers whose
 * projections read the same activations (an attention block's projections):
 * the problems' tiles form one list walked by one grid, so SMs that a small
 * problem alone would leave idle run the others' tiles.  The operation of
 * each problem is the one forge_wgrad_adamw states; the pages know no
 * batched form of it.
 *   X            device bf16 [K, N], shared by all problems.
 *   P            1 <= P <= 8 problems.
 *   dY, M, W, m, v   host arrays of P entries: device bf16 dY[j] [K, M[j]],
 *                device fp32 W[j] and state_dtype m[j], v[j] [N, M[j]]
 *                (pointers the caller owns; the arrays are read during the
 *                call only).  Problems must not share W, m or v.
 *   in_dtype     FORGE_BF16 only (else FORGE_ERR_UNSUPPORTED_DTYPE).
 *   state_dtype, lr, beta1, beta2, eps, wd, step: as forge_wgrad_adamw, the
 *                same for every problem.
 * Checks as forge_wgrad_adamw, per problem, before any launch; operands
 * whose rows TMA cannot address are staged into the library's memory pool
 * (one allocation per call), and a failed allocation returns FORGE_ERR_CUDA.
 */
FORGE_API forge_status forge_wgrad_adamw_multi(const void* X, int64_t N, int64_t K, int32_t P,
                                               const void* const* dY, const int64_t* M,
                                               float* const* W, void* const* m, void* const* v,
                                               forge_dtype in_dtype, forge_dtype state_dtype,
                                               float lr, float beta1, float beta2, float eps,
                                               float wd, int64_t step, forge_stream_t stream);

/*
 * Per-tensor e4m3 quantisation with an amax scale, the step in front of an
 * fp8 call (the fp8 rows of "Math verified, not asserted", P6; the recipe
 * s = amax / 448 of the fp8 workload):
 *   x       device [n] of x_dtype (FORGE_F32 or FORGE_BF16), read as a flat
 *           array (any tensor shape, row-major).
 *   codes   device [n] bytes: OCP e4m3fn codes, each the value nearest to
 *           x / s computed in fp32 (ties to even; magnitudes past 448 saturate).
 *   scale   device float[1]: receives s = amax|x| / 448 (an fp32 division),
 *           or 1 when amax is 0 (n == 0 included).  NaN entries of x are left
 *           out of the amax (their codes are NaN).
 * Pass codes and scale as X (or dY) and scales[0] (or scales[1]) of an e4m3
 * call.  Nothing is allocated: two passes over x, the first of which parks
 * one partial maximum per block (at most four blocks per SM) in an aligned
 * window of `codes`, which the second pass then overwrites with the codes.
 * codes must not overlap x or scale.  Errors: n < 0, scale NULL, or x / codes
 * NULL with n > 0 -> FORGE_ERR_INVALID_ARG; x_dtype -> FORGE_ERR_UNSUPPORTED_DTYPE;
 * x not aligned to its element size or scale not 4-byte aligned ->
 * FORGE_ERR_MISALIGNED; a pointer that is not device memory of the current
 * device -> FORGE_ERR_INVALID_ARG.
 */
FORGE_API forge_status forge_quantize_e4m3(const void* x, forge_dtype x_dtype, int64_t n,
                                           uint8_t* codes, float* scale, forge_stream_t stream);

/*
 * The input gradient dX = dY W^T (bf16 in, fp32 accumulation, bf16 out,
 * nearest even), the GEMM on the other side of the backward pass that must
 * read W before the fused update overwrites it ("Math verified, not
 * asserted", P1).
 *   dY  device [K, M] bf16 (the same tensor the weight gradient reads).
 *   Wb  device [N, M] bf16: the weight as the forward pass used it (for a
 *       fp32 master W, its bf16 copy).
 *   dX  device [K, N] bf16, written.
 * in_dtype must be FORGE_BF16; K may be 0 (nothing is written).  dY, Wb and
 * dX need bases aligned to their element size (else FORGE_ERR_MISALIGNED);
 * rows of any width are accepted: when dY's or Wb's base is not 16-byte
 * aligned or M * 2 is not a multiple of 16, that operand is first copied into
 * rows padded to 16 bytes in a stream-ordered scratch buffer from the
 * library's memory pool (freed on `stream` after the launch; a failed
 * allocation returns FORGE_ERR_CUDA).
 */
FORGE_API forge_status forge_dgrad(const void* dY, const void* Wb, void* dX, int64_t M, int64_t N,
                                   int64_t K, forge_dtype in_dtype, forge_stream_t stream);

/*
 * One backward-and-update step for a linear layer, in the order the in-place
 * update requires: dX = dY Wb^T first, then the fused dW = X^T dY + AdamW on
 * W, m, v (exactly forge_wgrad_adamw), both on `stream`, so dX always sees
 * the weights from before this step.  Wb is the bf16 copy of W the forward
 * pass used; with Wb == NULL the library first rounds W to bf16 (nearest
 * even) into a scratch copy (N rows of M * 2 bytes rounded up to 16) from its
 * memory pool, allocated and freed in stream order on `stream`, together with
 * any staging copy forge_dgrad would make.  bf16 inputs only.  Every argument
 * check of both halves runs before the first launch; the arguments are those
 * of forge_dgrad and forge_wgrad_adamw.
 */
FORGE_API forge_status forge_backward_adamw(const void* X, const void* dY, float* W, void* m,
                                            void* v, const void* Wb, void* dX, int64_t M,
                                            int64_t N, int64_t K, forge_dtype in_dtype,
                                            forge_dtype state_dtype, float lr, float beta1,
                                            float beta2, float eps, float wd, int64_t step,
                                            forge_stream_t stream);

/*
 * Fused dW = X^T dY and one SGD-momentum step on W and the momentum buffer
 * mom ([N, M] of state_dtype).  On the first step pass mom = 0 (then
 * mom' = g + wd W, as torch's SGD).  Other arguments as forge_wgrad_adamw.
 */
FORGE_API forge_status forge_wgrad_sgdm(const void* X, const void* dY, float* W, void* mom, int64_t M,
                              int64_t N, int64_t K, forge_dtype in_dtype, forge_dtype state_dtype,
                              float lr, float momentum, float wd, const float* scales,
                              forge_stream_t stream);

/*
 * dW = X^T dY alone, stored as fp32 [N, M] into dW (device).  This is the
 * only call that writes a gradient to device memory; it exists to check the
 * contraction by itself.
 */
FORGE_API forge_status forge_wgrad_only(const void* X, const void* dY, float* dW, int64_t M, int64_t N,
                              int64_t K, forge_dtype in_dtype, const float* scales,
                              forge_stream_t stream);

/*
 * Grouped (mixture-of-experts) form: E experts, each with its own W, m, v
 * block [N, M] (stacked as [E, N, M]) and its own token rows.  X [T, N] and
 * dY [T, M] hold the tokens packed by expert: expert e owns rows
 * [offsets[e], offsets[e+1]) (offsets: device int32 [E+1], non-decreasing,
 * offsets[0] >= 0, read on the device, so no host synchronisation).
 * The gradient of expert e is X_e^T dY_e over its own rows only.  An expert
 * with no rows still takes the AdamW step with g = 0 (P5).  `step` is the
 * same for every expert.  T_total = offsets[E] is bounded by `T_max`
 * (the number of rows of the X, dY allocations).  1 <= E <= 1024.
 */
FORGE_API forge_status forge_grouped_wgrad_adamw(const void* X, const void* dY, float* W, void* m, void* v,
                                       const int32_t* offsets, int32_t E, int64_t T_max,
                                       int64_t M, int64_t N, forge_dtype in_dtype,
                                       forge_dtype state_dtype, float lr, float beta1, float beta2,
                                       float eps, float wd, int64_t step, const float* scales,
                                       forge_stream_t stream);

/*
 * The owner's optimizer step behind a reduce-scatter (data parallelism with
 * the optimizer state sharded, ZeRO-2 style; "Math verified, not asserted",
 * P3: under a reduce-scatter every output tile has exactly one owner, which
 * alone applies the update).  Each rank contracts its own tokens into a
 * partial fp32 dW (forge_wgrad_only); a reduce-scatter sums the partials and
 * hands every rank the rows of W it owns; the owner then calls this on its
 * shard.  Unlike the fused calls this path reads a gradient from device
 * memory: the partial gradients exist because the collective exchanges them.
 *   G      device fp32 [n]: the summed gradient of the owner's shard.
 *   W      device fp32 [n], updated in place.
 *   m, v   device [n] of state_dtype (FORGE_F32 or FORGE_BF16), updated in place.
 *   n      elements in the shard (a row range [r0, r1) of a row-major [N, M]
 *          weight is the flat range [r0 M, r1 M)); n = 0 does nothing.
 *   lr, beta1, beta2, eps, wd, step: as forge_wgrad_adamw.
 * The update is the fused epilogue's arithmetic, operation for operation:
 * given the dW that forge_wgrad_only computes for (X, dY), the result equals
 * forge_wgrad_adamw's on (X, dY) bit for bit.  G must not overlap W, m, v.
 * Errors: n < 0 or a NULL pointer with n > 0, or a hyperparameter out of
 * range -> FORGE_ERR_INVALID_ARG; state_dtype -> FORGE_ERR_UNSUPPORTED_DTYPE;
 * pointers outside device memory of the current device ->
 * FORGE_ERR_INVALID_ARG; G, W not 4-byte aligned or m, v not aligned to
 * their element size -> FORGE_ERR_MISALIGNED.  Allocates nothing.
 */
FORGE_API forge_status forge_owner_adamw(const float* G, float* W, void* m, void* v, int64_t n,
                                         forge_dtype state_dtype, float lr, float beta1,
                                         float beta2, float eps, float wd, int64_t step,
                                         forge_stream_t stream);

/* The same for SGD with momentum (mom as forge_wgrad_sgdm's). */
FORGE_API forge_status forge_owner_sgdm(const float* G, float* W, void* mom, int64_t n,
                                        forge_dtype state_dtype, float lr, float momentum,
                                        float wd, forge_stream_t stream);

/* Static description of a status code; never NULL. */
FORGE_API const char* forge_status_string(forge_status status);

/*
 * Read and clear the device status word of the current device: FORGE_OK, or
 * FORGE_ERR_TIMEOUT if a kernel's bounded wait ran out since the last read.
 * Synchronises the current device.
 */
FORGE_API forge_status forge_get_device_status(void);

/*
 * Failure-detection self-test: launches one CTA that waits on a barrier no
 * one arrives at, with a limit of timeout_us microseconds; the wait runs out,
 * the kernel records FORGE_ERR_TIMEOUT in the device status word and
 * returns normally (no trap, the context stays usable).
 */
FORGE_API forge_status forge_selftest_wait_timeout(uint32_t timeout_us, forge_stream_t stream);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
FORGE_API int32_t forge_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FORGE_H */
