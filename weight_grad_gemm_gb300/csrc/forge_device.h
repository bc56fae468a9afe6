// forge_device.h -- host helpers shared by the entry points (defined in
// forge_api.cu): the device check, the device status word, the bounded-wait
// limit, TMA descriptor encoding and the AdamW argument checks.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "forge.h"

namespace forge {

// The current device, checked once per device for compute capability 10.3;
// on success *sms receives its SM count.
forge_status device_sms(int* sms);

// FORGE_OK when every non-null pointer of ptrs[0..n) is device memory of the
// current device (checked with cudaPointerGetAttributes), else
// FORGE_ERR_INVALID_ARG (or the device check's status).
forge_status device_resident(const void* const* ptrs, int n);

// Device address of the status word on the current device (after a
// successful device_sms call).
int* device_status_word();

// Bounded-wait limit in nanoseconds (FORGE_WAIT_TIMEOUT_MS, default 10 s).
int64_t wait_timeout();

// bf16 [rows, inner] row-major, 16-byte aligned base and row stride ld_bytes
// (a multiple of 16), read in boxes of 64 elements of the inner (contraction)
// dimension x box_rows rows with 128-byte swizzle: the K-major operand layout
// of tcgen05.mma.  Columns past `inner` read as zeros.
cudaError_t encode_bf16_kmajor(CUtensorMap* map, const void* base, int64_t inner, int64_t rows,
                               uint32_t box_rows, int64_t ld_bytes);

// Copies [rows, row_bytes] from src (rows packed, base aligned to at least the
// element size) into dst (256-byte aligned) with rows dst_row_bytes apart (a
// multiple of 16 and >= row_bytes), on `stream`: the staging copy that makes
// an operand TMA-addressable.  The padding after each row is left unwritten.
cudaError_t stage_padded_rows(const void* src, void* dst, int64_t rows, int64_t row_bytes,
                              int64_t dst_row_bytes, cudaStream_t stream);

// Stream-ordered scratch from the library's own memory pool on the current
// device (created on first use).  The pool keeps what it has reserved (its
// release threshold is unbounded), so a call after a synchronisation does not
// map fresh memory again; it holds at most the largest scratch in use at
// once.  scratch_free returns the block in stream order.
cudaError_t scratch_alloc(void** ptr, size_t bytes, cudaStream_t stream);
cudaError_t scratch_free(void* ptr, cudaStream_t stream);

struct Params;

// The owner-side optimizer step (forge_owner.cu): op OP_ADAMW or OP_SGDM,
// st ST_F32 or ST_BF16, over n elements of the flat gradient G and the state
// in p (W, s1, s2 and the step's coefficients); vec = every pointer aligned
// for four-element vectors.
cudaError_t launch_owner(int op, int st, const float* G, const Params& p, int64_t n, bool vec,
                         int sms, cudaStream_t stream);

// The host-side checks forge_wgrad_adamw makes before any launch, including
// the alignment of X, W, m and v (dY is the caller's to check).
forge_status adamw_checks(const void* X, const void* dY, const float* W, const void* m,
                          const void* v, int64_t M, int64_t N, int64_t K, forge_dtype in_dtype,
                          forge_dtype state_dtype, float lr, float beta1, float beta2, float eps,
                          float wd, int64_t step);

}  // namespace forge
