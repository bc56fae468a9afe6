// forge_static_stage.h -- the per-device staging buffer of the
// no-allocation entry point (defined in forge_static_stage.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstddef>

namespace forge {

// Bytes in the buffer (the same on every device).
size_t static_stage_capacity();

// Device address of the buffer on device `dev` (the current device).  The
// first call per device resolves it with cudaGetSymbolAddress, which loads
// the module that holds the buffer; later calls return the cached address.
// Thread-safe.
cudaError_t static_stage_address(int dev, void** out);

}  // namespace forge
