// Host helpers shared by the TMA kernels: encoded tensor maps (cached per
// device, base pointer and shape, so a repeated call with the same tensors
// encodes nothing) and the dynamic shared-memory opt-in of a kernel (set once
// per device).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssa {

// A bf16 tensor map of rank 2 or 3 with the 128-byte swizzle: dims[0] is the
// contiguous dimension (elements), strides[i] the byte stride of dims[i + 1],
// box the tile a copy moves. Rows outside a dimension read as zeros. Returns
// false when the driver rejects the map.
bool tmap_bf16_sw128(CUtensorMap* out, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for `func` on the current
// device, done once per (function, device).
cudaError_t set_max_dyn_smem(const void* func, int bytes);

}  // namespace ssa
