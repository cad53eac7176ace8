// Host entry points into the kernel translation unit.
#pragma once

#include <cuda_runtime.h>

#include "tk_device.h"

// Cooperative launch of the persistent kernel on `stream`; `maps` (n_maps
// CUtensorMap objects) selects the tensor-core variant when non-NULL.
cudaError_t tk_kernel_launch(const tkd::Params& params, const void* maps, int n_maps, int grid, size_t dyn_smem,
                             cudaStream_t stream);
// One-time per-device setup (dynamic shared memory limit of the variant).
cudaError_t tk_kernel_prepare(bool tc, size_t dyn_smem);
// Resident blocks per SM for the variant and dynamic shared memory.
cudaError_t tk_kernel_occupancy(int* blocks_per_sm, bool tc, size_t dyn_smem);
// Compiler resource attributes of the variant.
cudaError_t tk_kernel_attributes(cudaFuncAttributes* attr, bool tc);
