// Host entry points into the kernel translation unit.
#pragma once

#include <cuda_runtime.h>

#include "tk_device.h"

// Cooperative launch of the persistent kernel on `stream`.
cudaError_t tk_kernel_launch(const tkd::Params& params, int grid, size_t dyn_smem, cudaStream_t stream);
// Resident blocks per SM for the given dynamic shared memory.
cudaError_t tk_kernel_occupancy(int* blocks_per_sm, size_t dyn_smem);
// Compiler resource attributes of the kernel.
cudaError_t tk_kernel_attributes(cudaFuncAttributes* attr);
