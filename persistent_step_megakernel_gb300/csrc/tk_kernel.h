// Host entry points into the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "tk_device.h"

namespace tkd {

// Parameters of the tensor-core variants: the TMA descriptors travel by value
// as __grid_constant__ kernel parameters.  Two capacities keep the parameter
// block small for programs with few GEMMs.
constexpr int kSmallMaps = 32;

template <int NM>
struct ParamsTc {
  Params p;
  CUtensorMap maps[NM];
};

}  // namespace tkd

// The four entry points (host stubs), one per translation unit.
const void* tk_kernel_fn_plain();      // kernel_plain.cu
const void* tk_kernel_fn_tc_small();   // kernel_tc_small.cu: up to kSmallMaps descriptors
const void* tk_kernel_fn_tc_large();   // kernel_tc_large.cu: up to kMaxMaps descriptors
const void* tk_kernel_fn_tc_pair();    // kernel_tc_pair.cu: pair tiles, up to kMaxMaps descriptors
const void* tk_kernel_fn_tc_mcast();   // kernel_tc_mcast.cu: shared-B pair tiles, up to kMaxMaps descriptors

// Cooperative launch of the persistent kernel on `stream`; `maps` (n_maps
// CUtensorMap objects) selects a tensor-core variant when non-NULL, `pair` a
// pair-tile variant (clusters of two blocks; grid even): 1 cta_group::2 MMAs,
// 2 B shared by multicast.
cudaError_t tk_kernel_launch(const tkd::Params& params, const void* maps, int n_maps, int grid, size_t dyn_smem,
                             cudaStream_t stream, int pair);
// Setup on the current device (dynamic shared memory limit of the variants).
cudaError_t tk_kernel_prepare(bool tc, size_t dyn_smem);
// Resident blocks per SM for the variant and dynamic shared memory.
cudaError_t tk_kernel_occupancy(int* blocks_per_sm, bool tc, size_t dyn_smem);
// Clusters of two blocks of a pair-tile variant that can be resident at once.
cudaError_t tk_kernel_pair_clusters(int* clusters, size_t dyn_smem, int pair);
// Compiler resource attributes of the variant.
cudaError_t tk_kernel_attributes(cudaFuncAttributes* attr, bool tc, int pair);
