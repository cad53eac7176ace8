// Entry point of the persistent kernel for pair-tile programs: clusters of two
// blocks, every tensor-core GEMM on 256-row tiles of cta_group::2 MMAs (up to
// kMaxMaps TMA descriptors).
#include "megakernel.cuh"
#include "tk_kernel.h"

namespace tkk {
__global__ void __launch_bounds__(kThreads, 1) tk_persistent_tc_pair(const __grid_constant__ ParamsTc<kMaxMaps> p) {
  persistent_body<1>(p.p, p.maps);
}
}  // namespace tkk

const void* tk_kernel_fn_tc_pair() { return reinterpret_cast<const void*>(&tkk::tk_persistent_tc_pair); }
