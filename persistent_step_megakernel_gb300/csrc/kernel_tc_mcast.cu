// Entry point of the persistent kernel for shared-B pair-tile programs: clusters
// of two blocks, each running its own 128-row MMAs on B tiles multicast to both
// (up to kMaxMaps TMA descriptors).
#include "megakernel.cuh"
#include "tk_kernel.h"

namespace tkk {
__global__ void __launch_bounds__(kThreads, 1) tk_persistent_tc_mcast(const __grid_constant__ ParamsTc<kMaxMaps> p) {
  persistent_body<2>(p.p, p.maps);
}
}  // namespace tkk

const void* tk_kernel_fn_tc_mcast() { return reinterpret_cast<const void*>(&tkk::tk_persistent_tc_mcast); }
