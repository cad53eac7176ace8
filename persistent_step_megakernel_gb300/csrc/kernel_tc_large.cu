// Entry point of the persistent kernel for programs with tensor-core GEMMs
// (up to kMaxMaps TMA descriptors).
#include "megakernel.cuh"
#include "tk_kernel.h"

namespace tkk {
__global__ void __launch_bounds__(kThreads, 1) tk_persistent_tc_large(const __grid_constant__ ParamsTc<kMaxMaps> p) {
  persistent_body<0>(p.p, p.maps);
}
}  // namespace tkk

const void* tk_kernel_fn_tc_large() { return reinterpret_cast<const void*>(&tkk::tk_persistent_tc_large); }
