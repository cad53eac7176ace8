// Entry point of the persistent kernel for programs without tensor-core GEMMs.
#include "megakernel.cuh"
#include "tk_kernel.h"

namespace tkk {
__global__ void __launch_bounds__(kThreads, 1) tk_persistent(const __grid_constant__ Params p) {
  persistent_body<0>(p, nullptr);
}
}  // namespace tkk

const void* tk_kernel_fn_plain() { return reinterpret_cast<const void*>(&tkk::tk_persistent); }
