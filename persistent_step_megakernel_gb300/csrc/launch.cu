// Host side of the persistent kernel: launch, setup and queries.
//
// Each launch is one cooperative launch (all blocks resident, so the
// in-kernel grid barrier cannot deadlock).  The tensor-core variants take the
// TMA descriptors as __grid_constant__ parameters.
#include <cstring>
#include <mutex>

#include "tk_kernel.h"

namespace {

constexpr int kMaxDevices = 64;
enum Variant { V_PLAIN = 0, V_TC_SMALL = 1, V_TC_LARGE = 2, V_TC_PAIR = 3, V_TC_MCAST = 4, V_COUNT = 5 };

const void* kernel_of(int v) {
  return v == V_PLAIN      ? tk_kernel_fn_plain()
         : v == V_TC_SMALL ? tk_kernel_fn_tc_small()
         : v == V_TC_LARGE ? tk_kernel_fn_tc_large()
         : v == V_TC_PAIR  ? tk_kernel_fn_tc_pair()
                           : tk_kernel_fn_tc_mcast();
}

int pair_variant(int pair) { return pair == 1 ? V_TC_PAIR : V_TC_MCAST; }

// Per device and variant: the kernel's static shared memory (read once) and
// the shared-memory carveout last applied.  Function attributes belong to a
// device's context, so each device keeps its own record.
struct VariantState {
  bool known = false;
  size_t static_smem = 0;
  int carveout = -1;
};
std::mutex g_mutex;
VariantState g_state[kMaxDevices][V_COUNT];

// Shared-memory carveout: ask for just the shared memory a launch needs so the
// rest of the SM's unified L1/shared array stays L1 cache (operand loads and
// spilled registers hit it).  Applied only when it changes for this device.
cudaError_t set_carveout(int v, size_t dyn_smem) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  VariantState& st = g_state[dev][v];
  if (!st.known) {
    cudaFuncAttributes a;
    e = cudaFuncGetAttributes(&a, kernel_of(v));
    if (e != cudaSuccess) return e;
    st.static_smem = a.sharedSizeBytes;
    st.known = true;
  }
  const size_t need = dyn_smem + st.static_smem + 1024;
  int pct = int((need * 100 + 233471) / 233472) + 1;  // of the largest carveout (228 KB)
  pct = pct > 100 ? 100 : pct;
  if (pct == st.carveout) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel_of(v), cudaFuncAttributePreferredSharedMemoryCarveout, pct);
  if (e == cudaSuccess) st.carveout = pct;
  return e;
}

template <int NM>
cudaError_t launch_tc(const cudaLaunchConfig_t* cfg, const void* fn, const tkd::Params& params, const void* maps,
                      int n_maps) {
  static thread_local tkd::ParamsTc<NM> big;
  big.p = params;
  memcpy(big.maps, maps, size_t(n_maps) * sizeof(CUtensorMap));
  void* args[1] = {&big};
  return cudaLaunchKernelExC(cfg, fn, args);
}

}  // namespace

cudaError_t tk_kernel_launch(const tkd::Params& params, const void* maps, int n_maps, int grid, size_t dyn_smem,
                             cudaStream_t stream, int pair) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(tkd::kThreads);
  cfg.dynamicSmemBytes = dyn_smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pair ? 2 : 1;
  if (pair && (!maps || grid % 2)) return cudaErrorInvalidValue;
  const int v = !maps ? V_PLAIN : pair ? pair_variant(pair) : n_maps <= tkd::kSmallMaps ? V_TC_SMALL : V_TC_LARGE;
  if (maps && n_maps > tkd::kMaxMaps) return cudaErrorInvalidValue;
  cudaError_t e = set_carveout(v, dyn_smem);
  if (e != cudaSuccess) return e;
  if (v == V_PLAIN) {
    tkd::Params p = params;
    void* args[1] = {&p};
    return cudaLaunchKernelExC(&cfg, kernel_of(v), args);
  }
  if (v == V_TC_SMALL) return launch_tc<tkd::kSmallMaps>(&cfg, kernel_of(v), params, maps, n_maps);
  return launch_tc<tkd::kMaxMaps>(&cfg, kernel_of(v), params, maps, n_maps);
}

cudaError_t tk_kernel_pair_clusters(int* clusters, size_t dyn_smem, int pair) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(tkd::kThreads);
  cfg.dynamicSmemBytes = dyn_smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = set_carveout(pair_variant(pair), dyn_smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveClusters(clusters, kernel_of(pair_variant(pair)), &cfg);
}

// The dynamic shared-memory limit is raised to the largest any program uses,
// so programs of different sizes can be launched in any order.  Called for
// every program, with the program's device current.
cudaError_t tk_kernel_prepare(bool tc, size_t) {
  if (!tc) return cudaSuccess;
  for (int v : {V_TC_SMALL, V_TC_LARGE, V_TC_PAIR, V_TC_MCAST}) {
    cudaError_t e = cudaFuncSetAttribute(kernel_of(v), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tkd::kDynSmemBudget);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t tk_kernel_occupancy(int* blocks_per_sm, bool tc, size_t dyn_smem) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, kernel_of(tc ? V_TC_LARGE : V_PLAIN),
                                                       tkd::kThreads, dyn_smem);
}

cudaError_t tk_kernel_attributes(cudaFuncAttributes* attr, bool tc, int pair) {
  return cudaFuncGetAttributes(attr, kernel_of(!tc ? V_PLAIN : pair ? pair_variant(pair) : V_TC_LARGE));
}
