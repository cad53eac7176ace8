// tk_run_static: run a step with a workspace that lives inside this library
// instead of one the caller allocates.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they run a step -- code running inside a CUDA stream capture that must not
// add allocation calls, runtimes whose memory is fully pre-reserved by another
// allocator (so a cudaMalloc would fail or fragment it), and embedders that
// are only handed raw input/output pointers by a host framework that owns all
// allocations.  They still pass their own inputs and outputs; only the scratch
// memory (barrier counters, intermediate values, reduction partials) comes from
// the array below.
//
// The array is a file-scope static device variable, so every GPU on which this
// library's device code is loaded holds TK_STATIC_WORKSPACE_ELEMENTS floats
// (8 MiB) of it until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/tk.h"
#include "tk_device.h"

// Defined in tk_api.cpp: record the message tk_last_error() returns; the
// program's device ordinal.
tk_status tkapi_fail(tk_status s, const std::string& msg);
int tkapi_device(const tk_program* p);

// The built-in workspace.  In host code this name is only a stand-in; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float tk_static_workspace[TK_STATIC_WORKSPACE_ELEMENTS];

namespace {

constexpr int kMaxDevices = 256;
std::mutex g_mutex;
// Device address of the array, per device, with the context it was looked up
// in: a device reset (or a torn-down and recreated primary context) gives the
// device a new context, in which the old address is meaningless.
struct Slot {
  CUcontext ctx = nullptr;
  void* address = nullptr;
};
Slot g_slot[kMaxDevices];

// cuCtxGetCurrent from the driver, through the runtime's entry-point query
// (the library does not link the driver library directly).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(p);
    return static_cast<CtxGetCurrentFn>(nullptr);
  }();
  return fn;
}

}  // namespace

extern "C" tk_status tk_run_static(tk_program* program, const void* const* inputs, int32_t n_inputs,
                                   void* const* outputs, int32_t n_outputs, void* stream) {
  if (!program) return tkapi_fail(TK_ERR_INVALID, "program must not be NULL");
  const int device = tkapi_device(program);
  if (device < 0) return tkapi_fail(TK_ERR_DEVICE, "plan-only program (created with device -1)");
  if (device >= kMaxDevices) return tkapi_fail(TK_ERR_DEVICE, "device ordinal out of range");
  size_t need = 0;
  tk_status s = tk_allocate(program, &need);
  if (s != TK_OK) return s;
  if (need > size_t(TK_STATIC_WORKSPACE_ELEMENTS))
    return tkapi_fail(TK_ERR_WORKSPACE, "tk_run_static: this program needs a workspace of " + std::to_string(need) +
                                            " float elements but the built-in one holds " +
                                            std::to_string(TK_STATIC_WORKSPACE_ELEMENTS) +
                                            " (8 MiB); use tk_run with a caller-allocated workspace");

  // Set-up, once per device (and again if the device's context changed): the
  // host-side name of the array is not a device address, so look the address
  // up with that device current.
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    cudaError_t e = cudaSetDevice(device);
    CUcontext ctx = nullptr;
    CtxGetCurrentFn get = ctx_get_current();
    if (e == cudaSuccess && (!get || get(&ctx) != CUDA_SUCCESS)) e = cudaErrorUnknown;
    Slot& slot = g_slot[device];
    if (e == cudaSuccess && (!slot.address || slot.ctx != ctx)) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, tk_static_workspace);
      if (e == cudaSuccess) {
        slot.address = ptr;
        slot.ctx = ctx;
      }
    }
    if (prev >= 0 && prev != device) cudaSetDevice(prev);
    if (e != cudaSuccess)
      return tkapi_fail(TK_ERR_CUDA,
                        std::string("set-up of the built-in workspace (cudaGetSymbolAddress): ") + cudaGetErrorString(e));
    ws = slot.address;
  }

  // The array keeps whatever the previous call left; the header (barrier
  // counter, status word) must start at zero for every run.
  s = tk_workspace_init(program, static_cast<float*>(ws), TK_STATIC_WORKSPACE_ELEMENTS, stream);
  if (s != TK_OK) return s;
  return tk_run(program, inputs, n_inputs, outputs, n_outputs, static_cast<float*>(ws),
                TK_STATIC_WORKSPACE_ELEMENTS, stream);
}
