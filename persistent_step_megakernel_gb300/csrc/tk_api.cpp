// C ABI of libtk: program creation (plan + device op table), workspace
// sizing, the checked launch boundary and status/resource queries.
//
// The boundary checks mirror trainkernel's runtime (page "trainkernel 0.1.0
// -- trainkernel/runtime.py", `CompiledProgram.run_into`): buffer counts,
// workspace size, in-place outputs bound to exactly their declared input, an
// in-place target not shared with another input, and no overlap between
// outputs, the workspace and inputs.  With raw pointers the check is on byte
// ranges instead of torch storages.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/tk.h"
#include "planner.h"
#include "tk_device.h"
#include "tk_kernel.h"

struct tk_program {
  tkp::Plan plan;
  tk_options opt{};
  int device = -1;
  int sm_count = 0;
  int grid = 1;
  size_t dyn_smem = 0;
  void* d_table = nullptr;
  const tkd::Program* d_prog = nullptr;
  // TMA descriptors of the last run and the base pointers they encode, and
  // the set before it (host-fed steps alternate between two batch buffers)
  std::vector<CUtensorMap> maps, maps_prev;
  std::vector<const void*> map_bases, map_bases_prev;
  // tk_run_host: the stream of the batch copies; events: copy into buffer k
  // done (0, 1), step reading buffer k done (2, 3), entry (4)
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  // optional per-stage stamps at the end of the workspace (float units)
  int64_t prof_offset = -1;
};

namespace {

thread_local std::string g_error;

tk_status fail(tk_status s, const std::string& msg) {
  g_error = msg.rfind("tk: ", 0) == 0 ? msg : "tk: " + msg;
  return s;
}

tk_status cuda_fail(cudaError_t e, const char* what) {
  return fail(TK_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Copy the plan's tables into one device allocation and patch the pointers.
tk_status upload(tk_program* p) {
  const tkp::Plan& pl = p->plan;
  size_t off_prog = 0;
  size_t off_stages = align_up(sizeof(tkd::Program), 64);
  size_t off_tasks = align_up(off_stages + pl.stages.size() * sizeof(tkd::Stage), 64);
  size_t off_code = align_up(off_tasks + pl.tasks.size() * sizeof(tkd::Task), 64);
  size_t off_refs = align_up(off_code + pl.code.size() * sizeof(tkd::Instr), 64);
  size_t off_pf = align_up(off_refs + pl.refs.size() * sizeof(tkd::Ref), 64);
  // L2 prefetch pieces: the op table, then the program inputs in order while
  // their total stays within the budget.
  std::vector<tkd::Prefetch> pf;
  auto add_range = [&](int32_t space, int32_t slot, int64_t bytes) {
    bytes &= ~int64_t(15);
    for (int64_t o = 0; o < bytes; o += tkd::kPrefetchPiece)
      pf.push_back({space, slot, o, std::min<int64_t>(tkd::kPrefetchPiece, bytes - o)});
  };
  int64_t in_total = 0;
  for (int64_t b : pl.input_bytes) in_total += b;
  const bool pf_inputs = in_total <= tkd::kPrefetchInputBudget;
  // room for every piece: the table's (+1 for the piece list itself) and each input's
  size_t max_pieces = size_t((off_pf + tkd::kPrefetchPiece - 1) / tkd::kPrefetchPiece) + 1;
  if (pf_inputs) max_pieces += size_t(in_total / tkd::kPrefetchPiece) + pl.input_bytes.size();
  size_t total = align_up(off_pf + max_pieces * sizeof(tkd::Prefetch), 64);
  add_range(tkd::SP_TABLE, 0, int64_t(total));
  if (pf_inputs)
    for (size_t i = 0; i < pl.input_bytes.size(); ++i) add_range(tkd::SP_IN, int32_t(i), pl.input_bytes[i]);
  if (pf.size() > max_pieces) return fail(TK_ERR_INVALID, "internal: prefetch list overflow");
  std::vector<unsigned char> host(total, 0);
  void* dev = nullptr;
  cudaError_t e = cudaMalloc(&dev, total);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(op table)");
  auto* base = static_cast<unsigned char*>(dev);
  tkd::Program prog{};
  prog.n_stages = int32_t(pl.stages.size());
  prog.n_tasks = int32_t(pl.tasks.size());
  prog.n_code = int32_t(pl.code.size());
  prog.n_refs = int32_t(pl.refs.size());
  prog.stages = reinterpret_cast<const tkd::Stage*>(base + off_stages);
  prog.tasks = reinterpret_cast<const tkd::Task*>(base + off_tasks);
  prog.code = reinterpret_cast<const tkd::Instr*>(base + off_code);
  prog.refs = reinterpret_cast<const tkd::Ref*>(base + off_refs);
  prog.n_prefetch = int32_t(pf.size());
  prog.prefetch = reinterpret_cast<const tkd::Prefetch*>(base + off_pf);
  std::memcpy(host.data() + off_prog, &prog, sizeof(prog));
  if (!pf.empty()) std::memcpy(host.data() + off_pf, pf.data(), pf.size() * sizeof(tkd::Prefetch));
  if (!pl.stages.empty()) std::memcpy(host.data() + off_stages, pl.stages.data(), pl.stages.size() * sizeof(tkd::Stage));
  if (!pl.tasks.empty()) std::memcpy(host.data() + off_tasks, pl.tasks.data(), pl.tasks.size() * sizeof(tkd::Task));
  if (!pl.code.empty()) std::memcpy(host.data() + off_code, pl.code.data(), pl.code.size() * sizeof(tkd::Instr));
  if (!pl.refs.empty()) std::memcpy(host.data() + off_refs, pl.refs.data(), pl.refs.size() * sizeof(tkd::Ref));
  e = cudaMemcpy(dev, host.data(), total, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(dev);
    return cuda_fail(e, "cudaMemcpy(op table)");
  }
  p->d_table = dev;
  p->d_prog = reinterpret_cast<const tkd::Program*>(base + off_prog);
  return TK_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, through the runtime's entry-point query.
EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Encode every TMA operand of the plan for these base pointers (cached).
tk_status encode_maps(tk_program* p, const void* const* inputs, void* const* outputs, float* ws) {
  const auto& ops = p->plan.tma;
  std::vector<const void*> bases(ops.size());
  for (size_t i = 0; i < ops.size(); ++i) {
    const auto& o = ops[i];
    bases[i] = o.space == tkd::SP_IN ? inputs[o.slot] : o.space == tkd::SP_OUT ? outputs[o.slot] : ws;
  }
  if (bases == p->map_bases && p->maps.size() == ops.size()) return TK_OK;
  if (bases == p->map_bases_prev && p->maps_prev.size() == ops.size()) {
    p->maps.swap(p->maps_prev);
    p->map_bases.swap(p->map_bases_prev);
    return TK_OK;
  }
  EncodeTiledFn fn = encoder();
  if (!fn) return fail(TK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  std::vector<CUtensorMap> maps(ops.size());
  for (size_t i = 0; i < ops.size(); ++i) {
    const auto& o = ops[i];
    char* addr = static_cast<char*>(const_cast<void*>(bases[i])) + o.base_elems * 2;
    // 2-D: (inner, outer).  3-D (MN-major slabs): (MN within a 64-wide slab,
    // K, slab), the slab dim stepping 128 bytes along the contiguous MN rows.
    const bool slabs = o.chunks > 0;
    cuuint64_t dims[3] = {cuuint64_t(o.inner), cuuint64_t(o.outer), 1};
    cuuint64_t strides[2] = {cuuint64_t(o.outer_stride) * 2, 128};
    cuuint32_t box[3] = {cuuint32_t(o.box_inner), cuuint32_t(o.box_outer), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (slabs) {
      dims[0] = 64;
      dims[2] = cuuint64_t(o.inner / 64);
      box[2] = cuuint32_t(o.chunks);
    }
    // GEMM operand tiles: 128-byte swizzle (the MMA descriptors' layout);
    // epilogue chunks (32 x 64 bytes): 64-byte swizzle (the staging layout)
    const CUtensorMapSwizzle sw = o.swizzle == 1 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    CUresult r = fn(&maps[i], o.dtype == TK_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    slabs ? 3 : 2, addr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(TK_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string(int(r)) + ")");
  }
  p->maps_prev.swap(p->maps);
  p->map_bases_prev.swap(p->map_bases);
  p->maps.swap(maps);
  p->map_bases.swap(bases);
  return TK_OK;
}

struct Range {
  uintptr_t lo, hi;
};
bool overlaps(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi; }
Range range_of(const void* p, int64_t bytes) {
  uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return {lo, lo + uintptr_t(bytes > 0 ? bytes : 0)};
}

}  // namespace

// Internal helpers for the built-in-workspace entry point (tk_static.cu).
tk_status tkapi_fail(tk_status s, const std::string& msg) { return fail(s, msg); }
int tkapi_device(const tk_program* p) { return p ? p->device : -1; }

extern "C" {

const char* tk_last_error(void) { return g_error.c_str(); }

void tk_options_default(tk_options* opt) {
  if (!opt) return;
  std::memset(opt, 0, sizeof(*opt));
  opt->blocks_per_sm = 1;
  opt->max_blocks = 0;
  opt->fuse_pointwise = 1;
  opt->fuse_epilogues = 1;
  opt->inline_input_casts = 1;
  opt->tensor_cores = 1;
  opt->sm_count = 0;
  opt->barrier_timeout_s = 2.0;
  opt->split_k = 1;
  opt->overlap_reductions = 1;
}

tk_status tk_program_create(const tk_program_desc* desc, const tk_options* opt_in, int device, tk_program** out) {
  if (!out) return fail(TK_ERR_INVALID, "out must not be NULL");
  *out = nullptr;
  if (!desc) return fail(TK_ERR_INVALID, "desc must not be NULL");
  tk_options opt;
  tk_options_default(&opt);
  if (opt_in) opt = *opt_in;
  if (opt.blocks_per_sm < 1 || opt.blocks_per_sm > 8) return fail(TK_ERR_INVALID, "blocks_per_sm must be between 1 and 8");
  if (opt.expr_forms < 0 || opt.expr_forms > 2) return fail(TK_ERR_INVALID, "expr_forms must be 0, 1 or 2");
  if (!(opt.barrier_timeout_s > 0.0) || opt.barrier_timeout_s > 3600.0)
    return fail(TK_ERR_INVALID, "barrier_timeout_s must be in (0, 3600]");
  if (opt.sm_count < 0) return fail(TK_ERR_INVALID, "sm_count must be >= 0");
  if (opt.tile_n != 0 && opt.tile_n != 64 && opt.tile_n != 128 && opt.tile_n != 224 && opt.tile_n != 256)
    return fail(TK_ERR_INVALID, "tile_n must be 0, 64, 128, 224 or 256");
  if (opt.epi_stage_bytes < 0) return fail(TK_ERR_INVALID, "epi_stage_bytes must be >= 0");
  if (opt.cta_pairs < 0 || opt.cta_pairs > 2) return fail(TK_ERR_INVALID, "cta_pairs must be 0, 1 or 2");
  if (opt.overlap_reductions < 0 || opt.overlap_reductions > 2)
    return fail(TK_ERR_INVALID, "overlap_reductions must be 0, 1 or 2");

  int sms = opt.sm_count > 0 ? opt.sm_count : 152;
  if (device >= 0) {
    DeviceGuard g(device);
    if (!g.ok) return fail(TK_ERR_DEVICE, "cannot select CUDA device " + std::to_string(device));
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3)
      return fail(TK_ERR_DEVICE, "this build targets sm_103a (GB300); device is sm_" + std::to_string(prop.major) +
                                     std::to_string(prop.minor));
    if (!prop.cooperativeLaunch) return fail(TK_ERR_DEVICE, "device does not support cooperative launch");
    if (opt.sm_count == 0) sms = prop.multiProcessorCount;
  } else if (device != -1) {
    return fail(TK_ERR_INVALID, "device must be a CUDA ordinal or -1");
  }

  auto* p = new (std::nothrow) tk_program();
  if (!p) return fail(TK_ERR_INVALID, "out of host memory");
  try {
    p->plan = tkp::build_plan(*desc, opt, sms);
  } catch (const tkp::Error& e) {
    delete p;
    return fail(e.status, e.what());
  } catch (const std::exception& e) {
    delete p;
    return fail(TK_ERR_INVALID, e.what());
  }
  p->opt = opt;
  p->device = device;
  p->sm_count = sms;
  p->dyn_smem = p->plan.smem_bytes;
  int occupancy = 1;
  if (device >= 0) {
    DeviceGuard g(device);
    cudaError_t e = tk_kernel_prepare(p->plan.uses_tc, p->dyn_smem);
    if (e == cudaSuccess) e = tk_kernel_occupancy(&occupancy, p->plan.uses_tc, p->dyn_smem);
    if (e != cudaSuccess) {
      delete p;
      return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    }
    if (occupancy < 1) {
      delete p;
      return fail(TK_ERR_DEVICE, "kernel has no resident blocks");
    }
    tk_status s = upload(p);
    if (s != TK_OK) {
      delete p;
      return s;
    }
  }
  int64_t grid = int64_t(sms) * std::min(occupancy, opt.blocks_per_sm);
  grid = std::min<int64_t>(grid, p->plan.max_items);
  if (opt.max_blocks > 0) grid = std::min<int64_t>(grid, opt.max_blocks);
  if (p->plan.pair) {
    // one block per SM in clusters of two: an even grid of resident clusters
    int clusters = int(sms / 2);
    if (device >= 0) {
      DeviceGuard g(device);
      cudaError_t e = tk_kernel_pair_clusters(&clusters, p->dyn_smem, p->plan.pair);
      if (e != cudaSuccess) {
        tk_program_destroy(p);
        return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
      }
    }
    grid = std::min<int64_t>({int64_t(sms), grid + (grid & 1), 2 * int64_t(clusters)}) & ~int64_t(1);
    if (grid < 2) {
      tk_program_destroy(p);
      return fail(TK_ERR_DEVICE, "no two-block cluster fits on the device");
    }
  }
  p->grid = int(std::max<int64_t>(grid, 1));
  p->plan.stats.grid_blocks = p->grid;
  if (opt.profile) {
    p->prof_offset = p->plan.workspace_units;
    int64_t units = int64_t(p->plan.stages.size()) * p->grid * 2 * tkd::kProfStamps;  // int64 stamps
    p->plan.workspace_units += (units + 63) / 64 * 64;
    p->plan.stats.workspace_elements = p->plan.workspace_units;
  }
  *out = p;
  return TK_OK;
}

void tk_program_destroy(tk_program* p) {
  if (!p) return;
  if (p->d_table || p->copy_stream) {
    DeviceGuard g(p->device);
    if (p->d_table) cudaFree(p->d_table);
    for (cudaEvent_t e : p->ev)
      if (e) cudaEventDestroy(e);
    if (p->copy_stream) cudaStreamDestroy(p->copy_stream);
  }
  delete p;
}

tk_status tk_allocate(const tk_program* p, size_t* n) {
  if (!p || !n) return fail(TK_ERR_INVALID, "program and workspace_elements must not be NULL");
  *n = size_t(std::max<int64_t>(p->plan.workspace_units, 1));
  return TK_OK;
}

tk_status tk_workspace_init(const tk_program* p, float* ws, size_t n, void* stream) {
  if (!p) return fail(TK_ERR_INVALID, "program must not be NULL");
  if (p->device < 0) return fail(TK_ERR_DEVICE, "plan-only program (created with device -1)");
  if (!ws || n < size_t(p->plan.workspace_units))
    return fail(TK_ERR_WORKSPACE, "workspace does not match compiled requirements");
  DeviceGuard g(p->device);
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(tkd::Header), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace header)");
  return TK_OK;
}

namespace {

// Host-side checks of one step's buffers (tk_run's error contract).
tk_status check_run(const tk_program* p, const void* const* inputs, int32_t n_inputs, void* const* outputs,
                    int32_t n_outputs, const float* ws, size_t ws_elems) {
  if (!p) return fail(TK_ERR_INVALID, "program must not be NULL");
  if (p->device < 0) return fail(TK_ERR_DEVICE, "plan-only program (created with device -1)");
  const tkp::Plan& pl = p->plan;
  if (n_inputs != int32_t(pl.input_bytes.size()))
    return fail(TK_ERR_INVALID, "expected " + std::to_string(pl.input_bytes.size()) + " inputs, got " +
                                    std::to_string(n_inputs));
  if (n_outputs != int32_t(pl.output_bytes.size())) return fail(TK_ERR_INVALID, "incorrect output buffer count");
  if ((n_inputs && !inputs) || (n_outputs && !outputs)) return fail(TK_ERR_INVALID, "NULL buffer array");
  if (!ws || ws_elems < size_t(pl.workspace_units))
    return fail(TK_ERR_WORKSPACE, "workspace does not match compiled requirements");
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return fail(TK_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  for (int i = 0; i < n_inputs; ++i) {
    if (pl.input_bytes[i] > 0 && !inputs[i]) return fail(TK_ERR_INVALID, "input " + std::to_string(i) + " is NULL");
    if (reinterpret_cast<uintptr_t>(inputs[i]) % 16) return fail(TK_ERR_INVALID, "input pointers must be 16-byte aligned");
  }
  for (int j = 0; j < n_outputs; ++j) {
    if (pl.output_bytes[j] > 0 && !outputs[j]) return fail(TK_ERR_INVALID, "output " + std::to_string(j) + " is NULL");
    if (reinterpret_cast<uintptr_t>(outputs[j]) % 16) return fail(TK_ERR_INVALID, "output pointers must be 16-byte aligned");
  }
  // In-place outputs bind exactly their declared input; nothing else may overlap.
  std::vector<bool> is_inplace(n_outputs, false), is_target(n_inputs, false);
  for (const auto& kv : pl.inplace) {
    if (outputs[kv.first] != inputs[kv.second])
      return fail(TK_ERR_ALIAS, "inplace output must bind its declared input");
    is_inplace[kv.first] = true;
    is_target[kv.second] = true;
  }
  for (int i = 0; i < n_inputs; ++i) {
    if (!is_target[i] || pl.input_bytes[i] == 0) continue;
    Range t = range_of(inputs[i], pl.input_bytes[i]);
    for (int k = 0; k < n_inputs; ++k)
      if (k != i && overlaps(t, range_of(inputs[k], pl.input_bytes[k])))
        return fail(TK_ERR_ALIAS, "inplace target must not alias another input");
  }
  Range wsr = range_of(ws, int64_t(pl.workspace_units) * 4);
  std::vector<Range> written = {wsr};
  for (int j = 0; j < n_outputs; ++j)
    if (!is_inplace[j]) written.push_back(range_of(outputs[j], pl.output_bytes[j]));
  for (size_t a = 0; a < written.size(); ++a) {
    for (size_t b = a + 1; b < written.size(); ++b)
      if (overlaps(written[a], written[b])) return fail(TK_ERR_ALIAS, "execution buffers must not alias inputs or each other");
    for (int i = 0; i < n_inputs; ++i)
      if (overlaps(written[a], range_of(inputs[i], pl.input_bytes[i])))
        return fail(TK_ERR_ALIAS, "execution buffers must not alias inputs or each other");
  }
  return TK_OK;
}

// Launch one checked step on `stream`.
tk_status launch_run(tk_program* p, const void* const* inputs, int32_t n_inputs, void* const* outputs,
                     int32_t n_outputs, float* ws, void* stream) {
  const tkp::Plan& pl = p->plan;
  tkd::Params prm{};
  prm.prog = p->d_prog;
  prm.ws = reinterpret_cast<char*>(ws);
  prm.timeout_ns = static_cast<long long>(p->opt.barrier_timeout_s * 1e9);
  prm.prof = p->prof_offset >= 0 ? reinterpret_cast<long long*>(ws + p->prof_offset) : nullptr;
  prm.ring_stage_bytes = pl.ring_stage_bytes;
  prm.tmem_cols = pl.tmem_cols;
  prm.epi_warp_bytes = pl.epi_warp_bytes;
  prm.n_in = n_inputs;
  prm.n_out = n_outputs;
  for (int i = 0; i < n_inputs; ++i) prm.io[i] = const_cast<void*>(inputs[i]);
  for (int j = 0; j < n_outputs; ++j) prm.io[tkd::kMaxIO + j] = outputs[j];
  DeviceGuard g(p->device);
  const void* maps = nullptr;
  if (p->plan.uses_tc) {
    tk_status s = encode_maps(p, inputs, outputs, ws);
    if (s != TK_OK) return s;
    maps = p->maps.data();
    prm.n_maps = int(p->maps.size());
  }
  cudaError_t e = tk_kernel_launch(prm, maps, int(p->maps.size()), p->grid, p->dyn_smem,
                                   static_cast<cudaStream_t>(stream), p->plan.pair);
  if (e != cudaSuccess) return cuda_fail(e, "cooperative launch");
  return TK_OK;
}

}  // namespace

tk_status tk_run(tk_program* p, const void* const* inputs, int32_t n_inputs, void* const* outputs, int32_t n_outputs,
                 float* ws, size_t ws_elems, void* stream) {
  tk_status s = check_run(p, inputs, n_inputs, outputs, n_outputs, ws, ws_elems);
  if (s != TK_OK) return s;
  return launch_run(p, inputs, n_inputs, outputs, n_outputs, ws, stream);
}

tk_status tk_run_host(tk_program* p, int32_t n_steps, const void* const* inputs, int32_t n_inputs,
                      void* const* outputs, int32_t n_outputs, const int32_t* batch, int32_t n_batch,
                      void* const* batch_alt, const void* const* host_batches, const int32_t* results,
                      int32_t n_results, void* const* host_results, float* ws, size_t ws_elems, void* stream) {
  tk_status st = check_run(p, inputs, n_inputs, outputs, n_outputs, ws, ws_elems);
  if (st != TK_OK) return st;
  const tkp::Plan& pl = p->plan;
  if (n_steps < 0 || n_batch < 0 || n_results < 0) return fail(TK_ERR_INVALID, "negative count");
  if (n_batch > n_inputs) return fail(TK_ERR_INVALID, "more batch inputs than inputs");
  if ((n_batch && (!batch || !batch_alt)) || (n_steps && n_batch && !host_batches) ||
      (n_results && !results) || (n_steps && n_results && !host_results))
    return fail(TK_ERR_INVALID, "NULL array");
  std::vector<const void*> odd(inputs, inputs + n_inputs);
  std::vector<Range> alt;
  for (int b = 0; b < n_batch; ++b) {
    const int i = batch[b];
    if (i < 0 || i >= n_inputs) return fail(TK_ERR_INVALID, "batch index " + std::to_string(i) + " out of range");
    for (int c = 0; c < b; ++c)
      if (batch[c] == i) return fail(TK_ERR_INVALID, "batch input " + std::to_string(i) + " listed twice");
    for (const auto& kv : pl.inplace)
      if (kv.second == i) return fail(TK_ERR_INVALID, "batch input " + std::to_string(i) + " is an in-place target");
    if (pl.input_bytes[i] > 0 && !batch_alt[b]) return fail(TK_ERR_INVALID, "batch_alt buffer is NULL");
    if (reinterpret_cast<uintptr_t>(batch_alt[b]) % 16) return fail(TK_ERR_INVALID, "batch_alt pointers must be 16-byte aligned");
    for (int s = 0; s < n_steps; ++s)
      if (pl.input_bytes[i] > 0 && !host_batches[size_t(s) * n_batch + b])
        return fail(TK_ERR_INVALID, "host batch of step " + std::to_string(s) + " is NULL");
    odd[i] = batch_alt[b];
    alt.push_back(range_of(batch_alt[b], pl.input_bytes[i]));
  }
  // the odd steps' buffers pass the same checks, and no second buffer overlaps
  // a buffer of the even steps
  st = check_run(p, odd.data(), n_inputs, outputs, n_outputs, ws, ws_elems);
  if (st != TK_OK) return st;
  for (const Range& r : alt)
    for (int i = 0; i < n_inputs; ++i)
      if (overlaps(r, range_of(inputs[i], pl.input_bytes[i])))
        return fail(TK_ERR_ALIAS, "batch_alt buffers must not overlap another buffer");
  for (int r = 0; r < n_results; ++r) {
    if (results[r] < 0 || results[r] >= n_outputs) return fail(TK_ERR_INVALID, "result index out of range");
    for (int s = 0; s < n_steps; ++s)
      if (pl.output_bytes[results[r]] > 0 && !host_results[size_t(s) * n_results + r])
        return fail(TK_ERR_INVALID, "host result of step " + std::to_string(s) + " is NULL");
  }
  if (n_steps == 0) return TK_OK;

  DeviceGuard g(p->device);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (n_batch && !p->copy_stream) {
    e = cudaStreamCreateWithFlags(&p->copy_stream, cudaStreamNonBlocking);
    for (int k = 0; k < 5 && e == cudaSuccess; ++k) e = cudaEventCreateWithFlags(&p->ev[k], cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "creating the batch copy stream");
  }
  const cudaStream_t xs = p->copy_stream;
  auto copy_batch = [&](int s) -> cudaError_t {
    const int k = s & 1;
    cudaError_t r = cudaSuccess;
    // buffer k was last read by step s - 2
    if (s >= 2) r = cudaStreamWaitEvent(xs, p->ev[2 + k], 0);
    for (int b = 0; b < n_batch && r == cudaSuccess; ++b) {
      const int i = batch[b];
      if (pl.input_bytes[i] == 0) continue;
      void* dst = const_cast<void*>(k ? odd[i] : inputs[i]);
      r = cudaMemcpyAsync(dst, host_batches[size_t(s) * n_batch + b], size_t(pl.input_bytes[i]),
                          cudaMemcpyHostToDevice, xs);
    }
    if (r == cudaSuccess) r = cudaEventRecord(p->ev[k], xs);
    return r;
  };
  if (n_batch) {
    // the first copies wait for the work already on `stream` (which may read
    // either buffer)
    e = cudaEventRecord(p->ev[4], cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(xs, p->ev[4], 0);
    if (e == cudaSuccess) e = copy_batch(0);
    if (e != cudaSuccess) return cuda_fail(e, "enqueueing the first batch copy");
  }
  for (int s = 0; s < n_steps; ++s) {
    const int k = s & 1;
    if (n_batch) {
      if (s + 1 < n_steps) {
        e = copy_batch(s + 1);
        if (e != cudaSuccess) return cuda_fail(e, "enqueueing a batch copy");
      }
      e = cudaStreamWaitEvent(cs, p->ev[k], 0);
      if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
    }
    st = launch_run(p, k ? odd.data() : inputs, n_inputs, outputs, n_outputs, ws, stream);
    if (st != TK_OK) return st;
    if (n_batch) {
      e = cudaEventRecord(p->ev[2 + k], cs);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    }
    for (int r = 0; r < n_results; ++r) {
      const int j = results[r];
      if (pl.output_bytes[j] == 0) continue;
      e = cudaMemcpyAsync(host_results[size_t(s) * n_results + r], outputs[j], size_t(pl.output_bytes[j]),
                          cudaMemcpyDeviceToHost, cs);
      if (e != cudaSuccess) return cuda_fail(e, "enqueueing a result copy");
    }
  }
  return TK_OK;
}

tk_status tk_run_status(const tk_program* p, const float* ws, void* stream, int32_t* device_status, int32_t* stage) {
  if (!p || !ws || !device_status) return fail(TK_ERR_INVALID, "program, workspace and device_status must not be NULL");
  if (p->device < 0) return fail(TK_ERR_DEVICE, "plan-only program (created with device -1)");
  DeviceGuard g(p->device);
  int32_t h[4] = {0, 0, 0, 0};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the workspace header");
  *device_status = h[2];
  if (stage) *stage = h[3];
  return TK_OK;
}

tk_status tk_resource_usage(const tk_program* p, int64_t out[4]) {
  if (!p || !out) return fail(TK_ERR_INVALID, "program and out must not be NULL");
  if (p->device < 0) return fail(TK_ERR_DEVICE, "plan-only program (created with device -1)");
  DeviceGuard g(p->device);
  cudaFuncAttributes a;
  cudaError_t e = tk_kernel_attributes(&a, p->plan.uses_tc, p->plan.pair);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes");
  int occ = 0;
  e = tk_kernel_occupancy(&occ, p->plan.uses_tc, p->dyn_smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  out[0] = a.numRegs;
  out[1] = int64_t(a.localSizeBytes);
  out[2] = int64_t(a.sharedSizeBytes) + int64_t(p->dyn_smem);
  out[3] = occ;
  return TK_OK;
}

tk_status tk_profile_read(const tk_program* p, const float* ws, void* stream, int64_t* stamps, size_t n) {
  if (!p || !ws || !stamps) return fail(TK_ERR_INVALID, "program, workspace and stamps must not be NULL");
  if (p->device < 0) return fail(TK_ERR_DEVICE, "plan-only program (created with device -1)");
  if (p->prof_offset < 0) return fail(TK_ERR_INVALID, "program was created without profile = 1");
  size_t need = size_t(tkd::kProfStamps) * p->plan.stages.size() * size_t(p->grid);
  if (n < need) return fail(TK_ERR_INVALID, "stamps array too small: need " + std::to_string(need));
  DeviceGuard g(p->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(stamps, ws + p->prof_offset, need * sizeof(int64_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading profile stamps");
  return TK_OK;
}

tk_status tk_plan_stats_get(const tk_program* p, tk_plan_stats* s) {
  if (!p || !s) return fail(TK_ERR_INVALID, "program and stats must not be NULL");
  *s = p->plan.stats;
  return TK_OK;
}

tk_status tk_plan_task(const tk_program* p, int32_t index, tk_task_info* info) {
  if (!p || !info) return fail(TK_ERR_INVALID, "program and info must not be NULL");
  if (index < 0 || size_t(index) >= p->plan.tasks.size()) return fail(TK_ERR_INVALID, "task index out of range");
  const tkd::Task& t = p->plan.tasks[size_t(index)];
  tk_task_info r{};
  r.stage = t.stage;
  r.kind = t.kind;
  r.op_index = t.op_index;
  r.n_items = t.n_items;
  r.form = !t.chain.valid ? 0 : (t.chain.fast != tkd::FK_NONE ? 2 : 1);
  r.compiled_shape = r.form == 2 ? t.chain.fast : 0;
  const bool gemm = t.kind == tkd::T_GEMM_SIMT || t.kind == tkd::T_GEMM_TC;
  if (gemm) {
    r.m = t.m;
    r.n = t.n;
    r.k = t.k;
    r.tile_m = t.tile_m;
    r.tile_n = t.tile_n;
  }
  r.parts = t.parts > 0 ? t.parts : 1;
  r.staged_epilogue = t.epi_stage != 0;
  r.side_output = t.has_side != 0;
  r.staged_depth = t.epi_stage ? t.epi_depth + ((t.epi_stage & 16) ? 16 : 0) : 0;
  r.beside_tiles = t.bg != 0;
  r.folded = t.folded != 0;
  r.numel = t.numel;
  *info = r;
  return TK_OK;
}

}  // extern "C"
