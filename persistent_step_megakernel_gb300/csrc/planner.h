// Host planner: turns a tk_program_desc into the device op table.
#pragma once

#include <stdexcept>
#include <string>
#include <vector>

#include "../../include/tk.h"
#include "tk_device.h"

namespace tkp {

struct Error : std::runtime_error {
  tk_status status;
  Error(tk_status s, const std::string& m) : std::runtime_error("tk: " + m), status(s) {}
};

// One GEMM operand the tensor-core path loads with TMA.
struct TmaOperand {
  int32_t space, slot;      // where the matrix lives (Space / slot)
  int64_t base_elems;       // element offset of the view from the space's base
  int32_t dtype;
  int64_t inner, outer;     // extents: contiguous dim, strided dim
  int64_t outer_stride;     // elements between consecutive outer rows
  int32_t box_inner, box_outer;
  // > 0: an MN-major operand read as one box of `chunks` 64-wide MN slabs
  // (a 3-D view: MN within the slab, K, slab), stacked 8 KB apart in shared
  // memory exactly as `chunks` separate 2-D boxes would be.
  int32_t chunks;
  // Shared-memory layout: 0 = 128-byte swizzle (GEMM operand tiles), 1 =
  // 64-byte swizzle (32 x 32 epilogue chunks: loads of per-row operands and
  // stores of the outputs).
  int32_t swizzle;

  bool operator==(const TmaOperand& o) const {
    return space == o.space && slot == o.slot && base_elems == o.base_elems && dtype == o.dtype && inner == o.inner &&
           outer == o.outer && outer_stride == o.outer_stride && box_inner == o.box_inner &&
           box_outer == o.box_outer && chunks == o.chunks && swizzle == o.swizzle;
  }
};

struct Plan {
  std::vector<tkd::Stage> stages;
  std::vector<tkd::Task> tasks;
  std::vector<tkd::Instr> code;
  std::vector<tkd::Ref> refs;
  std::vector<TmaOperand> tma;
  int64_t workspace_units = 0;
  int64_t arena_units = 0;
  int32_t max_items = 1;
  size_t smem_bytes = 0;
  int ring_stage_bytes = 0;  // TMA ring slot size for the widest tensor-core tile
  int epi_warp_bytes = 0;    // epilogue staging per epilogue warp
  bool uses_tc = false;
  int pair = 0;              // pair-tile launch (clusters of two blocks): 1 cta_group::2 MMAs, 2 shared B
  int tmem_cols = 0;         // TMEM columns: two accumulators of the widest tile, a power of 2 >= 32
  tk_plan_stats stats{};
  // what tk_run checks
  std::vector<int64_t> input_bytes;
  std::vector<int64_t> output_bytes;
  std::vector<std::pair<int, int>> inplace;  // {output slot, input index}
};

// Throws Error for an invalid or unsupported program.
Plan build_plan(const tk_program_desc& desc, const tk_options& opt, int sm_count);

}  // namespace tkp
