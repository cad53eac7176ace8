// Host planner for the persistent training-step kernel.
//
// The planning rules follow trainkernel's generator (page "trainkernel 0.1.0
// -- trainkernel/codegen.py", class `_Generator`): operations run in the given
// topological order; a GEMM whose result feeds a chain of single-user,
// shape-preserving pointwise ops writes the chain's last value from its tile
// (`__init__`, epilogue detection); a pointwise value with one consumer is
// recomputed at that consumer (`self.inline`); an in-place output is written
// straight into its input when no later op reads that input (`direct_aliases`),
// otherwise it is committed after the last read (`generate`, transactional
// commit); intermediates live in a best-fit arena that recycles a slot after
// its last reader (`_plan_workspace`); and a grid barrier is placed only where
// a read-after-write, write-after-write or write-after-read overlap -- arena
// reuse included -- would otherwise occur inside a stage (`generate`).
//
// What differs, and why (GB300 build):
//   * one hand-written kernel interprets a device op table instead of a
//     generated kernel per program, so every expression is lowered to a small
//     register program (Instr) evaluated per element;
//   * low-precision intermediates are stored packed in their own dtype inside
//     the float32-sized workspace (half the bytes; values are already rounded);
//   * a value consumed as a GEMM A/B operand is never inlined (TMA and the
//     shared-memory staging read memory), and an expression needing more than
//     kVmRegs registers keeps its operands materialised;
//   * a split reduction keeps its own partial-sum slots and costs one barrier
//     between its partial and final passes; the pass after it joins the normal
//     hazard analysis.
#include "planner.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <set>
#include <unordered_map>

namespace tkp {
namespace {

using tkd::Instr;
using tkd::Ref;
using tkd::Stage;
using tkd::Task;
using Shape = std::vector<int64_t>;

bool is_pointwise(int k) { return k >= TK_OP_ADD && k <= TK_OP_CAST; }
bool is_mm(int k) { return k == TK_OP_MM || k == TK_OP_ADDMM; }
bool is_red(int k) { return k == TK_OP_SUM || k == TK_OP_MEAN; }
int64_t esize(int dt) { return dt == TK_F32 ? 4 : 2; }

Shape shape_of(const tk_tensor_spec& s) { return Shape(s.shape, s.shape + s.rank); }
Shape strides_of(const tk_tensor_spec& s) { return Shape(s.strides, s.strides + s.rank); }
int64_t numel_of(const Shape& sh) {
  int64_t n = 1;
  for (auto v : sh) n *= v;
  return n;
}
int64_t numel(const tk_tensor_spec& s) { return numel_of(shape_of(s)); }
Shape contig(const Shape& sh) {
  Shape st(sh.size());
  int64_t a = 1;
  for (int d = int(sh.size()) - 1; d >= 0; --d) {
    st[d] = a;
    a *= sh[d];
  }
  return st;
}
bool exact_contig(const tk_tensor_spec& s) { return s.offset == 0 && strides_of(s) == contig(shape_of(s)); }
bool relaxed_contig(const tk_tensor_spec& s) {
  Shape c = contig(shape_of(s));
  for (int d = 0; d < s.rank; ++d)
    if (s.shape[d] > 1 && s.strides[d] != c[d]) return false;
  return s.offset == 0;
}
// Elements a view can address: max index + 1 (0 for an empty view).
int64_t extent_of(const tk_tensor_spec& s) {
  if (numel(s) == 0) return 0;
  int64_t m = s.offset;
  for (int d = 0; d < s.rank; ++d) m += (s.shape[d] - 1) * s.strides[d];
  return m + 1;
}
int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Operand {
  bool scalar = false;
  double value = 0.0;
  tk_tensor_spec t{};
};

struct OpInfo {
  int index = 0;
  int kind = 0;
  std::vector<Operand> in;
  tk_tensor_spec out{};
  double alpha = 1, beta = 1, threshold = 0, exponent = 2, value = 0;
  int n_dims = -1;
  int dims[TK_MAX_RANK] = {0, 0, 0, 0};
};

struct Buf {
  int dtype = 0;
  Shape shape;
  int64_t extent = 0;
  int producer = -1;  // op index
  int input = -1;     // program input index
  std::vector<int> users;
};

struct Region {
  int space, slot;
  int64_t lo, hi;
};
bool overlap(const Region& a, const Region& b) {
  return a.space == b.space && a.slot == b.slot && a.lo < b.hi && b.lo < a.hi;
}

// Raised while lowering when an expression needs too many registers; the
// named inlined value is materialised instead and planning restarts.
struct RegisterOverflow {
  int buffer;
};

// Raised when a decision turns out not to fit the plan (an in-place side
// output that cannot be written directly); planning restarts without it.
struct Replan {};

float f32(double v) { return static_cast<float>(v); }

class Planner {
 public:
  Planner(const tk_program_desc& d, const tk_options& o, int sms)
      : opt_(o), sms_(std::max(sms, 1)), pair_(sms >= 2 ? o.cta_pairs : 0) {
    read_desc(d);
  }

  Plan run() {
    for (int attempt = 0;; ++attempt) {
      try {
        return plan_once();
      } catch (const RegisterOverflow& r) {
        if (attempt > 256) throw Error(TK_ERR_UNSUPPORTED, "expression too deep to evaluate inline");
        no_inline_.insert(r.buffer);
      } catch (const Replan&) {
        if (attempt > 256) throw Error(TK_ERR_UNSUPPORTED, "planning did not settle");
      }
    }
  }

 private:
  tk_options opt_;
  int sms_;
  // pair tiles: every tensor-core GEMM on 256-row tiles of a pair of SMs;
  // 1: cta_group::2 MMAs, 2: each SM its 128 rows, B shared by TMA multicast
  int pair_;
  std::vector<OpInfo> ops_;
  std::vector<tk_tensor_spec> inputs_, outputs_;
  std::map<int, int> inplace_;  // output slot -> input index
  std::unordered_map<int, Buf> bufs_;
  std::set<int> output_buffers_;
  std::set<int> no_inline_;
  std::set<int> no_side_;               // fused op indices that may not take a side output

  // per-attempt decisions
  struct Fused {
    std::vector<int> chain;
    int final_buf;
  };
  std::map<int, Fused> fused_;          // mm op index -> chain
  std::map<int, int> side_;             // fused mm op index -> pointwise op it also computes
  std::set<int> fused_skip_;            // buffers a fused GEMM makes unnecessary
  std::set<int> inline_;                // buffers evaluated at their consumer
  std::vector<int> schedule_;           // op indices (a fused mm stands for its chain)
  std::map<int, int> writer_;           // buffer -> scheduled op that stores it
  std::map<int, int> direct_;           // output slot -> input index, written directly
  std::map<int, int> binding_;          // buffer -> output slot it is written into
  std::map<int, int64_t> arena_off_;    // buffer -> arena offset (float units)
  std::map<int, int64_t> arena_units_;  // buffer -> units used
  int64_t arena_total_ = 0;

  // ---------------------------------------------------------------- input

  static void check_spec(const tk_tensor_spec& s) {
    if (s.rank < 0 || s.rank > TK_MAX_RANK) throw Error(TK_ERR_UNSUPPORTED, "tensor rank must be 0..4");
    for (int d = 0; d < s.rank; ++d)
      if (s.shape[d] < 0 || s.strides[d] < 0) throw Error(TK_ERR_INVALID, "invalid static shape or stride");
    if (s.offset < 0) throw Error(TK_ERR_INVALID, "invalid static offset");
    if (s.dtype < TK_F32 || s.dtype > TK_BF16) throw Error(TK_ERR_UNSUPPORTED, "unsupported dtype");
  }

  void check_view(const tk_tensor_spec& v) {
    check_spec(v);
    auto it = bufs_.find(v.buffer_id);
    if (it == bufs_.end())
      throw Error(TK_ERR_INVALID, "operation reads buffer " + std::to_string(v.buffer_id) +
                                      " before it is defined (ops must be in topological order)");
    if (v.dtype != it->second.dtype) throw Error(TK_ERR_INVALID, "a view must have its buffer's dtype");
    if (extent_of(v) > it->second.extent) throw Error(TK_ERR_INVALID, "view reads past the end of its buffer");
  }

  static void check_scalar(double v) {
    if (!std::isfinite(v)) throw Error(TK_ERR_UNSUPPORTED, "non-finite scalar constants are unsupported");
  }

  static void check_broadcast(const tk_tensor_spec& operand, const Shape& out) {
    if (operand.rank > int(out.size())) throw Error(TK_ERR_INVALID, "invalid broadcast rank");
    for (int d = 0; d < operand.rank; ++d) {
      int64_t want = out[d + out.size() - operand.rank];
      if (operand.shape[d] != 1 && operand.shape[d] != want)
        throw Error(TK_ERR_INVALID, "incompatible broadcast dimensions");
    }
  }

  void read_desc(const tk_program_desc& d) {
    if (d.n_inputs < 0 || d.n_outputs < 0 || d.n_ops < 0 || d.n_inplace < 0)
      throw Error(TK_ERR_INVALID, "negative count in program descriptor");
    if (d.n_inputs > tkd::kMaxIO || d.n_outputs > tkd::kMaxIO)
      throw Error(TK_ERR_UNSUPPORTED, "at most 256 inputs and 256 outputs");
    if ((d.n_inputs && !d.inputs) || (d.n_outputs && !d.outputs) || (d.n_ops && !d.ops) ||
        (d.n_inplace && !d.inplace))
      throw Error(TK_ERR_INVALID, "NULL array in program descriptor");
    for (int i = 0; i < d.n_inputs; ++i) {
      const auto& s = d.inputs[i];
      check_spec(s);
      if (bufs_.count(s.buffer_id)) throw Error(TK_ERR_INVALID, "buffer defined twice");
      Buf b;
      b.dtype = s.dtype;
      b.shape = shape_of(s);
      b.extent = extent_of(s);
      b.input = i;
      bufs_[s.buffer_id] = b;
      inputs_.push_back(s);
    }
    for (int i = 0; i < d.n_ops; ++i) {
      const tk_op& src = d.ops[i];
      OpInfo op;
      op.index = i;
      op.kind = src.kind;
      if (op.kind < TK_OP_ADD || op.kind > TK_OP_MEAN) throw Error(TK_ERR_UNSUPPORTED, "unsupported operation");
      if (src.n_inputs < 0 || src.n_inputs > TK_MAX_OPERANDS) throw Error(TK_ERR_INVALID, "bad operand count");
      op.alpha = src.alpha;
      op.beta = src.beta;
      op.threshold = src.threshold;
      op.exponent = src.exponent;
      op.value = src.value;
      op.n_dims = src.n_dims;
      for (int j = 0; j < TK_MAX_RANK; ++j) op.dims[j] = src.dims[j];
      for (int j = 0; j < src.n_inputs; ++j) {
        Operand o;
        if (src.scalar_mask & (1u << j)) {
          o.scalar = true;
          o.value = src.scalars[j];
          check_scalar(o.value);
        } else {
          o.t = src.inputs[j];
          check_view(o.t);
        }
        op.in.push_back(o);
      }
      op.out = src.output;
      check_spec(op.out);
      if (op.kind == TK_OP_FULL) {
        // full's value: the attribute when given, else a scalar operand, else 0
        // (codegen.py point_expr); kept in op.value with no operand left
        if (op.in.size() > 1 || (op.in.size() == 1 && !op.in[0].scalar))
          throw Error(TK_ERR_INVALID, "full takes at most one scalar value");
        if (!src.value_given) op.value = op.in.empty() ? 0.0 : op.in[0].value;
        op.in.clear();
      }
      if (bufs_.count(op.out.buffer_id)) throw Error(TK_ERR_INVALID, "buffer defined twice");
      if (!relaxed_contig(op.out))
        throw Error(TK_ERR_INVALID, "materialized output must be contiguous: op " + std::to_string(i));
      check_op(op);
      Buf b;
      b.dtype = op.out.dtype;
      b.shape = shape_of(op.out);
      b.extent = numel(op.out);
      b.producer = i;
      bufs_[op.out.buffer_id] = b;
      for (const auto& o : op.in)
        if (!o.scalar) bufs_[o.t.buffer_id].users.push_back(i);
      ops_.push_back(op);
    }
    for (int j = 0; j < d.n_outputs; ++j) {
      const auto& s = d.outputs[j];
      check_view(s);
      outputs_.push_back(s);
      output_buffers_.insert(s.buffer_id);
    }
    std::set<int> targets;
    for (int k = 0; k < d.n_inplace; ++k) {
      int slot = d.inplace[2 * k], idx = d.inplace[2 * k + 1];
      if (slot < 0 || slot >= d.n_outputs || idx < 0 || idx >= d.n_inputs || inplace_.count(slot))
        throw Error(TK_ERR_INVALID, "invalid inplace output/input index");
      if (!targets.insert(idx).second) throw Error(TK_ERR_INVALID, "inplace outputs must target distinct inputs");
      const auto &o = outputs_[slot], &in = inputs_[idx];
      if (shape_of(o) != shape_of(in) || o.dtype != in.dtype || !exact_contig(in))
        throw Error(TK_ERR_INVALID, "inplace output must match a contiguous input shape and dtype");
      if (bufs_[o.buffer_id].producer < 0)
        throw Error(TK_ERR_INVALID, "inplace outputs must be computed values, not input views");
      inplace_[slot] = idx;
    }
  }

  void check_op(OpInfo& op) {
    const Shape out = shape_of(op.out);
    auto need = [&](size_t lo, size_t hi) {
      if (op.in.size() < lo || op.in.size() > hi) throw Error(TK_ERR_INVALID, "wrong operand count");
    };
    switch (op.kind) {
      case TK_OP_ADD:
      case TK_OP_SUB:
        need(2, 2);
        check_scalar(op.alpha);
        break;
      case TK_OP_MUL:
      case TK_OP_DIV:
        need(2, 2);
        break;
      case TK_OP_THRESHOLD_BACKWARD:
        need(2, 2);
        check_scalar(op.threshold);
        break;
      case TK_OP_NEG:
      case TK_OP_RELU:
      case TK_OP_CAST:
        need(1, 1);
        break;
      case TK_OP_POW:
        need(1, 2);
        if (op.in.size() == 2 && !op.in[1].scalar) throw Error(TK_ERR_UNSUPPORTED, "pow exponent must be a scalar");
        if (op.in.size() == 1) check_scalar(op.exponent);
        if (op.in[0].scalar) throw Error(TK_ERR_UNSUPPORTED, "pow base must be a tensor");
        break;
      case TK_OP_FULL:
        need(0, 0);
        check_scalar(op.value);
        break;
      case TK_OP_MM:
      case TK_OP_ADDMM: {
        size_t base = op.kind == TK_OP_ADDMM ? 1 : 0;
        need(base + 2, base + 2);
        const Operand &a = op.in[base], &b = op.in[base + 1];
        if (a.scalar || b.scalar || a.t.rank != 2 || b.t.rank != 2 || a.t.shape[1] != b.t.shape[0])
          throw Error(TK_ERR_INVALID, "mm requires compatible rank-two tensors");
        if (op.out.rank != 2 || op.out.shape[0] != a.t.shape[0] || op.out.shape[1] != b.t.shape[1])
          throw Error(TK_ERR_INVALID, "matrix output shape does not match its inputs");
        if (op.kind == TK_OP_ADDMM) {
          check_scalar(op.alpha);
          check_scalar(op.beta);
          if (!op.in[0].scalar) check_broadcast(op.in[0].t, out);
        }
        return;
      }
      case TK_OP_SUM:
      case TK_OP_MEAN: {
        need(1, 1);
        if (op.in[0].scalar) throw Error(TK_ERR_INVALID, "reduction requires a tensor");
        const auto& s = op.in[0].t;
        if (op.n_dims > TK_MAX_RANK || op.n_dims < -1) throw Error(TK_ERR_INVALID, "bad reduction dims");
        if (op.n_dims > 0 && s.rank == 0) throw Error(TK_ERR_INVALID, "bad reduction dims");
        for (int j = 0; j < op.n_dims; ++j)
          if (op.dims[j] >= s.rank || op.dims[j] < -s.rank) throw Error(TK_ERR_INVALID, "bad reduction dims");
        int64_t kept = 1;
        std::vector<bool> red = reduced_mask(op);
        for (int d = 0; d < s.rank; ++d)
          if (!red[d]) kept *= s.shape[d];
        if (kept != numel(op.out))
          throw Error(TK_ERR_INVALID, "reduction output shape does not match its axes");
        return;
      }
      default:
        throw Error(TK_ERR_UNSUPPORTED, "unsupported operation");
    }
    for (const auto& o : op.in)
      if (!o.scalar) check_broadcast(o.t, out);
  }

  static std::vector<bool> reduced_mask(const OpInfo& op) {
    const auto& s = op.in[0].t;
    std::vector<bool> red(s.rank, op.n_dims < 0);
    for (int j = 0; j < op.n_dims; ++j) red[((op.dims[j] % s.rank) + s.rank) % s.rank] = true;
    return red;
  }

  // ------------------------------------------------------------ decisions

  // Is a view of an op's contiguous output an affine, per-dimension read of it?
  // Returns, for each producer dim, the view dim that drives it (-1: index 0).
  static bool compose_dims(const tk_tensor_spec& v, const Shape& prod_shape, std::vector<int>* view_dim_of) {
    Shape c = contig(prod_shape);
    std::vector<int> of(prod_shape.size(), -1);
    if (v.offset != 0) return false;
    for (int d = 0; d < v.rank; ++d) {
      if (v.shape[d] <= 1) continue;
      int found = -1;
      for (int e = 0; e < int(prod_shape.size()); ++e)
        if (prod_shape[e] > 1 && c[e] == v.strides[d]) found = e;
      if (found < 0 || of[found] >= 0 || v.shape[d] > prod_shape[found]) return false;
      of[found] = d;
    }
    if (view_dim_of) *view_dim_of = of;
    return true;
  }

  bool reads_as_gemm_operand(int buffer) const {
    for (int u : bufs_.at(buffer).users) {
      const OpInfo& op = ops_[u];
      if (!is_mm(op.kind)) continue;
      size_t base = op.kind == TK_OP_ADDMM ? 1 : 0;
      for (size_t j = base; j < base + 2; ++j)
        if (!op.in[j].scalar && op.in[j].t.buffer_id == buffer) return true;
    }
    return false;
  }

  void detect_epilogues() {
    if (!opt_.fuse_epilogues) return;
    for (const OpInfo& mm : ops_) {
      if (!is_mm(mm.kind) || output_buffers_.count(mm.out.buffer_id)) continue;
      std::vector<int> chain, skipped;
      int current = mm.out.buffer_id;
      while (bufs_[current].users.size() == 1) {
        const OpInfo& nxt = ops_[bufs_[current].users[0]];
        // A chain may end at a program output (its value is then stored
        // straight from the tile) but not pass through one.
        const bool ends_at_output = output_buffers_.count(nxt.out.buffer_id) > 0;
        if (!is_pointwise(nxt.kind)) break;
        // The GEMM root must be read with its own logical layout.
        bool any = false, ok = true;
        for (const auto& o : nxt.in) {
          if (o.scalar || o.t.buffer_id != current) continue;
          any = true;
          if (shape_of(o.t) != bufs_[current].shape || !exact_contig(o.t)) ok = false;
        }
        if (!any || !ok) break;
        chain.push_back(nxt.index);
        skipped.push_back(current);
        current = nxt.out.buffer_id;
        if (ends_at_output || bufs_[current].users.size() != 1) break;
      }
      if (chain.empty()) continue;
      bool safe = true;
      std::set<int> chain_bufs = {mm.out.buffer_id};
      for (int ci : chain) {
        const auto& c = ops_[ci];
        if (shape_of(c.out) != shape_of(mm.out) || !exact_contig(c.out)) safe = false;
        chain_bufs.insert(c.out.buffer_id);
      }
      for (int ci : chain)
        for (const auto& o : ops_[ci].in) {
          if (o.scalar || chain_bufs.count(o.t.buffer_id)) continue;
          if (!exact_contig(o.t)) safe = false;
          int p = bufs_[o.t.buffer_id].producer;
          if (p >= 0 && p >= mm.index && !scaled_input(o.t.buffer_id)) safe = false;
        }
      if (!safe) continue;
      Fused f;
      f.chain = chain;
      f.final_buf = current;
      fused_[mm.index] = f;
      for (int b : skipped) fused_skip_.insert(b);
      fused_skip_.insert(current);
    }
  }

  // Reduction epilogues (a GB300 addition): the single-user pointwise chain
  // after a sum/mean whose output is not returned, e.g. gb = sum(g, 0) then the
  // in-place b' = b - lr*gb.  Only chains the kernel evaluates in chain form
  // are taken: every other operand is a scalar or a contiguous view (of the
  // output's shape) of a program input or of a GEMM/reduction result, at most
  // two loads and four steps.
  void detect_reduction_epilogues() {
    if (!opt_.fuse_epilogues || opt_.expr_forms >= 2) return;
    for (const OpInfo& r : ops_) {
      if (!is_red(r.kind) || output_buffers_.count(r.out.buffer_id) || fused_.count(r.index)) continue;
      std::vector<int> chain;
      int current = r.out.buffer_id, loads = 0;
      bool ok = true;
      while (ok && bufs_[current].users.size() == 1 && chain.size() < size_t(tkd::kChainSteps)) {
        const OpInfo& nxt = ops_[bufs_[current].users[0]];
        if (!is_pointwise(nxt.kind) || nxt.kind == TK_OP_FULL) break;
        if (nxt.kind == TK_OP_POW && (nxt.in.size() > 1 ? nxt.in[1].value : nxt.exponent) != 2.0) break;
        if (shape_of(nxt.out) != bufs_[current].shape || !exact_contig(nxt.out)) break;
        int roots_seen = 0;
        for (const auto& o : nxt.in) {
          if (o.scalar) continue;
          if (o.t.buffer_id == current) {
            if (shape_of(o.t) != bufs_[current].shape || !exact_contig(o.t)) ok = false;
            ++roots_seen;
            continue;
          }
          const Buf& b = bufs_.at(o.t.buffer_id);
          const bool materialised = b.input >= 0 || scaled_input(o.t.buffer_id) ||
                                    (b.producer >= 0 && !is_pointwise(ops_[b.producer].kind) && b.producer < r.index);
          if (!materialised || shape_of(o.t) != bufs_[current].shape || !exact_contig(o.t)) ok = false;
          ++loads;
        }
        if (roots_seen != 1 || loads > 2) ok = false;
        if (!ok) break;
        chain.push_back(nxt.index);
        current = nxt.out.buffer_id;
        if (output_buffers_.count(current)) break;
      }
      if (!ok || chain.empty()) continue;
      Fused f;
      f.chain = chain;
      f.final_buf = current;
      fused_[r.index] = f;
      fused_skip_.insert(r.out.buffer_id);
      for (size_t i = 0; i + 1 < chain.size(); ++i) fused_skip_.insert(ops_[chain[i]].out.buffer_id);
      fused_skip_.insert(current);
    }
  }

  // Side outputs (the page's second epilogue case, "returned pointwise
  // descendants from the same output tile", in a restricted form): a fused
  // GEMM or reduction whose final value is stored and read again (it has
  // several users, or it is returned and has a user) also writes one of those
  // users from the same tile, when that user is
  //   * a one-operand pointwise op of the final value (x*c, -x, a cast), e.g.
  //     the loss gradient 2/N * d next to d, that would be stored anyway (a GEMM
  //     operand, a returned value or a value with several users); or
  //   * an add/sub of the final value and a contiguous view of a program input
  //     of the same shape (a "loaded" side), e.g. the momentum step
  //     W' = W - lr*v' next to v', or W' = W - lr*gW next to a returned gW.
  // A loaded side may be an in-place output only of the input it loads (each
  // element is read, then overwritten by the same thread); it must then be
  // written directly (see check_sides), or the side is dropped.  A GEMM or
  // reduction without a chain (its own result returned, e.g. an exported
  // weight gradient next to the weight's update) takes a side too.
  void detect_side_outputs() {
    for (const OpInfo& mm : ops_) {
      if (!is_mm(mm.kind) && !is_red(mm.kind)) continue;
      if (no_side_.count(mm.index) || (!opt_.fuse_epilogues && !fused_.count(mm.index))) continue;
      auto fu = fused_.find(mm.index);
      const int fin = fu != fused_.end() ? fu->second.final_buf : mm.out.buffer_id;
      const Buf& fb = bufs_.at(fin);
      if (fb.users.empty() || (fb.users.size() < 2 && !output_buffers_.count(fin))) continue;
      for (int u : fb.users) {
        const OpInfo& op = ops_[u];
        if (!is_pointwise(op.kind) || op.kind == TK_OP_FULL || fused_skip_.count(op.out.buffer_id)) continue;
        if (shape_of(op.out) != fb.shape || !exact_contig(op.out)) continue;
        const bool unary = op.kind == TK_OP_MUL || op.kind == TK_OP_NEG || op.kind == TK_OP_CAST;
        const bool axpy = op.kind == TK_OP_ADD || op.kind == TK_OP_SUB;
        if (!unary && !axpy) continue;
        int roots_seen = 0, loads = 0, loaded = -1;
        bool ok = true;
        for (const auto& o : op.in) {
          if (o.scalar) continue;
          if (o.t.buffer_id == fin) {
            if (shape_of(o.t) == fb.shape && exact_contig(o.t)) ++roots_seen;
            else ok = false;
          } else if (axpy && bufs_.at(o.t.buffer_id).input >= 0 && shape_of(o.t) == fb.shape && exact_contig(o.t)) {
            ++loads;
            loaded = o.t.buffer_id;
          } else {
            ok = false;
          }
        }
        if (!ok || roots_seen != 1 || (axpy && loads != 1) || (unary && loads != 0)) continue;
        if (is_red(mm.kind) && !axpy) continue;  // reductions take loaded sides only
        const int target = inplace_target(op.out.buffer_id);
        if (target >= 0 && (!axpy || target != loaded)) continue;
        const Buf& ub = bufs_.at(op.out.buffer_id);
        const bool stored = output_buffers_.count(op.out.buffer_id) || ub.users.size() != 1 ||
                            reads_as_gemm_operand(op.out.buffer_id);
        if (!stored) continue;
        if (fu == fused_.end()) {
          if (is_red(mm.kind) && opt_.expr_forms >= 2) continue;  // a reduction's side needs its chain form
          Fused f;
          f.final_buf = fin;
          fused_[mm.index] = f;
        }
        side_[mm.index] = u;
        fused_skip_.insert(op.out.buffer_id);
        break;
      }
    }
  }

  // An in-place side output must be written directly into its input (the
  // tile reads the old value at the same index just before); when the plan
  // cannot do that, drop the side and plan again.
  void check_sides() {
    for (const auto& kv : side_) {
      const int out_buf = ops_[kv.second].out.buffer_id;
      for (const auto& io : inplace_)
        if (outputs_[io.first].buffer_id == out_buf && !direct_.count(io.first)) {
          no_side_.insert(kv.first);
          throw Replan{};
        }
    }
  }

  // Buffers scheduled op s stores: its (final) output and a side output.
  std::vector<int> stored_buffers(int s) const {
    std::vector<int> r = {out_buffer_of(s)};
    auto it = side_.find(s);
    if (it != side_.end()) r.push_back(ops_[it->second].out.buffer_id);
    return r;
  }

  // A single-use value c * (contiguous view of a program input): evaluated
  // inside whatever consumes it, so it may be produced after a GEMM whose
  // epilogue reads it (the momentum term mul(v, 0.9)).
  bool scaled_input(int buffer) const {
    const Buf& b = bufs_.at(buffer);
    if (b.producer < 0 || b.users.size() != 1 || output_buffers_.count(buffer) || !opt_.fuse_pointwise) return false;
    const OpInfo& op = ops_[b.producer];
    if (op.kind != TK_OP_MUL || op.in.size() != 2 || op.in[0].scalar == op.in[1].scalar) return false;
    const Operand& v = op.in[0].scalar ? op.in[1] : op.in[0];
    return bufs_.at(v.t.buffer_id).input >= 0 && exact_contig(v.t) && shape_of(v.t) == b.shape;
  }

  bool is_chain_final(int buffer) const {
    for (const auto& kv : fused_)
      if (kv.second.final_buf == buffer) return true;
    return false;
  }

  void choose_inline() {
    if (!opt_.fuse_pointwise) return;
    for (const OpInfo& op : ops_) {
      int b = op.out.buffer_id;
      if (!is_pointwise(op.kind) || output_buffers_.count(b) || is_chain_final(b) || no_inline_.count(b)) continue;
      const Buf& buf = bufs_[b];
      bool input_cast = opt_.inline_input_casts && op.kind == TK_OP_CAST && !op.in[0].scalar &&
                        bufs_[op.in[0].t.buffer_id].input >= 0;
      if (!(buf.users.size() == 1 || input_cast)) continue;
      if (reads_as_gemm_operand(b)) continue;
      bool composable = true;
      for (int u : buf.users)
        for (const auto& o : ops_[u].in)
          if (!o.scalar && o.t.buffer_id == b && !compose_dims(o.t, buf.shape, nullptr)) composable = false;
      if (!composable) continue;
      inline_.insert(b);
    }
  }

  int out_buffer_of(int op_index) const {
    auto it = fused_.find(op_index);
    return it != fused_.end() ? it->second.final_buf : ops_[op_index].out.buffer_id;
  }

  void build_schedule() {
    for (const OpInfo& op : ops_) {
      if (fused_.count(op.index)) {
        schedule_.push_back(op.index);
      } else if (!fused_skip_.count(op.out.buffer_id) && !inline_.count(op.out.buffer_id)) {
        schedule_.push_back(op.index);
      }
    }
    defer_inplace_epilogues();
    for (int s : schedule_)
      for (int b : stored_buffers(s)) writer_[b] = s;
  }

  // Input buffer an in-place output overwrites (-1: not in place).
  int inplace_target(int buffer) const {
    for (const auto& kv : inplace_)
      if (outputs_[kv.first].buffer_id == buffer) return inputs_[kv.second].buffer_id;
    return -1;
  }

  // A fused GEMM or reduction that writes an in-place output (its chain's
  // final value or its side output: e.g. a weight-gradient GEMM ending in the
  // SGD update of that weight, or writing the momentum buffer and the weight)
  // moves after the last scheduled op that still reads an old value it
  // overwrites (the input-gradient GEMM of the same layer), so that it can
  // write the new values directly.  Moving it later is legal when only
  // program outputs depend on what it writes.
  void defer_inplace_epilogues() {
    for (size_t i = 0; i < schedule_.size(); ++i) {
      const int f = schedule_[i];
      if (!fused_.count(f)) continue;
      std::set<int> targets, written;
      for (int b : stored_buffers(f)) {
        written.insert(b);
        const int t = inplace_target(b);
        if (t >= 0) targets.insert(t);
      }
      if (targets.empty()) continue;
      size_t last = i;
      bool blocked = false;
      for (size_t j = i + 1; j < schedule_.size(); ++j) {
        bool reads_target = false;
        for (const auto& v : reads_of(schedule_[j])) {
          const std::set<int> raw = raw_inputs(v.buffer_id);
          for (int t : targets)
            if (raw.count(t)) reads_target = true;
          for (int b : roots(v.buffer_id))
            if (written.count(b)) blocked = true;
        }
        if (blocked) break;
        if (reads_target) last = j;
      }
      if (blocked || last == i) continue;
      schedule_.erase(schedule_.begin() + i);
      schedule_.insert(schedule_.begin() + last, f);
      --i;  // the op now at position i has not been examined
    }
  }

  // Every tensor operand a scheduled op reads (GEMM + chain externals).
  std::vector<tk_tensor_spec> reads_of(int op_index) const {
    std::vector<tk_tensor_spec> r;
    for (const auto& o : ops_[op_index].in)
      if (!o.scalar) r.push_back(o.t);
    auto it = fused_.find(op_index);
    if (it != fused_.end()) {
      std::set<int> chain_bufs = {ops_[op_index].out.buffer_id};
      for (int ci : it->second.chain) chain_bufs.insert(ops_[ci].out.buffer_id);
      for (int ci : it->second.chain)
        for (const auto& o : ops_[ci].in)
          if (!o.scalar && !chain_bufs.count(o.t.buffer_id)) r.push_back(o.t);
    }
    auto sd = side_.find(op_index);
    if (sd != side_.end()) {
      const int fin = out_buffer_of(op_index);
      for (const auto& o : ops_[sd->second].in)
        if (!o.scalar && o.t.buffer_id != fin) r.push_back(o.t);
    }
    return r;
  }

  std::set<int> raw_inputs(int buffer) const {
    const Buf& b = bufs_.at(buffer);
    if (b.input >= 0) return {buffer};
    std::set<int> r;
    if (inline_.count(buffer))
      for (const auto& o : ops_[b.producer].in)
        if (!o.scalar) {
          auto s = raw_inputs(o.t.buffer_id);
          r.insert(s.begin(), s.end());
        }
    return r;
  }

  bool identity_access(const tk_tensor_spec& spec, int target, const Shape& shape) const {
    if (!raw_inputs(spec.buffer_id).count(target)) return true;
    if (shape_of(spec) != shape || !exact_contig(spec)) return false;
    if (spec.buffer_id == target) return true;
    for (const auto& o : ops_[bufs_.at(spec.buffer_id).producer].in)
      if (!o.scalar && !identity_access(o.t, target, shape)) return false;
    return true;
  }

  void choose_direct_aliases() {
    std::map<int, int> out_count;
    for (const auto& o : outputs_) out_count[o.buffer_id]++;
    for (const auto& kv : inplace_) {
      int slot = kv.first, idx = kv.second;
      const auto& out = outputs_[slot];
      int target = inputs_[idx].buffer_id;
      int pos = -1;
      for (size_t i = 0; i < schedule_.size(); ++i)
        for (int b : stored_buffers(schedule_[i]))
          if (b == out.buffer_id) pos = int(i);
      if (pos < 0 || out_count[out.buffer_id] != 1) continue;
      const bool fused_gemm = fused_.count(schedule_[pos]) > 0;
      if (!fused_gemm && !is_pointwise(ops_[schedule_[pos]].kind)) continue;
      if (!exact_contig(out)) continue;
      bool target_is_output = false;
      for (const auto& o : outputs_)
        if (o.buffer_id == target) target_is_output = true;
      if (target_is_output) continue;
      bool later_read = false;
      for (size_t i = pos + 1; i < schedule_.size() && !later_read; ++i)
        for (const auto& v : reads_of(schedule_[i]))
          if (raw_inputs(v.buffer_id).count(target)) later_read = true;
      if (later_read) continue;
      bool ident = true;
      for (const auto& v : reads_of(schedule_[pos]))
        if (!identity_access(v, target, shape_of(out))) ident = false;
      if (!ident) continue;
      direct_[slot] = idx;
    }
  }

  void choose_bindings() {
    for (size_t j = 0; j < outputs_.size(); ++j) {
      if (inplace_.count(int(j)) && !direct_.count(int(j))) continue;
      const auto& spec = outputs_[j];
      auto w = writer_.find(spec.buffer_id);
      if (w == writer_.end()) continue;  // an input view: copied at the end
      const Buf& b = bufs_[spec.buffer_id];
      if (b.dtype == spec.dtype && relaxed_contig(spec) && numel(spec) == numel_of(b.shape))
        binding_.emplace(spec.buffer_id, int(j));
    }
  }

  int64_t units_of(int buffer) const {
    const Buf& b = bufs_.at(buffer);
    return ceil_div(numel_of(b.shape) * esize(b.dtype), 4);
  }

  std::set<int> roots(int buffer) const {
    if (!inline_.count(buffer)) return {buffer};
    std::set<int> r;
    for (const auto& o : ops_[bufs_.at(buffer).producer].in)
      if (!o.scalar) {
        auto s = roots(o.t.buffer_id);
        r.insert(s.begin(), s.end());
      }
    return r;
  }

  // Arena offsets of the stored intermediate values in schedule order.  With
  // `reuse`, a value takes the smallest sufficient freed slot (on a tie the
  // one freed first) whose previous occupant was last accessed in an earlier
  // stage (stage_of_ from a first pass); without it every value has its own.
  void plan_arena(bool reuse) {
    std::map<int, int> last;
    for (size_t i = 0; i < schedule_.size(); ++i)
      for (const auto& v : reads_of(schedule_[i]))
        for (int r : roots(v.buffer_id)) last[r] = int(i);
    for (const auto& o : outputs_)
      for (int r : roots(o.buffer_id)) last[r] = int(schedule_.size());
    struct Slot {
      int buf;
      int64_t start, size;
      int pos;  // schedule position of the writer
    };
    struct Free {
      int64_t start, size;
      int stage;  // stage of the last access to the previous occupant
    };
    std::vector<Slot> active;
    std::vector<Free> free_list;
    int64_t total = 0;
    for (size_t i = 0; i < schedule_.size(); ++i)
     for (int b : stored_buffers(schedule_[i])) {
      if (binding_.count(b)) continue;
      std::vector<Slot> keep;
      for (const auto& s : active) {
        auto it = last.find(s.buf);
        const int l = it == last.end() ? -1 : it->second;
        if (l < int(i))
          free_list.push_back({s.start, s.size, reuse ? stage_of_[size_t(std::max(l, s.pos))] : 0});
        else
          keep.push_back(s);
      }
      active = keep;
      int64_t size = std::max<int64_t>(64, round_up(units_of(b), 64));
      int best = -1;
      for (size_t j = 0; j < free_list.size() && reuse; ++j) {
        if (free_list[j].size < size || free_list[j].stage >= stage_of_[i]) continue;
        if (best < 0 || free_list[j].size < free_list[best].size) best = int(j);
      }
      int64_t start;
      if (best >= 0) {
        start = free_list[best].start;
        const int64_t n = free_list[best].size;
        const int st = free_list[best].stage;
        free_list.erase(free_list.begin() + best);
        if (n > size) free_list.push_back({start + size, n - size, st});
      } else {
        start = total;
        total += size;
      }
      arena_off_[b] = start;
      arena_units_[b] = units_of(b);
      active.push_back({b, start, size, int(i)});
    }
    arena_total_ = total;
  }

  // ------------------------------------------------------------ locations

  // Where buffer b is stored: (space, slot, element base).
  void location(int b, int* space, int* slot, int64_t* base) const {
    const Buf& buf = bufs_.at(b);
    if (buf.input >= 0) {
      *space = tkd::SP_IN;
      *slot = buf.input;
      *base = 0;
      return;
    }
    auto bind = binding_.find(b);
    if (bind != binding_.end()) {
      *space = tkd::SP_OUT;
      *slot = bind->second;
      *base = 0;
      return;
    }
    auto it = arena_off_.find(b);
    if (it == arena_off_.end()) throw Error(TK_ERR_INVALID, "internal: value has no storage");
    *space = tkd::SP_WS;
    *slot = 0;
    *base = (tkd::kHeaderUnits + it->second) * 4 / esize(buf.dtype);
  }

  Region storage_region(int b) const {
    const Buf& buf = bufs_.at(b);
    if (buf.input >= 0) return {tkd::SP_IN, buf.input, 0, buf.extent};
    auto bind = binding_.find(b);
    if (bind != binding_.end()) {
      auto d = direct_.find(bind->second);
      if (d != direct_.end()) return {tkd::SP_IN, d->second, 0, bufs_.at(inputs_[d->second].buffer_id).extent};
      return {tkd::SP_OUT, bind->second, 0, numel(outputs_[bind->second])};
    }
    int64_t off = arena_off_.at(b);
    return {tkd::SP_WS, 0, off, off + arena_units_.at(b)};
  }

  void read_regions(const tk_tensor_spec& v, std::vector<Region>& out) const {
    if (inline_.count(v.buffer_id)) {
      for (const auto& o : ops_[bufs_.at(v.buffer_id).producer].in)
        if (!o.scalar) read_regions(o.t, out);
      return;
    }
    const Buf& b = bufs_.at(v.buffer_id);
    if (b.input >= 0) {
      if (!direct_.empty()) out.push_back({tkd::SP_IN, b.input, 0, b.extent});
      return;
    }
    out.push_back(storage_region(v.buffer_id));
  }

  // ------------------------------------------------------------ lowering

  struct Emit {
    Plan* plan;
    const Planner* P;
    int task_ref_begin;
    Shape space;
    int root_buf = -1;
    int max_reg = 0;

    void push(uint8_t op, int dst, int a, int b, int round, float imm = 0.f, int ref = -1) {
      if (dst >= tkd::kVmRegs || a >= tkd::kVmRegs || b >= tkd::kVmRegs) throw RegisterOverflow{-1};
      Instr in{};
      in.op = op;
      in.dst = uint8_t(dst);
      in.a = uint8_t(a);
      in.b = uint8_t(b);
      in.round = uint8_t(round);
      in.imm = imm;
      in.ref = ref;
      plan->code.push_back(in);
      max_reg = std::max(max_reg, std::max(dst, std::max(a, b)));
    }

    int add_ref(const tk_tensor_spec& v, const std::vector<int>& dimmap) {
      Ref r{};
      int64_t base;
      P->location(v.buffer_id, &r.space, &r.slot, &base);
      r.dtype = v.dtype;
      r.base = base + v.offset;
      for (int d = 0; d < v.rank; ++d)
        if (v.shape[d] > 1 && dimmap[d] >= 0) r.stride[dimmap[d]] += v.strides[d];
      plan->refs.push_back(r);
      return int(plan->refs.size()) - 1 - task_ref_begin;
    }

    // Value of view v into register r; dimmap[d] = index dim driving view dim d.
    void value(const tk_tensor_spec& v, const std::vector<int>& dimmap, int r) {
      if (v.buffer_id == root_buf) {
        if (r != 0) push(tkd::OP_MOV, r, 0, 0, TK_F32);
        return;
      }
      if (P->inline_.count(v.buffer_id)) {
        const Buf& b = P->bufs_.at(v.buffer_id);
        std::vector<int> of;
        if (!compose_dims(v, b.shape, &of)) throw Error(TK_ERR_INVALID, "internal: non-affine inline view");
        std::vector<int> pmap(b.shape.size(), -1);
        for (size_t e = 0; e < of.size(); ++e) pmap[e] = of[e] >= 0 ? dimmap[of[e]] : -1;
        try {
          op_value(P->ops_[b.producer], pmap, r);
        } catch (const RegisterOverflow&) {
          throw RegisterOverflow{v.buffer_id};
        }
        return;
      }
      push(tkd::OP_LOAD, r, 0, 0, TK_F32, 0.f, add_ref(v, dimmap));
    }

    // Value of pointwise op `op` into register r (temporaries above r);
    // outmap[d] = index dim driving output dim d.
    void op_value(const OpInfo& op, const std::vector<int>& outmap, int r) {
      int rank = op.out.rank;
      auto operand = [&](int j, int reg) {
        const Operand& o = op.in[j];
        if (o.scalar) {
          push(tkd::OP_CONST, reg, 0, 0, TK_F32, f32(o.value));
          return;
        }
        std::vector<int> m(o.t.rank, -1);
        for (int d = 0; d < o.t.rank; ++d)
          m[d] = o.t.shape[d] == 1 ? -1 : outmap[d + rank - o.t.rank];
        value(o.t, m, reg);
      };
      int rd = op.out.dtype;
      switch (op.kind) {
        case TK_OP_ADD:
        case TK_OP_SUB:
        case TK_OP_MUL:
        case TK_OP_DIV:
        case TK_OP_THRESHOLD_BACKWARD: {
          operand(0, r);
          operand(1, r + 1);
          uint8_t code = op.kind == TK_OP_ADD ? tkd::OP_ADD
                         : op.kind == TK_OP_SUB ? tkd::OP_SUB
                         : op.kind == TK_OP_MUL ? tkd::OP_MUL
                         : op.kind == TK_OP_DIV ? tkd::OP_DIV
                                                : tkd::OP_THRESH;
          float imm = (op.kind == TK_OP_ADD || op.kind == TK_OP_SUB) ? f32(op.alpha)
                      : op.kind == TK_OP_THRESHOLD_BACKWARD        ? f32(op.threshold)
                                                                   : 0.f;
          push(code, r, r, r + 1, rd, imm);
          return;
        }
        case TK_OP_NEG:
          operand(0, r);
          push(tkd::OP_NEG, r, r, r, rd);
          return;
        case TK_OP_RELU:
          operand(0, r);
          push(tkd::OP_RELU, r, r, r, rd);
          return;
        case TK_OP_CAST:
          operand(0, r);
          push(tkd::OP_MOV, r, r, r, rd);
          return;
        case TK_OP_POW: {
          double e = op.in.size() > 1 ? op.in[1].value : op.exponent;
          operand(0, r);
          if (e == 2.0)
            push(tkd::OP_SQUARE, r, r, r, rd);
          else
            push(tkd::OP_POW, r, r, r, rd, f32(e));
          return;
        }
        case TK_OP_FULL:
          push(tkd::OP_CONST, r, 0, 0, rd, f32(op.value));
          return;
        default:
          throw Error(TK_ERR_INVALID, "internal: not a pointwise op");
      }
    }
  };

  // Builds the linear-chain form of an expression (see tkd::Chain); `fail`
  // is set when the expression is not a chain with at most two loads.
  struct ChainBuild {
    Plan* plan;
    const Planner* P;
    int task_ref_begin;
    tkd::Chain ch{};
    int root_buf = -1;
    bool fail = false;
    bool started = false;

    int add_ref(const tk_tensor_spec& v, const std::vector<int>& dimmap) {
      Emit e{plan, P, task_ref_begin, {}};
      return e.add_ref(v, dimmap);
    }
    int load_slot(const tk_tensor_spec& v, const std::vector<int>& dimmap) {
      if (ch.n_loads >= 2) {
        fail = true;
        return 0;
      }
      ch.load_ref[ch.n_loads] = add_ref(v, dimmap);
      return ch.n_loads++;
    }
    void step(int op, int round, int ext, int second, float imm, float cval) {
      if (ch.n_steps >= tkd::kChainSteps) {
        fail = true;
        return;
      }
      tkd::ChainStep& st = ch.steps[ch.n_steps++];
      st.op = uint8_t(op);
      st.round = uint8_t(round);
      st.ext = uint8_t(ext);
      st.second = uint8_t(second);
      st.imm = imm;
      st.cval = cval;
    }
    bool is_tree(const Operand& o) const {
      return !o.scalar && (o.t.buffer_id == root_buf || P->inline_.count(o.t.buffer_id));
    }
    // The running value becomes view v.
    void spine(const tk_tensor_spec& v, const std::vector<int>& dimmap) {
      if (fail) return;
      if (v.buffer_id == root_buf) return;
      if (P->inline_.count(v.buffer_id)) {
        const Buf& b = P->bufs_.at(v.buffer_id);
        std::vector<int> of;
        if (!compose_dims(v, b.shape, &of)) {
          fail = true;
          return;
        }
        std::vector<int> pmap(b.shape.size(), -1);
        for (size_t e = 0; e < of.size(); ++e) pmap[e] = of[e] >= 0 ? dimmap[of[e]] : -1;
        spine_op(P->ops_[b.producer], pmap);
        return;
      }
      if (started || ch.n_loads) {
        fail = true;
        return;
      }
      ch.start = tkd::CH_LOAD;
      load_slot(v, dimmap);
      started = true;
    }
    std::vector<int> operand_map(const OpInfo& op, const Operand& o, const std::vector<int>& outmap) const {
      std::vector<int> m(o.t.rank, -1);
      for (int d = 0; d < o.t.rank; ++d) m[d] = o.t.shape[d] == 1 ? -1 : outmap[d + op.out.rank - o.t.rank];
      return m;
    }
    void spine_op(const OpInfo& op, const std::vector<int>& outmap) {
      if (fail) return;
      const int rd = op.out.dtype;
      auto start_const = [&](double v) {
        if (started) {
          fail = true;
          return;
        }
        ch.start = tkd::CH_CONST;
        ch.start_const = f32(v);
        started = true;
      };
      auto unary_spine = [&](const Operand& o) {
        if (o.scalar)
          start_const(o.value);
        else
          spine(o.t, operand_map(op, o, outmap));
      };
      switch (op.kind) {
        case TK_OP_NEG:
        case TK_OP_RELU:
        case TK_OP_CAST:
          unary_spine(op.in[0]);
          step(op.kind == TK_OP_NEG ? tkd::OP_NEG : op.kind == TK_OP_RELU ? tkd::OP_RELU : tkd::OP_MOV, rd, 0, 0, 0.f,
               0.f);
          return;
        case TK_OP_POW: {
          double e = op.in.size() > 1 ? op.in[1].value : op.exponent;
          if (e != 2.0) {  // general powf stays in the instruction form
            fail = true;
            return;
          }
          unary_spine(op.in[0]);
          step(tkd::OP_SQUARE, rd, 0, 0, f32(e), 0.f);
          return;
        }
        case TK_OP_FULL:
          start_const(op.value);
          step(tkd::OP_MOV, rd, 0, 0, 0.f, 0.f);
          return;
        default:
          break;
      }
      const Operand &o0 = op.in[0], &o1 = op.in[1];
      bool t0 = is_tree(o0), t1 = is_tree(o1);
      // an inlined c * input next to the running value is loaded and scaled
      const OpInfo* scaled = nullptr;
      if (t0 && t1 && root_buf >= 0) {
        const int oi = o0.t.buffer_id == root_buf ? 1 : o1.t.buffer_id == root_buf ? 0 : -1;
        const Operand& other = oi == 1 ? o1 : o0;
        if (oi >= 0 && P->inline_.count(other.t.buffer_id) && P->scaled_input(other.t.buffer_id) &&
            shape_of(other.t) == P->bufs_.at(other.t.buffer_id).shape && exact_contig(other.t)) {
          scaled = &P->ops_[P->bufs_.at(other.t.buffer_id).producer];
          (oi == 1 ? t1 : t0) = false;
        }
      }
      if (t0 && t1) {
        fail = true;
        return;
      }
      const int side = t0 ? 0 : t1 ? 1 : (o0.scalar ? 1 : 0);
      const Operand& sp = side == 0 ? o0 : o1;
      const Operand& other = side == 0 ? o1 : o0;
      unary_spine(sp);
      int ext;
      float cval = 0.f;
      uint8_t ext_mul = 0, ext_round = 0;
      if (other.scalar) {
        ext = tkd::EXT_CONST;
        cval = f32(other.value);
      } else if (scaled) {
        const Operand& v = scaled->in[0].scalar ? scaled->in[1] : scaled->in[0];
        const double c = scaled->in[0].scalar ? scaled->in[0].value : scaled->in[1].value;
        ext = load_slot(v.t, operand_map(op, other, outmap)) == 0 ? tkd::EXT_LOAD0 : tkd::EXT_LOAD1;
        cval = f32(c);
        ext_mul = 1;
        ext_round = uint8_t(scaled->out.dtype);
      } else {
        ext = load_slot(other.t, operand_map(op, other, outmap)) == 0 ? tkd::EXT_LOAD0 : tkd::EXT_LOAD1;
      }
      const int code = op.kind == TK_OP_ADD ? tkd::OP_ADD
                       : op.kind == TK_OP_SUB ? tkd::OP_SUB
                       : op.kind == TK_OP_MUL ? tkd::OP_MUL
                       : op.kind == TK_OP_DIV ? tkd::OP_DIV
                                              : tkd::OP_THRESH;
      const float imm = (op.kind == TK_OP_ADD || op.kind == TK_OP_SUB) ? f32(op.alpha)
                        : op.kind == TK_OP_THRESHOLD_BACKWARD        ? f32(op.threshold)
                                                                     : 0.f;
      step(code, rd, ext, side, imm, cval);
      if (!fail) {
        ch.steps[ch.n_steps - 1].ext_mul = ext_mul;
        ch.steps[ch.n_steps - 1].ext_round = ext_round;
      }
    }
  };

  // Chain form of task t's expression into t.chain; false leaves no trace.
  template <typename F>
  bool try_chain(Plan& plan, Task& t, F&& build) const {
    if (opt_.expr_forms >= 2) return false;
    ChainBuild cb{&plan, this, t.ref_begin};
    build(cb);
    for (size_t i = t.ref_begin; i < plan.refs.size() && !cb.fail; ++i) {
      const int64_t es = plan.refs[i].dtype == TK_F32 ? 4 : 2;
      for (int d = 0; d < tkd::kMaxRank; ++d)
        if (plan.refs[i].stride[d] * es >= (int64_t(1) << 31)) cb.fail = true;
    }
    if (cb.fail) {
      plan.refs.resize(t.ref_begin);
      return false;
    }
    cb.ch.valid = 1;
    t.chain = cb.ch;
    t.code_len = 0;
    t.n_refs = int(plan.refs.size()) - t.ref_begin;
    return true;
  }

  static std::vector<int> identity_map(int rank) {
    std::vector<int> m(rank);
    for (int d = 0; d < rank; ++d) m[d] = d;
    return m;
  }

  Task new_task(int kind, const Shape& space) const {
    Task t{};
    t.kind = kind;
    t.rank = int(space.size());
    for (int d = 0; d < t.rank; ++d) t.shape[d] = space[d];
    t.numel = numel_of(space);
    if (t.numel >= (int64_t(1) << 31)) throw Error(TK_ERR_UNSUPPORTED, "tensors of 2^31 or more elements");
    t.vec = (t.rank >= 1 && t.shape[t.rank - 1] % 8 == 0 && t.numel > 0) ? 8 : 1;
    t.tma_a = t.tma_b = -1;
    t.tma_out = t.tma_out2 = t.tma_ld0 = t.tma_ld1 = t.tma_sd = -1;
    t.op_index = -1;
    t.k_splits = 1;
    return t;
  }

  Ref out_ref(int buffer) const {
    Ref r{};
    int64_t base;
    location(buffer, &r.space, &r.slot, &base);
    r.dtype = bufs_.at(buffer).dtype;
    r.base = base;
    r.vmode = tkd::VM_CONTIG;
    return r;
  }

  // Fill vector modes once the task's vector width is known.
  void finish_refs(Plan& plan, Task& t) const {
    for (int i = 0; i < t.n_refs; ++i) {
      Ref& r = plan.refs[t.ref_begin + i];
      r.vmode = tkd::VM_GATHER;
      if (t.vec != 8 || t.rank == 0) continue;
      int64_t s = r.stride[t.rank - 1];
      if (s == 0) {
        r.vmode = tkd::VM_BCAST;
      } else if (s == 1 && r.base % 8 == 0) {
        bool ok = true;
        for (int d = 0; d < t.rank - 1; ++d)
          if (r.stride[d] % 8) ok = false;
        if (ok) r.vmode = tkd::VM_CONTIG;
      }
    }
  }

  // Staged epilogue of a compiled GEMM epilogue with a 16-bit output: which
  // load slots are read per row (row stride != 0; 16-bit, 16-byte aligned
  // rows) and go through shared memory.  -1: not eligible.
  int epi_stage_mask(const Plan& plan, const Task& t) const {
    const tkd::Chain& ch = t.chain;
    if (t.kind != tkd::T_GEMM_TC || t.k_splits > 1 || !ch.valid || ch.fast < tkd::FK_E_ACC ||
        (ch.fast > tkd::FK_E_ACC_THRESH && ch.fast != tkd::FK_E_UPDATE && ch.fast != tkd::FK_E_MOMENTUM))
      return -1;
    if (t.out.dtype == TK_F32 || t.out.base % 8 != 0 || t.n % 8 != 0) return -1;
    if (t.has_side && (t.out2.dtype == TK_F32 || t.out2.base % 8 != 0)) return -1;
    // the last rounding is to the output type (the kernel folds it into the store)
    const int last = ch.n_steps ? ch.steps[ch.n_steps - 1].round : ch.round0;
    if (last != t.out.dtype) return -1;
    int mask = 4;
    // a loaded side's operand goes through shared memory like a per-row operand
    if (t.has_side && t.side.ext == tkd::EXT_LOAD1) {
      if (t.side_ld.dtype == TK_F32 || t.side_ld.base % 8 != 0) return -1;
      mask |= 8;
    }
    for (int s = 0; s < ch.n_loads; ++s) {
      const Ref& r = plan.refs[t.ref_begin + ch.load_ref[s]];
      if (r.dtype == TK_F32 || r.base % 8 != 0) return -1;
      if (r.stride[0] == 0) continue;  // one row for all tile rows: read directly
      if ((r.stride[0] * 2) % 16 != 0) return -1;
      mask |= 1 << s;
    }
    if (epi_uniform_dtype(plan, t) == 0) return -1;
    return mask;
  }

  // How many of a stage's other items (reductions, pointwise, split-K sums)
  // one tensor-core tile is worth, from rough per-SM costs: a tile ~0.4 us
  // per 64-deep k block (its operand ring is latency-bound) plus ~2 us of
  // epilogue; an item ~1 us plus its bytes at ~25 GB/s.  Blocks with one
  // tile fewer than the busiest ones take that many items each first, so
  // that the stage's items fill the wave's last partial round of tiles
  // (stages whose tiles loop over at least 15 k blocks).
  static int light_items(const Plan& plan, const Stage& S) {
    if (S.n_tc_items == 0 || S.n_items == S.n_tc_items) return 0;
    double tile_us = 0.0, item_us = 0.0;
    int64_t items = 0;
    for (int i = S.task_begin; i < int(plan.tasks.size()); ++i) {
      const Task& t = plan.tasks[i];
      if (t.kind == tkd::T_GEMM_TC) {
        tile_us = std::max(tile_us, 2.0 + 0.4 * t.kb_split);
      } else if (t.n_items > 0 && !t.bg) {
        const bool red = t.kind == tkd::T_REDUCE_ROW || t.kind == tkd::T_REDUCE_COL || t.kind == tkd::T_REDUCE_FINAL;
        const double elems = double(t.numel) / double(t.n_items);
        const double bytes = elems * 2.0 * (red ? std::max(1, t.chain.n_loads) : 1 + t.chain.n_loads);
        item_us += double(t.n_items) * (1.0 + bytes / 25e3);
        items += t.n_items;
      }
    }
    // short tiles (a few k blocks) finish within an item or two of each
    // other: plain round-robin balances those stages better
    if (items == 0 || item_us <= 0.0 || tile_us < 8.0) return 0;
    return int(std::min(64.0, std::floor(tile_us / (item_us / double(items)))));
  }

  // The one 16-bit type of every operand, rounding and output of a GEMM
  // epilogue (with its side output), or 0 if they mix types.  The staged
  // epilogue is compiled per type, so that its conversions carry no
  // branches on a type read at run time.
  static int epi_uniform_dtype(const Plan& plan, const Task& t) {
    const tkd::Chain& ch = t.chain;
    const int dt = t.out.dtype;
    if (dt != TK_BF16 && dt != TK_F16) return 0;
    bool same = ch.round0 == dt;
    for (int i = 0; i < ch.n_steps; ++i) {
      same = same && ch.steps[i].round == dt;
      if (ch.steps[i].ext_mul) same = same && ch.steps[i].ext_round == dt;
    }
    for (int s = 0; s < ch.n_loads; ++s) same = same && plan.refs[t.ref_begin + ch.load_ref[s]].dtype == dt;
    if (t.has_side) {
      same = same && t.out2.dtype == dt && t.side.round == dt;
      if (t.side.ext == tkd::EXT_LOAD1) same = same && t.side_ld.dtype == dt;
    }
    return same ? dt : 0;
  }

  // Staging bytes per epilogue warp at a ring depth of `depth` chunks: per
  // chunk one buffer per per-row operand (the output is written in place into
  // the first, else it has its own buffer), one for a loaded side's operand and
  // one for a unary side output when `side_buf`; then one tile row per one-row
  // operand.
  static int epi_stage_bytes(const Task& t, int mask, int depth, bool side_buf) {
    const int rows = (mask & 1) + ((mask >> 1) & 1);
    const int bcast = t.chain.n_loads - rows;
    const int bufs = (rows ? rows : 1) + ((mask & 8) ? 1 : 0) + (side_buf ? 1 : 0);
    return depth * bufs * tkd::kEpiBufBytes + bcast * tkd::kBcastBytes;
  }

  // Ring depth (chunks staged at once: 2, 4 or 8, at most the tile's chunks)
  // and whether a unary side output gets buffers of its own, for the staging
  // bytes `avail` an epilogue warp may use: the deepest ring first, side
  // buffers before depth (without them every chunk waits for its output's
  // store to leave shared memory).  Returns the bytes used, 0 if nothing fits.
  static int epi_stage_fit(const Task& t, int mask, int avail, int* depth, bool* side_buf) {
    const bool unary_side = t.has_side && !(mask & 8);
    const int nch = t.tile_n / 32;
    int top = tkd::kEpiMaxDepth;
    while (top > nch) top /= 2;
    for (int sb = unary_side ? 1 : 0; sb >= 0; --sb)
      for (int d = top; d >= 2; d /= 2) {
        const int need = epi_stage_bytes(t, mask, d, sb != 0);
        if (need <= avail) {
          *depth = d;
          *side_buf = sb != 0;
          return need;
        }
      }
    return 0;
  }

  // Recognise the chain shapes the kernel runs as compiled loops (FastKind).
  // Called once the task's refs have their vector modes.
  void classify_fast(Plan& plan, Task& t) const {
    tkd::Chain& ch = t.chain;
    ch.fast = tkd::FK_NONE;
    if (!ch.valid || t.vec != 8 || opt_.expr_forms >= 1) return;
    auto ref = [&](int slot) -> const Ref& { return plan.refs[t.ref_begin + ch.load_ref[slot]]; };
    auto contig = [&](int slot) { return slot < ch.n_loads && ref(slot).vmode == tkd::VM_CONTIG; };
    Shape sp(t.shape, t.shape + t.rank);
    Shape cs = contig_strides_of(sp);
    auto flat = [&](int slot) {
      if (slot >= ch.n_loads) return false;
      const Ref& r = ref(slot);
      for (int d = 0; d < t.rank; ++d)
        if (t.shape[d] > 1 && r.stride[d] != cs[d]) return false;
      return r.base % 8 == 0;
    };
    const tkd::ChainStep& s0 = ch.steps[0];
    const tkd::ChainStep& s1 = ch.steps[1];
    for (int i = 0; i < ch.n_steps; ++i)
      if (ch.steps[i].ext_mul && !(t.kind == tkd::T_GEMM_TC && i == 0)) return;
    auto axpy = [](const tkd::ChainStep& st, int ext) {
      return (st.op == tkd::OP_ADD || st.op == tkd::OP_SUB) && st.ext == ext && !st.second && !st.ext_mul;
    };
    if (t.kind == tkd::T_GEMM_TC) {
      if (ch.start != tkd::CH_ACC) return;
      if (ch.addmm_mode == tkd::AM_ACC && ch.bias == -1) {
        if (ch.n_steps == 0 && ch.n_loads == 0) ch.fast = tkd::FK_E_ACC;
        if (ch.n_steps == 1 && ch.n_loads == 1 && s0.op == tkd::OP_THRESH && s0.ext == tkd::EXT_LOAD0 &&
            !s0.second && contig(0))
          ch.fast = tkd::FK_E_ACC_THRESH;
        if (ch.n_steps == 1 && ch.n_loads == 1 && (s0.op == tkd::OP_ADD || s0.op == tkd::OP_SUB) &&
            s0.ext == tkd::EXT_LOAD0 && s0.second && contig(0))
          ch.fast = s0.ext_mul ? (s0.op == tkd::OP_ADD ? tkd::FK_E_MOMENTUM : tkd::FK_NONE) : tkd::FK_E_UPDATE;
      }
      for (int i = 0; i < ch.n_steps; ++i)
        if (ch.steps[i].ext_mul && ch.fast != tkd::FK_E_MOMENTUM) ch.fast = tkd::FK_NONE;
      if (ch.addmm_mode == tkd::AM_ACC && ch.bias == -1) {
      } else if (ch.addmm_mode == tkd::AM_SUM && ch.bias == 0 && contig(0)) {
        if (ch.n_steps == 0 && ch.n_loads == 1) ch.fast = tkd::FK_E_BIAS;
        if (ch.n_steps == 1 && ch.n_loads == 1 && s0.op == tkd::OP_RELU) ch.fast = tkd::FK_E_BIAS_RELU;
        if (ch.n_steps == 1 && ch.n_loads == 2 && axpy(s0, tkd::EXT_LOAD1) && contig(1)) ch.fast = tkd::FK_E_BIAS_AXPY;
      }
      return;
    }
    if (t.kind != tkd::T_POINTWISE && t.kind != tkd::T_REDUCE_ROW && t.kind != tkd::T_REDUCE_COL) return;
    if (ch.start != tkd::CH_LOAD || !flat(0)) return;
    if (ch.n_steps == 0 && ch.n_loads == 1) ch.fast = tkd::FK_L;
    if (ch.n_steps == 1 && ch.n_loads == 1) {
      if (s0.op == tkd::OP_MOV) ch.fast = tkd::FK_L_MOV;
      if (s0.op == tkd::OP_SQUARE) ch.fast = tkd::FK_L_SQUARE;
      if (s0.op == tkd::OP_MUL && s0.ext == tkd::EXT_CONST) ch.fast = tkd::FK_L_SCALE;
    }
    if (ch.n_steps == 1 && ch.n_loads == 2 && axpy(s0, tkd::EXT_LOAD1) && flat(1)) ch.fast = tkd::FK_L_AXPY;
    if (ch.n_steps == 2 && ch.n_loads == 2 && s0.op == tkd::OP_MUL && s0.ext == tkd::EXT_CONST &&
        axpy(s1, tkd::EXT_LOAD1) && flat(1))
      ch.fast = tkd::FK_L_SCALE_AXPY;
  }

  static Shape contig_strides_of(const Shape& sh) { return contig(sh); }

  // Compiled loops whose operands and output are all 16-bit keep twice as
  // many loads in flight (their raw 16-byte vectors fit in registers).
  int pointwise_unroll(const Plan& plan, const Task& t) const {
    if (t.vec != 8) return 1;
    if (t.chain.fast < tkd::FK_L || t.chain.fast > tkd::FK_L_SCALE_AXPY || t.out.dtype == TK_F32)
      return tkd::kPointwiseUnroll;
    for (int i = 0; i < t.chain.n_loads; ++i)
      if (plan.refs[t.ref_begin + t.chain.load_ref[i]].dtype == TK_F32) return tkd::kPointwiseUnroll;
    return tkd::kPointwiseUnroll16;
  }

  int items_pointwise(const Task& t) const {
    const int64_t per = int64_t(tkd::kThreads) * t.vec * std::max(1, t.pw_unroll);
    return int(ceil_div(t.numel, per));
  }

  // A pointwise task computing `op` (or copying a view when op == nullptr).
  Task lower_pointwise(Plan& plan, const OpInfo* op, const tk_tensor_spec* copy_src, const Shape& space,
                       Ref out, int round) {
    Task t = new_task(tkd::T_POINTWISE, space);
    t.code_begin = int(plan.code.size());
    t.ref_begin = int(plan.refs.size());
    bool chained = try_chain(plan, t, [&](ChainBuild& cb) {
      if (op) {
        cb.spine_op(*op, identity_map(int(space.size())));
      } else {
        cb.spine(*copy_src, identity_map(copy_src->rank));
        cb.step(tkd::OP_MOV, round, 0, 0, 0.f, 0.f);
      }
    });
    if (!chained) {
      Emit e{&plan, this, t.ref_begin, space};
      if (op) {
        e.op_value(*op, identity_map(int(space.size())), 0);
      } else {
        e.value(*copy_src, identity_map(copy_src->rank), 0);
        e.push(tkd::OP_MOV, 0, 0, 0, round);
      }
      t.code_len = int(plan.code.size()) - t.code_begin;
      t.n_refs = int(plan.refs.size()) - t.ref_begin;
    }
    t.out = out;
    finish_refs(plan, t);
    classify_fast(plan, t);
    t.pw_unroll = pointwise_unroll(plan, t);
    t.n_items = items_pointwise(t);
    return t;
  }

  // TMA view of one GEMM operand: the contiguous dim is the box's inner dim.
  // A is [M,K], B is [K,N]; "K-major" means K is the contiguous dim.
  // *mn_major: 0 K-major, 1 MN-major in 64-wide boxes, 2 MN-major in one box
  // of box_rows / 64 slabs (MN a multiple of 64, so no slab crosses the end).
  bool tma_operand(const tk_tensor_spec& v, bool is_a, int box_rows, TmaOperand* out, int* mn_major) const {
    int64_t base;
    int space, slot;
    location(v.buffer_id, &space, &slot, &base);
    base += v.offset;
    const int k_dim = is_a ? 1 : 0, mn_dim = is_a ? 0 : 1;
    TmaOperand o{};
    o.space = space;
    o.slot = slot;
    o.base_elems = base;
    o.dtype = v.dtype;
    o.box_inner = tkd::kTileK;
    if (v.strides[k_dim] == 1 && v.shape[k_dim] >= 1) {
      *mn_major = 0;
      o.inner = v.shape[k_dim];
      o.outer = v.shape[mn_dim];
      o.outer_stride = v.strides[mn_dim];
      o.box_outer = box_rows;
    } else if (v.strides[mn_dim] == 1) {
      *mn_major = 1;
      o.inner = v.shape[mn_dim];
      o.outer = v.shape[k_dim];
      o.outer_stride = v.strides[k_dim];
      o.box_outer = tkd::kTileK;
      if (box_rows > 64 && o.inner % 64 == 0) {
        o.chunks = box_rows / 64;
        *mn_major = 2;
      }
    } else {
      return false;
    }
    if (o.outer <= 1) o.outer_stride = round_up(std::max<int64_t>(o.inner, 8), 8);
    // TMA: 16-byte aligned start and row pitch, at least 16 bytes per row
    if (base % 8 || o.outer_stride % 8 || o.inner < 8 || o.outer_stride < o.inner) return false;
    if (o.inner >= (int64_t(1) << 32) || o.outer >= (int64_t(1) << 32)) return false;
    *out = o;
    return true;
  }

  // Index of TMA descriptor o in the plan, shared with an equal one.
  static int map_index(Plan& plan, const TmaOperand& o) {
    for (size_t i = 0; i < plan.tma.size(); ++i)
      if (plan.tma[i] == o) return int(i);
    plan.tma.push_back(o);
    return int(plan.tma.size()) - 1;
  }

  // A 32 x 32 epilogue-chunk descriptor over an [m, n] view with row stride
  // `row` (elements) at ref r's location.
  static TmaOperand chunk_map(const Ref& r, int64_t m, int64_t n, int64_t row) {
    TmaOperand o{};
    o.space = r.space;
    o.slot = r.slot;
    o.base_elems = r.base;
    o.dtype = r.dtype;
    o.inner = n;
    o.outer = m;
    o.outer_stride = row;
    o.box_inner = 32;
    o.box_outer = 32;
    o.swizzle = 1;
    return o;
  }

  // Descriptors for a staged epilogue (false, and nothing added, when they do
  // not fit the descriptor budget).
  bool epilogue_maps(Plan& plan, Task& t, int mask) const {
    std::vector<TmaOperand> want;
    auto add = [&](const Ref& r, int64_t row) {
      want.push_back(chunk_map(r, t.m, t.n, row));
      return int(want.size()) - 1;
    };
    int out = add(t.out, t.n), out2 = -1, ld0 = -1, ld1 = -1, sd = -1;
    if (t.has_side) out2 = add(t.out2, t.n);
    if (mask & 1) ld0 = add(plan.refs[t.ref_begin + t.chain.load_ref[0]], plan.refs[t.ref_begin + t.chain.load_ref[0]].stride[0]);
    if (mask & 2) ld1 = add(plan.refs[t.ref_begin + t.chain.load_ref[1]], plan.refs[t.ref_begin + t.chain.load_ref[1]].stride[0]);
    if (mask & 8) sd = add(t.side_ld, t.n);
    size_t extra = 0;
    for (const auto& o : want) {
      bool have = false;
      for (const auto& p : plan.tma) have = have || p == o;
      extra += have ? 0 : 1;
    }
    if (plan.tma.size() + extra > size_t(tkd::kMaxMaps)) return false;
    auto idx = [&](int i) { return i < 0 ? -1 : map_index(plan, want[size_t(i)]); };
    t.tma_out = idx(out);
    t.tma_out2 = idx(out2);
    t.tma_ld0 = idx(ld0);
    t.tma_ld1 = idx(ld1);
    t.tma_sd = idx(sd);
    return true;
  }

  bool try_tensor_core(Plan& plan, Task& t, const tk_tensor_spec& A, const tk_tensor_spec& B) const {
    if (!opt_.tensor_cores || A.dtype != B.dtype || (A.dtype != TK_BF16 && A.dtype != TK_F16)) return false;
    const int64_t M = t.m, N = t.n, K = t.k;
    if (M < 1 || N < 1 || K < 1) return false;
    if (plan.tma.size() + 2 > size_t(tkd::kMaxMaps)) return false;  // (a bound: equal maps are shared)
    // widest N tile that still spreads the tiles over the SMs (or the forced
    // width); a pair-tile launch deals 256-row tiles to pairs of SMs
    const int64_t tm = pair_ ? 2 * tkd::kTileM : tkd::kTileM, units = pair_ ? sms_ / 2 : sms_;
    int bn = pair_ ? 128 : 64;
    for (int cand : {256, 128}) {
      if (ceil_div(M, tm) * ceil_div(N, cand) >= (cand == 256 ? units : units / 2)) {
        bn = cand;
        break;
      }
    }
    if (opt_.tile_n > 0) bn = pair_ ? std::max(opt_.tile_n, 128) : opt_.tile_n;
    // each block of a pair stages half of B's columns
    const int bdiv = pair_ ? 2 : 1;  // each block loads half of B's columns
    TmaOperand ta, tb;
    int a_mn = 0, b_mn = 0;
    if (!tma_operand(A, true, tkd::kTileM, &ta, &a_mn) ||
        !tma_operand(B, false, (bn == 224 ? 256 : bn) / bdiv, &tb, &b_mn))
      return false;
    // A K-major B tile may also be 224 wide (seven 32-column chunks; MN-major
    // B tiles load whole 64-wide slabs).  Where the 256-wide tiles leave a
    // partial last wave on the SMs, take 224 if it makes the waves times the
    // bytes each k block stages (A tile + B tile) smaller: 4096 x 4096 outputs
    // take 512 tiles = 3.4 waves at 256, 608 = 4 waves at 224.
    if (opt_.tile_n == 0 && bn == 256 && b_mn == 0) {
      auto cost = [&](int w) {
        return ceil_div(ceil_div(M, tm) * ceil_div(N, w), units) * (tkd::kStageBytesA + w / bdiv * tkd::kTileK * 2);
      };
      if (cost(224) < cost(256)) bn = 224;
    }
    if (bn == 224 && b_mn != 0) bn = 256;
    if (bn == 224 && !tma_operand(B, false, bn / bdiv, &tb, &b_mn)) return false;
    t.kind = tkd::T_GEMM_TC;
    t.tile_m = int(tm);
    t.tile_n = bn;
    t.tiles_n = int(ceil_div(N, bn));
    t.k_blocks = int(ceil_div(K, tkd::kTileK));
    t.n_items = int(ceil_div(M, tm) * t.tiles_n);
    t.a_mn_major = a_mn;
    t.b_mn_major = b_mn;
    t.tma_a = map_index(plan, ta);
    t.tma_b = map_index(plan, tb);
    // instruction descriptor, kind::f16: D f32 (bits 4-5), A/B type (7-9, 10-12:
    // 0 f16, 1 bf16), A/B MN-major (15, 16), N >> 3 (17-22), M >> 4 (24-28)
    uint32_t ab = A.dtype == TK_BF16 ? 1u : 0u;
    // (a shared-B pair's blocks each run their own 128-row MMAs)
    const int64_t mma_m = pair_ == 1 ? tm : tkd::kTileM;
    t.idesc = (1u << 4) | (ab << 7) | (ab << 10) | (uint32_t(a_mn != 0) << 15) | (uint32_t(b_mn != 0) << 16) |
              (uint32_t(bn >> 3) << 17) | (uint32_t(mma_m >> 4) << 24);
    // Split-K when the tiles leave most SMs idle and each tile has a long K
    // loop (at least 8 k blocks per split).
    t.k_splits = 1;
    t.kb_split = t.k_blocks;
    if (opt_.split_k && !pair_ && 2 * int64_t(t.n_items) <= sms_ && t.k_blocks >= 16 && N % 8 == 0) {
      const int splits = int(std::min<int64_t>({int64_t(t.k_blocks / 8), int64_t(sms_ / t.n_items), 8}));
      if (splits >= 2) {
        t.kb_split = int(ceil_div(t.k_blocks, splits));
        t.k_splits = int(ceil_div(t.k_blocks, t.kb_split));
        t.n_items *= t.k_splits;
      }
    }
    return true;
  }

  // The side output of fused GEMM or reduction mm (if any) as one chain step
  // on the final value.
  void attach_side(Task& t, const OpInfo& mm) const {
    auto it = side_.find(mm.index);
    if (it == side_.end()) return;
    const OpInfo& op = ops_[it->second];
    const int fin = fused_.at(mm.index).final_buf;
    tkd::ChainStep st{};
    st.round = uint8_t(op.out.dtype);
    st.ext = tkd::EXT_NONE;
    if (op.kind == TK_OP_ADD || op.kind == TK_OP_SUB) {
      // a loaded side: final +/- alpha*input or input +/- alpha*final, the
      // input read at the output's flat index from side_ld
      const bool root_first = op.in[0].t.buffer_id == fin;
      const tk_tensor_spec& in = op.in[root_first ? 1 : 0].t;
      st.op = op.kind == TK_OP_ADD ? tkd::OP_ADD : tkd::OP_SUB;
      st.imm = f32(op.alpha);
      st.ext = tkd::EXT_LOAD1;
      st.second = root_first ? 0 : 1;
      Ref r{};
      int64_t base;
      location(in.buffer_id, &r.space, &r.slot, &base);
      r.dtype = in.dtype;
      r.base = base + in.offset;
      r.vmode = tkd::VM_CONTIG;
      t.side_ld = r;
    } else if (op.kind == TK_OP_MUL) {  // x*c (= c*x), -x, or a cast
      const bool root_first = !op.in[0].scalar && op.in[0].t.buffer_id == fin;
      st.op = tkd::OP_MUL;
      st.ext = tkd::EXT_CONST;
      st.cval = f32(root_first ? op.in[1].value : op.in[0].value);
    } else {
      st.op = op.kind == TK_OP_NEG ? tkd::OP_NEG : tkd::OP_MOV;
    }
    t.has_side = 1;
    t.side = st;
    t.out2 = out_ref(op.out.buffer_id);
  }

  // A split-K GEMM (k_splits > 1) leaves its epilogue to a second task.
  std::vector<Task> lower_gemm_tasks(Plan& plan, const OpInfo& mm, int64_t* scratch_cursor) {
    Task t = lower_gemm(plan, mm);
    if (t.kind != tkd::T_GEMM_TC || t.k_splits <= 1) return {t};
    Task f = t;
    f.kind = tkd::T_SPLITK_FINAL;
    f.tma_a = f.tma_b = -1;
    f.n_items = int(ceil_div(t.numel, int64_t(tkd::kThreads) * t.vec));
    f.scratch = t.scratch = tkd::kHeaderUnits + arena_total_ + *scratch_cursor;
    *scratch_cursor += round_up(int64_t(t.k_splits) * t.numel, 64);
    t.chain.fast = tkd::FK_NONE;
    f.chain.fast = tkd::FK_NONE;
    return {t, f};
  }

  Task lower_gemm(Plan& plan, const OpInfo& mm) {
    size_t base = mm.kind == TK_OP_ADDMM ? 1 : 0;
    const tk_tensor_spec &A = mm.in[base].t, &B = mm.in[base + 1].t;
    int64_t M = A.shape[0], K = A.shape[1], N = B.shape[1];
    Shape space = {M, N};
    Task t = new_task(tkd::T_GEMM_SIMT, space);
    t.m = int(M);
    t.n = int(N);
    t.k = int(K);
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) throw Error(TK_ERR_UNSUPPORTED, "GEMM too large");
    auto operand_ref = [&](const tk_tensor_spec& v) {
      Ref r{};
      int64_t b;
      location(v.buffer_id, &r.space, &r.slot, &b);
      r.dtype = v.dtype;
      r.base = b + v.offset;
      r.stride[0] = v.strides[0];
      r.stride[1] = v.strides[1];
      return r;
    };
    t.a = operand_ref(A);
    t.b = operand_ref(B);
    t.a_kcontig = A.strides[1] == 1 || A.shape[0] <= 1;
    t.b_ncontig = B.strides[1] == 1 || B.shape[0] <= 1;
    // One row (the online, batch-1 step) with K-contiguous, 16-byte aligned
    // operands: a warp per output, vector loads along K, a fixed-order tree sum.
    const bool gemv = M == 1 && K % 8 == 0 && A.strides[1] == 1 && B.strides[0] == 1 &&
                      (N <= 1 || B.strides[1] % 8 == 0) && t.a.base % 8 == 0 && t.b.base % 8 == 0;
    if (gemv) {
      t.kind = tkd::T_GEMV;
      t.n_items = int(ceil_div(N, tkd::kThreads / 32));
    } else if (!try_tensor_core(plan, t, A, B)) {
      // CUDA-core tile: the largest of 64/32/16 that still gives every SM a tile
      int tile = 16;
      for (int cand : {64, 32}) {
        if (ceil_div(M, cand) * ceil_div(N, cand) >= sms_) {
          tile = cand;
          break;
        }
      }
      t.tile_m = t.tile_n = tile;
      t.tiles_n = int(ceil_div(N, tile));
      t.n_items = int(ceil_div(M, tile) * ceil_div(N, tile));
    }
    if (M == 0 || N == 0) t.n_items = 0;

    // epilogue: addmm formula, rounding to the GEMM dtype, then the chain
    t.code_begin = int(plan.code.size());
    t.ref_begin = int(plan.refs.size());
    auto fused_it = fused_.find(mm.index);
    bool chained = try_chain(plan, t, [&](ChainBuild& cb) {
      tkd::Chain& ch = cb.ch;
      ch.start = tkd::CH_ACC;
      ch.round0 = mm.out.dtype;
      ch.alpha = f32(mm.alpha);
      ch.beta = f32(mm.beta);
      ch.bias = -1;
      cb.started = true;
      if (mm.kind == TK_OP_MM) {
        ch.addmm_mode = tkd::AM_ACC;
      } else {
        ch.addmm_mode = (mm.alpha == 0.0 && mm.beta == 0.0) ? tkd::AM_ZERO
                        : mm.beta == 0.0                   ? tkd::AM_ALPHA
                        : mm.alpha == 0.0                  ? tkd::AM_BETA
                        : (mm.alpha == 1.0 && mm.beta == 1.0) ? tkd::AM_SUM
                                                             : tkd::AM_FULL;
        const Operand& o = mm.in[0];
        if (ch.addmm_mode != tkd::AM_ZERO && ch.addmm_mode != tkd::AM_ALPHA) {
          if (o.scalar) {
            ch.bias = 2;
            ch.bias_const = f32(o.value);
          } else if (inline_.count(o.t.buffer_id)) {
            cb.fail = true;
          } else {
            std::vector<int> m(o.t.rank, -1);
            for (int d = 0; d < o.t.rank; ++d) m[d] = o.t.shape[d] == 1 ? -1 : d + 2 - o.t.rank;
            ch.bias = cb.load_slot(o.t, m);
          }
        }
      }
      int root = mm.out.buffer_id;
      if (fused_it != fused_.end())
        for (int ci : fused_it->second.chain) {
          cb.root_buf = root;
          cb.spine_op(ops_[ci], identity_map(2));
          root = ops_[ci].out.buffer_id;
        }
    });
    attach_side(t, mm);
    if (chained) {
      int out_buf = fused_it != fused_.end() ? fused_it->second.final_buf : mm.out.buffer_id;
      t.out = out_ref(out_buf);
      finish_refs(plan, t);
      classify_fast(plan, t);
      return t;
    }
    Emit e{&plan, this, t.ref_begin, space};
    std::vector<int> idmap = identity_map(2);
    int rd = mm.out.dtype;
    if (mm.kind == TK_OP_MM) {
      e.push(tkd::OP_ACC, 0, 0, 0, rd);
    } else {
      auto bias = [&](int reg) {
        const Operand& o = mm.in[0];
        if (o.scalar) {
          e.push(tkd::OP_CONST, reg, 0, 0, TK_F32, f32(o.value));
        } else {
          std::vector<int> m(o.t.rank, -1);
          for (int d = 0; d < o.t.rank; ++d) m[d] = o.t.shape[d] == 1 ? -1 : d + 2 - o.t.rank;
          e.value(o.t, m, reg);
        }
      };
      if (mm.alpha == 0.0 && mm.beta == 0.0) {
        e.push(tkd::OP_CONST, 0, 0, 0, rd, 0.f);
      } else if (mm.beta == 0.0) {
        e.push(tkd::OP_ACC, 0, 0, 0, TK_F32);
        e.push(tkd::OP_CONST, 1, 0, 0, TK_F32, f32(mm.alpha));
        e.push(tkd::OP_MUL, 0, 0, 1, rd);
      } else if (mm.alpha == 0.0) {
        bias(0);
        e.push(tkd::OP_CONST, 1, 0, 0, TK_F32, f32(mm.beta));
        e.push(tkd::OP_MUL, 0, 0, 1, rd);
      } else {
        e.push(tkd::OP_ACC, 0, 0, 0, TK_F32);
        if (mm.alpha != 1.0) {
          e.push(tkd::OP_CONST, 1, 0, 0, TK_F32, f32(mm.alpha));
          e.push(tkd::OP_MUL, 0, 0, 1, TK_F32);
        }
        bias(1);
        if (mm.beta != 1.0) {
          e.push(tkd::OP_CONST, 2, 0, 0, TK_F32, f32(mm.beta));
          e.push(tkd::OP_MUL, 1, 1, 2, TK_F32);
        }
        e.push(tkd::OP_ADD, 0, 0, 1, rd, 1.0f);
      }
    }
    int out_buf = mm.out.buffer_id;
    auto it = fused_.find(mm.index);
    if (it != fused_.end()) {
      for (int ci : it->second.chain) {
        const OpInfo& c = ops_[ci];
        e.root_buf = out_buf;
        // operands go to registers 1.., the running root stays in register 0
        e.op_value(c, idmap, 1);
        e.push(tkd::OP_MOV, 0, 1, 1, TK_F32);
        out_buf = c.out.buffer_id;
      }
      e.root_buf = -1;
    }
    t.code_len = int(plan.code.size()) - t.code_begin;
    t.n_refs = int(plan.refs.size()) - t.ref_begin;
    t.out = out_ref(out_buf);
    finish_refs(plan, t);
    classify_fast(plan, t);
    return t;
  }

  // Reduction as one task (parts == 1) or partials + a final task.
  std::vector<Task> lower_reduction(Plan& plan, const OpInfo& op, int64_t* scratch_cursor) {
    const tk_tensor_spec& src = op.in[0].t;
    std::vector<bool> red = reduced_mask(op);
    std::vector<int> kept, reduced;
    for (int d = 0; d < src.rank; ++d) (red[d] ? reduced : kept).push_back(d);
    bool row = src.rank == 0 || red[src.rank - 1];
    std::vector<int> perm;
    if (row) {
      perm = kept;
      perm.insert(perm.end(), reduced.begin(), reduced.end());
    } else {
      perm = reduced;
      perm.insert(perm.end(), kept.begin(), kept.end());
    }
    Shape space;
    for (int d : perm) space.push_back(src.shape[d]);
    std::vector<int> dimmap(src.rank);
    for (size_t j = 0; j < perm.size(); ++j) dimmap[perm[j]] = int(j);
    int64_t n_out = 1, n_red = 1;
    for (int d : kept) n_out *= src.shape[d];
    for (int d : reduced) n_red *= src.shape[d];

    Task t = new_task(row ? tkd::T_REDUCE_ROW : tkd::T_REDUCE_COL, space);
    t.code_begin = int(plan.code.size());
    t.ref_begin = int(plan.refs.size());
    if (!try_chain(plan, t, [&](ChainBuild& cb) { cb.spine(src, dimmap); })) {
      Emit e{&plan, this, t.ref_begin, space};
      e.value(src, dimmap, 0);
      t.code_len = int(plan.code.size()) - t.code_begin;
      t.n_refs = int(plan.refs.size()) - t.ref_begin;
    }
    auto fused_it = fused_.find(op.index);
    t.out = out_ref(fused_it != fused_.end() ? fused_it->second.final_buf : op.out.buffer_id);
    t.red_mean = op.kind == TK_OP_MEAN;
    t.size_f = float(double(n_red));
    if (row) {
      // vectors run along the reduced dims: the innermost index dim is reduced
      t.vec = (!reduced.empty() && src.shape[src.rank - 1] % 8 == 0 && n_red > 0) ? 8 : 1;
      t.red_outer = n_out;
      t.red_inner = n_red;
      int64_t parts = 1;
      if (n_out < sms_ && n_red > 16384) {
        parts = std::min<int64_t>(ceil_div(n_red, 8192), std::max<int64_t>(1, ceil_div(2 * sms_, n_out)));
        parts = std::min<int64_t>(parts, 1024);
      }
      int64_t step = int64_t(tkd::kThreads) * t.vec;
      t.part_len = round_up(ceil_div(std::max<int64_t>(n_red, 1), parts), step);
      t.parts = int(ceil_div(std::max<int64_t>(n_red, 1), t.part_len));
      t.n_items = int(n_out * t.parts);
    } else {
      t.red_outer = n_red;
      t.red_inner = n_out;
      int64_t cw = 32 * t.vec;
      int64_t chunks = ceil_div(n_out, cw);
      int64_t parts = 1;
      if (chunks < sms_ / 2 && n_red > 512)
        parts = std::min<int64_t>(ceil_div(n_red, 128), std::max<int64_t>(1, ceil_div(2 * sms_, chunks)));
      t.part_len = ceil_div(std::max<int64_t>(n_red, 1), parts);
      t.parts = int(ceil_div(std::max<int64_t>(n_red, 1), t.part_len));
      t.n_items = int(chunks * t.parts);
    }
    if (t.parts <= 1 && fused_it != fused_.end()) {
      lower_post_chain(plan, t, op, fused_it->second);
      attach_side(t, op);
    }
    finish_refs(plan, t);
    classify_fast(plan, t);
    // compiled sources over 16-bit operands stream with more loads in flight
    // (pw_unroll marks them, as for pointwise tasks; the output type does not matter)
    t.pw_unroll = tkd::kPointwiseUnroll;
    // (only long parts: a short one gains nothing from deeper loads and pays
    // for the larger loop)
    const bool long_part = row ? t.part_len >= 16 * tkd::kThreads * 8 : t.part_len >= 128;
    if (long_part && t.vec == 8 && t.chain.fast >= tkd::FK_L && t.chain.fast <= tkd::FK_L_SCALE_AXPY) {
      t.pw_unroll = tkd::kPointwiseUnroll16;
      for (int i = 0; i < t.chain.n_loads; ++i)
        if (plan.refs[t.ref_begin + t.chain.load_ref[i]].dtype == TK_F32) t.pw_unroll = tkd::kPointwiseUnroll;
    }
    if (n_out == 0) t.n_items = 0;
    if (t.parts <= 1) {
      t.parts = 1;
      return {t};
    }
    t.scratch = tkd::kHeaderUnits + arena_total_ + *scratch_cursor;
    *scratch_cursor += round_up(n_out * t.parts, 64);
    Task f = new_task(tkd::T_REDUCE_FINAL, Shape{n_out});
    f.out = t.out;
    f.red_mean = t.red_mean;
    f.size_f = t.size_f;
    f.parts = t.parts;
    f.scratch = t.scratch;
    f.red_outer = n_out;
    f.final_block = n_out < 64;
    f.n_items = int(f.final_block ? n_out : ceil_div(n_out, tkd::kThreads));
    f.code_begin = int(plan.code.size());
    f.ref_begin = int(plan.refs.size());
    if (fused_it != fused_.end()) {
      lower_post_chain(plan, f, op, fused_it->second);
      attach_side(f, op);
      finish_refs(plan, f);
    }
    return {t, f};
  }

  // The chain after reduction r, evaluated per finished output of task t.
  void lower_post_chain(Plan& plan, Task& t, const OpInfo& r, const Fused& fu) {
    const Shape out_shape = shape_of(r.out);
    t.post_rank = int(out_shape.size());
    for (size_t d = 0; d < out_shape.size(); ++d) t.post_shape[d] = out_shape[d];
    ChainBuild cb{&plan, this, t.ref_begin};
    cb.ch.start = tkd::CH_ACC;
    cb.ch.addmm_mode = tkd::AM_ACC;
    cb.ch.bias = -1;
    cb.ch.round0 = r.out.dtype;
    cb.started = true;
    int root = r.out.buffer_id;
    for (int ci : fu.chain) {
      cb.root_buf = root;
      cb.spine_op(ops_[ci], identity_map(int(out_shape.size())));
      root = ops_[ci].out.buffer_id;
    }
    if (cb.fail) throw Error(TK_ERR_INVALID, "internal: reduction epilogue is not a chain");
    cb.ch.valid = 1;
    // p -/+ a*round(v) with p contiguous over the outputs: the compiled update
    const tkd::ChainStep& s0 = cb.ch.steps[0];
    if (opt_.expr_forms == 0 && cb.ch.n_steps == 1 && cb.ch.n_loads == 1 && s0.ext == tkd::EXT_LOAD0 && s0.second &&
        !s0.ext_mul && (s0.op == tkd::OP_ADD || s0.op == tkd::OP_SUB)) {
      const Ref& r = plan.refs[t.ref_begin + cb.ch.load_ref[0]];
      bool flat = true;
      Shape cs = contig(out_shape);
      for (int d = 0; d < t.post_rank; ++d)
        if (out_shape[d] > 1 && r.stride[d] != cs[d]) flat = false;
      if (flat) cb.ch.fast = tkd::FK_E_UPDATE;
    }
    t.post = cb.ch;
    t.n_refs = int(plan.refs.size()) - t.ref_begin;
  }

  // ------------------------------------------------------------ the plan

  Plan plan_once() {
    fused_.clear();
    side_.clear();
    fused_skip_.clear();
    inline_.clear();
    schedule_.clear();
    writer_.clear();
    direct_.clear();
    binding_.clear();
    arena_off_.clear();
    arena_units_.clear();
    arena_total_ = 0;

    detect_epilogues();
    detect_reduction_epilogues();
    detect_side_outputs();
    choose_inline();
    build_schedule();
    choose_direct_aliases();
    check_sides();
    choose_bindings();
    // Stages first with a private slot per intermediate value, then the arena
    // reuses a slot only for a value written in a later stage than the last
    // read of its previous occupant: slot reuse never adds a barrier.
    plan_arena(false);
    lower_and_stage();
    arena_off_.clear();
    arena_units_.clear();
    plan_arena(true);
    return lower_and_stage();
  }

  std::vector<int> stage_of_;  // stage of each schedule position (last stage for split reductions)
  // split reductions (by partials scratch offset) whose final pass could run
  // in the stage of their partial sums: its writes (and reads) conflict with
  // no other task of that stage
  std::set<int64_t> fold_ok_;

  Plan lower_and_stage() {
    stage_of_.assign(schedule_.size(), 0);
    fold_ok_.clear();
    Plan plan;
    std::vector<std::vector<Task>> stages(1);
    std::vector<Region> stage_reads, stage_writes;
    int64_t scratch = 0;
    int split = 0;
    // Final passes of split reductions wait here and join the next stage
    // that starts for any reason (or the one a reader of their result forces),
    // instead of forcing a barrier right after their partial sums.
    struct Pending {
      Task f;
      size_t pos;
      std::vector<Region> reads, writes;
      bool reads_operands = false;  // the final pass reads the op's operands (epilogue chain)
    };
    std::vector<Pending> pending;
    auto barrier = [&]() {
      stages.emplace_back();
      stage_reads.clear();
      stage_writes.clear();
      for (auto& p : pending) {
        stages.back().push_back(p.f);
        stage_of_[p.pos] = int(stages.size()) - 1;
        if (p.f.post.valid || p.reads_operands) stage_reads.insert(stage_reads.end(), p.reads.begin(), p.reads.end());
        stage_writes.insert(stage_writes.end(), p.writes.begin(), p.writes.end());
      }
      pending.clear();
    };
    auto conflicts_pending = [&](const std::vector<Region>& reads, const std::vector<Region>& writes) {
      for (const auto& p : pending) {
        for (const auto& w : p.writes) {
          for (const auto& r : reads)
            if (overlap(w, r)) return true;
          for (const auto& r : writes)
            if (overlap(w, r)) return true;
        }
        if (p.f.post.valid || p.reads_operands)
          for (const auto& r : p.reads)
            for (const auto& w : writes)
              if (overlap(r, w)) return true;
      }
      return false;
    };
    auto hazard = [&](const std::vector<Region>& reads, const std::vector<Region>& writes) {
      for (const auto& w : stage_writes) {
        for (const auto& r : reads)
          if (overlap(w, r)) return true;
        for (const auto& r : writes)
          if (overlap(w, r)) return true;
      }
      for (const auto& r : stage_reads)
        for (const auto& w : writes)
          if (overlap(r, w)) return true;
      return false;
    };

    for (size_t pos = 0; pos < schedule_.size(); ++pos) {
      const int s = schedule_[pos];
      const OpInfo& op = ops_[s];
      std::vector<Region> reads, writes;
      for (const auto& v : reads_of(s)) read_regions(v, reads);
      for (int b : stored_buffers(s)) writes.push_back(storage_region(b));
      if (is_red(op.kind)) {
        std::vector<Task> ts = lower_reduction(plan, op, &scratch);
        for (auto& t : ts) t.op_index = op.index;
        if (ts.size() == 2) {
          ++split;
          if (conflicts_pending(reads, {})) barrier();
          while (hazard(reads, {})) barrier();
          // (tasks placed in this stage later never conflict with a pending
          // final pass: they would start the next stage first)
          if (ts[1].kind == tkd::T_REDUCE_FINAL && !ts[1].final_block &&
              !hazard(ts[1].post.valid ? reads : std::vector<Region>{}, writes))
            fold_ok_.insert(ts[1].scratch);
          stages.back().push_back(ts[0]);
          stage_reads.insert(stage_reads.end(), reads.begin(), reads.end());
          // the final pass also reads a reduction epilogue's operands
          pending.push_back({ts[1], pos, reads, writes});
          continue;
        }
        if (conflicts_pending(reads, writes)) barrier();
        while (hazard(reads, writes)) barrier();
        stages.back().push_back(ts[0]);
      } else {
        std::vector<Task> ts =
            is_mm(op.kind) ? lower_gemm_tasks(plan, op, &scratch)
                           : std::vector<Task>{lower_pointwise(plan, &op, nullptr, shape_of(op.out),
                                                               out_ref(op.out.buffer_id), op.out.dtype)};
        for (auto& t : ts) t.op_index = op.index;
        if (ts.size() == 2) {
          // split-K: the partial products now, their sum and the epilogue with the next stage
          if (conflicts_pending(reads, {})) barrier();
          while (hazard(reads, {})) barrier();
          stages.back().push_back(ts[0]);
          stage_reads.insert(stage_reads.end(), reads.begin(), reads.end());
          pending.push_back({ts[1], pos, reads, writes, true});
          continue;
        }
        if (conflicts_pending(reads, writes)) barrier();
        while (hazard(reads, writes)) barrier();
        stages.back().push_back(ts[0]);
      }
      stage_of_[pos] = int(stages.size()) - 1;
      stage_reads.insert(stage_reads.end(), reads.begin(), reads.end());
      stage_writes.insert(stage_writes.end(), writes.begin(), writes.end());
    }

    if (!pending.empty()) barrier();

    // End-of-kernel output copies, then transactional commits of in-place outputs.
    int copies = 0;
    bool needs_copy = false;
    for (size_t j = 0; j < outputs_.size(); ++j) {
      auto b = binding_.find(outputs_[j].buffer_id);
      if (b == binding_.end() || b->second != int(j)) needs_copy = true;
    }
    if (!stage_writes.empty() && needs_copy) barrier();
    bool copied = false;
    for (size_t j = 0; j < outputs_.size(); ++j) {
      if (inplace_.count(int(j))) continue;
      auto b = binding_.find(outputs_[j].buffer_id);
      if (b != binding_.end() && b->second == int(j)) continue;
      Ref out{};
      out.space = tkd::SP_OUT;
      out.slot = int(j);
      out.dtype = outputs_[j].dtype;
      stages.back().push_back(
          lower_pointwise(plan, nullptr, &outputs_[j], shape_of(outputs_[j]), out, outputs_[j].dtype));
      copied = true;
      ++copies;
    }
    if (!inplace_.empty()) {
      bool any_commit = false;
      for (const auto& kv : inplace_)
        if (!direct_.count(kv.first)) any_commit = true;
      if (any_commit && copied) barrier();
      for (const auto& kv : inplace_) {
        if (direct_.count(kv.first)) continue;
        const auto& spec = outputs_[kv.first];
        Ref out{};
        out.space = tkd::SP_OUT;
        out.slot = kv.first;
        out.dtype = spec.dtype;
        stages.back().push_back(lower_pointwise(plan, nullptr, &spec, shape_of(spec), out, spec.dtype));
        ++copies;
      }
    }
    while (stages.size() > 1 && stages.back().empty()) stages.pop_back();

    // Flatten: tensor-core tasks first inside each stage.
    int tc_ops = 0;
    int fold_used = 0;
    std::vector<bool> emptied(stages.size(), false);
    for (size_t si = 0; si < stages.size(); ++si) {
      auto& st = stages[si];
      if (emptied[si] && st.empty()) continue;  // its final passes all ran in the stage before
      std::stable_sort(st.begin(), st.end(), [](const Task& a, const Task& b) {
        return (a.kind == tkd::T_GEMM_TC) > (b.kind == tkd::T_GEMM_TC);
      });
      Stage S{};
      S.task_begin = int(plan.tasks.size());
      S.code_lo = S.ref_lo = INT32_MAX;
      S.code_hi = S.ref_hi = 0;
      for (auto& t : st) {
        t.stage = int(plan.stages.size());
        if (t.code_len) {
          S.code_lo = std::min(S.code_lo, t.code_begin);
          S.code_hi = std::max(S.code_hi, t.code_begin + t.code_len);
        }
        if (t.n_refs) {
          S.ref_lo = std::min(S.ref_lo, t.ref_begin);
          S.ref_hi = std::max(S.ref_hi, t.ref_begin + t.n_refs);
        }
        S.n_items += t.n_items;
        if (t.kind == tkd::T_GEMM_TC) {
          S.n_tc_items += t.n_items;
          ++tc_ops;
        }
        plan.tasks.push_back(t);
      }
      S.task_end = int(plan.tasks.size());
      // a stage's compiled row and column reductions run on warps 2 and 3
      // while its tensor-core tiles run (the same additions in the same
      // order), as long as they fit in 90 % of the tiles' time: one warp
      // streams an item at ~2 GB/s (+1 us), a block's tiles take ~0.4 us per
      // 64-deep k block each (+4 us of epilogue); only beside long tiles (15
      // or more k blocks)
      if (S.n_tc_items > 0 && opt_.overlap_reductions) {
        double tile_us = 0.0;
        for (int i = S.task_begin; i < S.task_end; ++i)
          if (plan.tasks[i].kind == tkd::T_GEMM_TC) tile_us = std::max(tile_us, 4.0 + 0.4 * plan.tasks[i].kb_split);
        const double units = pair_ ? sms_ / 2 : sms_;
        const double tiles_us = std::ceil(S.n_tc_items / units) * tile_us;
        // (2 runs every eligible reduction beside the tiles: for tests)
        const bool force = opt_.overlap_reductions == 2;
        double bg_us = tile_us < 10.0 && !force ? 1e30 : 0.0;
        for (int i = S.task_begin; i < S.task_end; ++i) {
          Task& t = plan.tasks[i];
          if ((t.kind == tkd::T_REDUCE_ROW || t.kind == tkd::T_REDUCE_COL) && t.vec == 8 &&
              (t.chain.fast == tkd::FK_L || t.chain.fast == tkd::FK_L_SQUARE) && t.chain.n_loads == 1 &&
              t.n_items > 0) {
            // (a 16-bit operand: the kernel compiles these per type)
            const int dt = plan.refs[t.ref_begin + t.chain.load_ref[0]].dtype;
            const double item_us = 1.0 + double(t.numel) / double(t.n_items) * 2.0 / 2e3;
            const double us = std::ceil(t.n_items / (2.0 * sms_)) * item_us;
            if ((dt == TK_BF16 || dt == TK_F16) && (force || bg_us + us <= 0.9 * tiles_us)) {
              t.bg = dt;
              S.has_bg = 1;
              bg_us += us;
            }
          }
        }
      }
      // a split column reduction beside the tiles takes its final pass along
      // (Task::fold): the warp adding a chunk's last part finishes the chunk,
      // so the final's own stage (and barrier) can go when nothing else is in it
      if (S.has_bg && si + 1 < stages.size()) {
        for (int i = S.task_begin; i < S.task_end; ++i) {
          const Task t = plan.tasks[i];
          if (!t.bg || t.kind != tkd::T_REDUCE_COL || t.parts <= 1 || !fold_ok_.count(t.scratch)) continue;
          auto& next = stages[si + 1];
          auto it = std::find_if(next.begin(), next.end(), [&](const Task& f) {
            return f.kind == tkd::T_REDUCE_FINAL && f.scratch == t.scratch && !f.final_block;
          });
          const int chunks = t.n_items / t.parts;
          if (it == next.end() || it->n_items != chunks || fold_used + chunks > tkd::kFoldCounters) continue;
          Task f = *it;
          next.erase(it);
          emptied[si + 1] = true;
          f.stage = int(plan.stages.size());
          f.folded = 1;
          f.n_items = 0;  // run by the part items' warps only
          plan.tasks.push_back(f);
          plan.tasks[i].fold = int(plan.tasks.size());
          plan.tasks[i].fold_ctr = fold_used;
          fold_used += chunks;
          S.task_end = int(plan.tasks.size());
          if (f.code_len) {
            S.code_lo = std::min(S.code_lo, f.code_begin);
            S.code_hi = std::max(S.code_hi, f.code_begin + f.code_len);
          }
          if (f.n_refs) {
            S.ref_lo = std::min(S.ref_lo, f.ref_begin);
            S.ref_hi = std::max(S.ref_hi, f.ref_begin + f.n_refs);
          }
        }
      }
      S.light_items = light_items(plan, S);
      if (S.code_lo > S.code_hi) S.code_lo = S.code_hi = 0;
      if (S.ref_lo > S.ref_hi) S.ref_lo = S.ref_hi = 0;
      plan.stages.push_back(S);
      plan.max_items = std::max(plan.max_items, S.n_items);
    }

    plan.arena_units = arena_total_;
    plan.workspace_units = tkd::kHeaderUnits + arena_total_ + scratch;
    plan.uses_tc = tc_ops > 0;
    int max_bn = 0;
    for (const auto& t : plan.tasks)
      if (t.kind == tkd::T_GEMM_TC) max_bn = std::max(max_bn, t.tile_n);
    // Ring slots sized for the widest tile: smaller rings leave more of the
    // SM's unified L1/shared memory to the L1 cache.
    // (a pair-tile launch stages half of each B tile per block)
    plan.pair = tc_ops > 0 ? pair_ : 0;
    plan.tmem_cols = 32;
    while (plan.tmem_cols < 2 * max_bn) plan.tmem_cols *= 2;
    // (a shared-B pair keeps whole B tiles: each block's half arrives by multicast)
    plan.ring_stage_bytes = tkd::kStageBytesA + (plan.pair == 1 ? max_bn / 2 : max_bn) * tkd::kTileK * 2;
    const size_t ring = 1024 + size_t(plan.pair == 1 ? tkd::kPairStages : tkd::kStages) * plan.ring_stage_bytes;
    // every staged task may use the staging bytes left beside the ring
    const int avail = ring < size_t(tkd::kDynSmemBudget) ? int((size_t(tkd::kDynSmemBudget) - ring) / 4) : 0;
    for (auto& t : plan.tasks) {
      t.epi_stage = 0;
      t.epi_depth = 0;
      t.epi_dtype = 0;
      t.tma_out = t.tma_out2 = t.tma_ld0 = t.tma_ld1 = t.tma_sd = -1;
      int mask = epi_stage_mask(plan, t), depth = 0;
      bool side_buf = false;
      if (mask < 0) continue;
      const int need = epi_stage_fit(t, mask, opt_.epi_stage_bytes > 0 ? std::min(avail, opt_.epi_stage_bytes) : avail,
                                     &depth, &side_buf);
      if (need == 0 || !epilogue_maps(plan, t, mask)) continue;
      plan.epi_warp_bytes = std::max(plan.epi_warp_bytes, need);
      t.epi_stage = mask | (side_buf ? 16 : 0);
      t.epi_depth = depth;
      t.epi_dtype = epi_uniform_dtype(plan, t);
    }
    plan.smem_bytes = plan.uses_tc ? ring + 4 * size_t(plan.epi_warp_bytes) : 1024 + size_t(tkd::kWorkFloats) * 4;
    for (const auto& s : inputs_) plan.input_bytes.push_back(extent_of(s) * esize(s.dtype));
    for (const auto& s : outputs_) plan.output_bytes.push_back(numel(s) * esize(s.dtype));
    for (const auto& kv : inplace_) plan.inplace.push_back({kv.first, kv.second});

    tk_plan_stats& st = plan.stats;
    st.materialized_ops = int(schedule_.size());
    st.inlined_ops = int(inline_.size());
    st.fused_epilogues = int(fused_.size());
    st.tensor_core_ops = tc_ops;
    st.cta_pairs = plan.pair;
    st.stages = int(plan.stages.size());
    st.grid_barriers = st.stages - 1;
    st.direct_outputs = int(binding_.size());
    st.direct_state_commits = int(direct_.size());
    st.max_work_items = plan.max_items;
    st.output_copies = copies;
    st.split_reductions = split;
    st.workspace_elements = plan.workspace_units;
    st.arena_elements = arena_total_;
    st.tasks = int(plan.tasks.size());
    st.tma_descriptors = int(plan.tma.size());
    for (const auto& t : plan.tasks) {
      if (t.chain.valid && t.chain.fast != tkd::FK_NONE) ++st.compiled_tasks;
      else if (t.chain.valid) ++st.chain_tasks;
    }
    return plan;
  }
};

}  // namespace

Plan build_plan(const tk_program_desc& desc, const tk_options& opt, int sm_count) {
  Planner p(desc, opt, sm_count);
  return p.run();
}

}  // namespace tkp
