// The persistent training-step kernel for sm_103a (GB300): device code.
//
// This header holds the kernel body; kernel_plain.cu, kernel_tc_small.cu and
// kernel_tc_large.cu each instantiate one entry point from it, so the three
// variants compile in parallel.  launch.cu launches them.
//
// One cooperative launch runs a whole training step.  Every block walks the
// device op table stage by stage; inside a stage the work items of all tasks
// are dealt round-robin to blocks, and a grid barrier built on global atomics
// separates stages (trainkernel's generated kernel uses cooperative-groups
// grid.sync() between hazard stages: page "trainkernel 0.1.0 --
// trainkernel/codegen.py", `_CUDA_PREAMBLE` / `generate`).  Here the kernel is
// written once and interprets the table, so one binary serves every program.
//
// Numerics follow the same page: each op computes in float32 and rounds its
// result to its output dtype with round-to-nearest-even (`_round`); pointwise
// arithmetic uses one IEEE operation per step with no contraction (the page's
// runtime compiles with --fmad=false); GEMMs accumulate in float32.
//
// Every wait is bounded: a barrier that does not complete within the
// program's timeout records TK_ERR_BARRIER_TIMEOUT and the stage in the
// workspace header, raises an abort flag and returns; blocks that see the
// flag return too.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/tk.h"
#include "tk_device.h"

namespace tkk {
// Internal linkage: every kernel translation unit holds its own copy.
namespace {

using namespace tkd;

struct Prep;

// Descriptor pointers are indexed with global task/instruction/ref indices;
// for the current stage they usually point into shared memory.
struct Ctx {
  const Task* tasks;
  const Instr* code;
  const Ref* refs;
  char* ws;
  Header* hdr;
  void* const* io;  // shared-memory copy of Params::io
  long long timeout_ns;
  Prep* prep;       // shared memory: one prepared chain per warp
  int stage;        // stage being run (for failure reports)
  // bulk-streamed reductions (tensor-core launches): shared addresses of the
  // slots and of their mbarriers, the slot count (0: none) and the block's
  // running count of slots consumed, which fixes each slot's next phase
  uint32_t bulk, bulk_bar;
  int bulk_slots;
  uint32_t* bulk_it;
  uint32_t col_bar;   // column sums: the same slots, mbarriers counting every thread
  uint32_t* col_it;
};

// ------------------------------------------------------------------ memory

__device__ __forceinline__ char* space_ptr(const Ctx& c, int space, int slot) {
  if (space == SP_WS) return c.ws;
  return static_cast<char*>(c.io[space == SP_IN ? slot : kMaxIO + slot]);
}

__device__ __forceinline__ float round_to(float v, int dt) {
  if (dt == TK_BF16) return __bfloat162float(__float2bfloat16_rn(v));
  if (dt == TK_F16) return __half2float(__float2half_rn(v));
  return v;
}

__device__ __forceinline__ float load1(const char* p, int dt, int64_t i) {
  if (dt == TK_F32) return reinterpret_cast<const float*>(p)[i];
  if (dt == TK_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return __half2float(reinterpret_cast<const __half*>(p)[i]);
}

__device__ __forceinline__ void store1(char* p, int dt, int64_t i, float v) {
  if (dt == TK_F32)
    reinterpret_cast<float*>(p)[i] = v;
  else if (dt == TK_BF16)
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
}

// 8 bf16 or fp16 values packed in 16 bytes <-> floats.
__device__ __forceinline__ void unpack8(uint4 raw, int dt, float (&v)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (dt == TK_BF16) {
      __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[j]);
      v[2 * j] = __low2float(h);
      v[2 * j + 1] = __high2float(h);
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
      v[2 * j] = __low2float(h);
      v[2 * j + 1] = __high2float(h);
    }
  }
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8], int dt) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (dt == TK_BF16) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      w[j] = *reinterpret_cast<uint32_t*>(&h);
    } else {
      __half2 h = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
      w[j] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// 8 consecutive elements from a 16-byte aligned address.
__device__ __forceinline__ void load8(const char* p, int dt, int64_t i, float (&v)[8]) {
  if (dt == TK_F32) {
    const float4* q = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i);
    float4 x = q[0], y = q[1];
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
  } else {
    unpack8(*reinterpret_cast<const uint4*>(p + i * 2), dt, v);
  }
}

__device__ __forceinline__ void store8(char* p, int dt, int64_t i, const float (&v)[8]) {
  if (dt == TK_F32) {
    float4* q = reinterpret_cast<float4*>(reinterpret_cast<float*>(p) + i);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    *reinterpret_cast<uint4*>(p + i * 2) = pack8(v, dt);
  }
}

template <int V>
__device__ __forceinline__ void store_out(const Ctx& c, const Ref& o, int64_t flat, const float (&v)[V]) {
  char* p = space_ptr(c, o.space, o.slot);
  if constexpr (V == 8) {
    store8(p, o.dtype, o.base + flat, v);
  } else {
#pragma unroll
    for (int j = 0; j < V; ++j) store1(p, o.dtype, o.base + flat + j, v[j]);
  }
}

// ------------------------------------------------------ expression machine

// Index-space coordinates of flat index f (the planner keeps every index
// space below 2^31 elements, so 32-bit division suffices).
__device__ __forceinline__ void unravel(const Task& t, int64_t f, int64_t* crd) {
  uint32_t g = uint32_t(f);
#pragma unroll
  for (int d = kMaxRank - 1; d >= 0; --d) {
    if (d < t.rank) {
      const uint32_t n = uint32_t(t.shape[d]);
      const uint32_t q = g / n;
      crd[d] = int64_t(g - q * n);
      g = q;
    } else {
      crd[d] = 0;
    }
  }
}

template <int V>
__device__ __forceinline__ void load_ref(const Ctx& c, const Task& t, const Ref& r, const int64_t* crd,
                                         float (&out)[V]) {
  const char* p = space_ptr(c, r.space, r.slot);
  int64_t idx = r.base;
#pragma unroll
  for (int d = 0; d < kMaxRank; ++d) idx += crd[d] * r.stride[d];
  if constexpr (V == 8) {
    if (r.vmode == VM_CONTIG) {
      load8(p, r.dtype, idx, out);
    } else if (r.vmode == VM_BCAST) {
      float x = load1(p, r.dtype, idx);
#pragma unroll
      for (int j = 0; j < 8; ++j) out[j] = x;
    } else {
      int64_t s = t.rank ? r.stride[t.rank - 1] : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) out[j] = load1(p, r.dtype, idx + j * s);
    }
  } else {
    out[0] = load1(p, r.dtype, idx);
  }
}

template <int V>
struct Regs {
  float r[kVmRegs][V];

  __device__ __forceinline__ void get(int i, float (&out)[V]) const {
    switch (i) {
#define TK_GET(k)                                        \
  case k:                                                \
    _Pragma("unroll") for (int j = 0; j < V; ++j) out[j] = r[k][j]; \
    break;
      TK_GET(0) TK_GET(1) TK_GET(2) TK_GET(3)
#undef TK_GET
    }
  }
  __device__ __forceinline__ void set(int i, const float (&in)[V]) {
    switch (i) {
#define TK_SET(k)                                        \
  case k:                                                \
    _Pragma("unroll") for (int j = 0; j < V; ++j) r[k][j] = in[j]; \
    break;
      TK_SET(0) TK_SET(1) TK_SET(2) TK_SET(3)
#undef TK_SET
    }
  }
};

// Evaluate the task's expression for V consecutive elements whose first
// element has index-space coordinates crd; acc supplies OP_ACC values.
template <int V>
__device__ __forceinline__ void vm_eval(const Ctx& c, const Task& t, const int64_t* crd, const float* acc,
                                        float (&res)[V]) {
  Regs<V> R;
  const Instr* code = c.code + t.code_begin;
  const Ref* refs = c.refs + t.ref_begin;
  for (int pc = 0; pc < t.code_len; ++pc) {
    const Instr in = code[pc];
    float a[V], b[V], r[V];
    switch (in.op) {
      case OP_LOAD:
        load_ref<V>(c, t, refs[in.ref], crd, r);
        break;
      case OP_CONST:
#pragma unroll
        for (int j = 0; j < V; ++j) r[j] = in.imm;
        break;
      case OP_ACC:
#pragma unroll
        for (int j = 0; j < V; ++j) r[j] = acc[j];
        break;
      default:
        R.get(in.a, a);
        R.get(in.b, b);
        switch (in.op) {
          case OP_MOV:
#pragma unroll
            for (int j = 0; j < V; ++j) r[j] = a[j];
            break;
          case OP_ADD:
#pragma unroll
            for (int j = 0; j < V; ++j) r[j] = __fadd_rn(a[j], __fmul_rn(in.imm, b[j]));
            break;
          case OP_SUB:
#pragma unroll
            for (int j = 0; j < V; ++j) r[j] = __fsub_rn(a[j], __fmul_rn(in.imm, b[j]));
            break;
          case OP_MUL:
#pragma unroll
            for (int j = 0; j < V; ++j) r[j] = __fmul_rn(a[j], b[j]);
            break;
          case OP_DIV:
#pragma unroll
            for (int j = 0; j < V; ++j) r[j] = __fdiv_rn(a[j], b[j]);
            break;
          case OP_NEG:
#pragma unroll
            for (int j = 0; j < V; ++j) r[j] = -a[j];
            break;
          case OP_RELU:
#pragma unroll
            for (int j = 0; j < V; ++j) r[j] = a[j] < 0.0f ? 0.0f : a[j];
            break;
          case OP_SQUARE:
#pragma unroll
            for (int j = 0; j < V; ++j) r[j] = __fmul_rn(a[j], a[j]);
            break;
          case OP_POW:
#pragma unroll
            for (int j = 0; j < V; ++j) r[j] = powf(a[j], in.imm);
            break;
          case OP_THRESH:
#pragma unroll
            for (int j = 0; j < V; ++j) r[j] = b[j] <= in.imm ? 0.0f : a[j];
            break;
          default:
#pragma unroll
            for (int j = 0; j < V; ++j) r[j] = 0.0f;
            break;
        }
    }
    if (in.round != TK_F32) {
#pragma unroll
      for (int j = 0; j < V; ++j) r[j] = round_to(r[j], in.round);
    }
    R.set(in.dst, r);
  }
  R.get(0, res);
}

// ------------------------------------------------------------- chains

template <int V>
__device__ __forceinline__ void chain_load(const Ctx& c, const Task& t, const int64_t* crd, float (&L)[2][V]) {
  const Chain& ch = t.chain;
  const Ref* refs = c.refs + t.ref_begin;
  if (ch.n_loads > 0) load_ref<V>(c, t, refs[ch.load_ref[0]], crd, L[0]);
  if (ch.n_loads > 1) load_ref<V>(c, t, refs[ch.load_ref[1]], crd, L[1]);
}

// A chain with its operands resolved to byte pointers and 32-bit byte strides,
// prepared once per work item into the warp's slot in shared memory: the hot
// loops read it with shared-memory loads instead of holding ~60 values in
// registers (which spilled to local memory, i.e. to L2 behind a small L1).  (Index spaces are below 2^31 elements and the planner
// keeps chain operand strides below 2^31 bytes.)
struct PLoad {
  const char* p;            // operand element (0,...,0)
  int32_t sb[kMaxRank];     // byte stride per index dim
  int32_t dtype, vmode, inner_b;
};

struct Prep {
  Chain ch;
  PLoad ld[2];
  char* out;                // output element 0
  int32_t out_dtype;
};

__device__ __forceinline__ int esize_of(int dt) { return dt == TK_F32 ? 4 : 2; }

__device__ __forceinline__ void prepare(const Ctx& c, const Task& t, Prep& P) {
  P.ch = t.chain;
  const Ref* refs = c.refs + t.ref_begin;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (i < P.ch.n_loads) {
      const Ref& r = refs[P.ch.load_ref[i]];
      const int es = esize_of(r.dtype);
      P.ld[i].p = space_ptr(c, r.space, r.slot) + r.base * es;
#pragma unroll
      for (int d = 0; d < kMaxRank; ++d) P.ld[i].sb[d] = int32_t(r.stride[d] * es);
      P.ld[i].dtype = r.dtype;
      P.ld[i].vmode = r.vmode;
      P.ld[i].inner_b = t.rank ? int32_t(r.stride[t.rank - 1] * es) : 0;
    }
  }
  P.out = space_ptr(c, t.out.space, t.out.slot) + t.out.base * esize_of(t.out.dtype);
  P.out_dtype = t.out.dtype;
}

__device__ __forceinline__ float ld1b(const char* a, int dt) {
  if (dt == TK_F32) return *reinterpret_cast<const float*>(a);
  if (dt == TK_BF16) return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(a));
  return __half2float(*reinterpret_cast<const __half*>(a));
}

template <int V>
__device__ __forceinline__ void pload(const PLoad& l, const int32_t* crd, float (&out)[V]) {
  int64_t off = 0;
#pragma unroll
  for (int d = 0; d < kMaxRank; ++d) off += int64_t(crd[d]) * l.sb[d];
  const char* a = l.p + off;
  if constexpr (V == 8) {
    if (l.vmode == VM_CONTIG) {
      load8(a, l.dtype, 0, out);
    } else if (l.vmode == VM_BCAST) {
      const float x = ld1b(a, l.dtype);
#pragma unroll
      for (int j = 0; j < 8; ++j) out[j] = x;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) out[j] = ld1b(a + j * l.inner_b, l.dtype);
    }
  } else {
    out[0] = ld1b(a, l.dtype);
  }
}

template <int V>
__device__ __forceinline__ void prep_load(const Prep& P, const int32_t* crd, float (&L)[2][V]) {
  if (P.ch.n_loads > 0) pload<V>(P.ld[0], crd, L[0]);
  if (P.ch.n_loads > 1) pload<V>(P.ld[1], crd, L[1]);
}

template <int V>
__device__ __forceinline__ void prep_store(const Prep& P, int64_t flat, const float (&v)[V]) {
  if constexpr (V == 8) {
    store8(P.out, P.out_dtype, flat, v);
  } else {
#pragma unroll
    for (int j = 0; j < V; ++j) store1(P.out, P.out_dtype, flat + j, v[j]);
  }
}

// 32-bit index-space coordinates of flat index f.
__device__ __forceinline__ void unravel32(const Task& t, uint32_t f, int32_t* crd) {
#pragma unroll
  for (int d = kMaxRank - 1; d >= 0; --d) {
    if (d < t.rank) {
      const uint32_t n = uint32_t(t.shape[d]);
      const uint32_t q = f / n;
      crd[d] = int32_t(f - q * n);
      f = q;
    } else {
      crd[d] = 0;
    }
  }
}

template <int V>
__device__ __forceinline__ void round_vec(float (&x)[V], int dt) {
  // pairs go through the packed conversions (each element rounded on its own)
  if (dt == TK_BF16) {
#pragma unroll
    for (int j = 0; j + 1 < V; j += 2) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[j], x[j + 1]);
      x[j] = __low2float(h);
      x[j + 1] = __high2float(h);
    }
    if (V & 1) x[V - 1] = __bfloat162float(__float2bfloat16_rn(x[V - 1]));
  } else if (dt == TK_F16) {
#pragma unroll
    for (int j = 0; j + 1 < V; j += 2) {
      const __half2 h = __floats2half2_rn(x[j], x[j + 1]);
      x[j] = __low2float(h);
      x[j + 1] = __high2float(h);
    }
    if (V & 1) x[V - 1] = __half2float(__float2half_rn(x[V - 1]));
  }
}

// The chain's value for V elements from their loaded operands (and the GEMM
// accumulator for CH_ACC): same arithmetic, operation by operation, as the
// instruction form.  Every branch is uniform across the block.
template <int V>
__device__ __forceinline__ void chain_compute(const Chain& ch, const float (&L)[2][V], const float* acc, float (&x)[V]) {
  if (ch.start == CH_LOAD) {
#pragma unroll
    for (int j = 0; j < V; ++j) x[j] = L[0][j];
  } else if (ch.start == CH_CONST) {
#pragma unroll
    for (int j = 0; j < V; ++j) x[j] = ch.start_const;
  } else {
    float b[V];
    if (ch.bias == 0) {
#pragma unroll
      for (int j = 0; j < V; ++j) b[j] = L[0][j];
    } else if (ch.bias == 1) {
#pragma unroll
      for (int j = 0; j < V; ++j) b[j] = L[1][j];
    } else {
#pragma unroll
      for (int j = 0; j < V; ++j) b[j] = ch.bias_const;
    }
    switch (ch.addmm_mode) {
      case AM_ACC:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = acc[j];
        break;
      case AM_SUM:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = __fadd_rn(acc[j], b[j]);
        break;
      case AM_ZERO:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = 0.0f;
        break;
      case AM_ALPHA:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = __fmul_rn(ch.alpha, acc[j]);
        break;
      case AM_BETA:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = __fmul_rn(ch.beta, b[j]);
        break;
      default:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = __fadd_rn(__fmul_rn(ch.alpha, acc[j]), __fmul_rn(ch.beta, b[j]));
        break;
    }
    round_vec<V>(x, ch.round0);
  }
#pragma unroll
  for (int s = 0; s < kChainSteps; ++s) {
    if (s >= ch.n_steps) break;
    const ChainStep st = ch.steps[s];
    float e[V];
    if (st.ext == EXT_LOAD0) {
#pragma unroll
      for (int j = 0; j < V; ++j) e[j] = L[0][j];
    } else if (st.ext == EXT_LOAD1) {
#pragma unroll
      for (int j = 0; j < V; ++j) e[j] = L[1][j];
    } else {
#pragma unroll
      for (int j = 0; j < V; ++j) e[j] = st.cval;
    }
    if (st.ext_mul) {  // an inlined c * input
#pragma unroll
      for (int j = 0; j < V; ++j) e[j] = __fmul_rn(e[j], st.cval);
      round_vec<V>(e, st.ext_round);
    }
    if (st.second) {  // running value is the second operand: swap roles
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const float tmp = e[j];
        e[j] = x[j];
        x[j] = tmp;
      }
    }
    // now x holds operand a, e holds operand b
    switch (st.op) {
      case OP_ADD:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = __fadd_rn(x[j], __fmul_rn(st.imm, e[j]));
        break;
      case OP_SUB:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = __fsub_rn(x[j], __fmul_rn(st.imm, e[j]));
        break;
      case OP_MUL:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = __fmul_rn(x[j], e[j]);
        break;
      case OP_DIV:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = __fdiv_rn(x[j], e[j]);
        break;
      case OP_NEG:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = -x[j];
        break;
      case OP_RELU:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = x[j] < 0.0f ? 0.0f : x[j];
        break;
      case OP_SQUARE:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = __fmul_rn(x[j], x[j]);
        break;
      case OP_THRESH:
#pragma unroll
        for (int j = 0; j < V; ++j) x[j] = e[j] <= st.imm ? 0.0f : x[j];
        break;
      default:
        break;
    }
    round_vec<V>(x, st.round);
  }
}

// A side output: one op on the stored (rounded) final value x, the same
// arithmetic as the chain step it stands for: x*c, -x, a cast, or (a loaded
// side) x +/- a*e / e +/- a*x with e the side operand.
__device__ __forceinline__ float side_value(const ChainStep& st, float x, float e) {
  float y;
  if (st.op == OP_ADD || st.op == OP_SUB) {
    const float a = st.second ? e : x, b = st.second ? x : e;
    const float p = __fmul_rn(st.imm, b);
    y = st.op == OP_ADD ? __fadd_rn(a, p) : __fsub_rn(a, p);
  } else {
    y = st.op == OP_MUL ? __fmul_rn(x, st.cval) : st.op == OP_NEG ? -x : x;
  }
  return round_to(y, st.round);
}

// Out of line, so that the epilogues without a side output carry no code for it.
template <int V>
__device__ __noinline__ void store_side(const Ctx c, const Task& t, int64_t flat, const float (&x)[V]) {
  float e[V], y[V];
  if (t.side.ext == EXT_LOAD1) {
    const char* p = space_ptr(c, t.side_ld.space, t.side_ld.slot);
    if constexpr (V == 8) {
      load8(p, t.side_ld.dtype, t.side_ld.base + flat, e);
    } else {
#pragma unroll
      for (int j = 0; j < V; ++j) e[j] = load1(p, t.side_ld.dtype, t.side_ld.base + flat + j);
    }
  } else {
#pragma unroll
    for (int j = 0; j < V; ++j) e[j] = 0.0f;
  }
#pragma unroll 1
  for (int j = 0; j < V; ++j) y[j] = side_value(t.side, x[j], e[j]);
  store_out<V>(c, t.out2, flat, y);
}

// ------------------------------------------------- compiled chain shapes
//
// Parameters of a FastKind chain, read once per work item into registers.
struct Fast {
  const char* p0;
  const char* p1;
  int32_t rs0, rs1;   // byte stride per index-space row (GEMM epilogues)
  int32_t dt0, dt1;   // operand dtypes
  int32_t r0, r1, r2; // rounding: start value, step 0, step 1
  float a0, a1, c0;   // step 0 / step 1 alpha or threshold; step 0 constant
  int32_t sub0, sub1; // the add/sub step subtracts
  int32_t er;         // rounding of a scaled operand (momentum)
  char* out;
  int32_t out_dt;
};

__device__ __forceinline__ Fast fast_params(const Ctx& c, const Task& t) {
  const Chain& ch = t.chain;
  const Ref* refs = c.refs + t.ref_begin;
  Fast F;
  F.p0 = F.p1 = nullptr;
  F.rs0 = F.rs1 = 0;
  F.dt0 = F.dt1 = TK_F32;
  if (ch.n_loads > 0) {
    const Ref& r = refs[ch.load_ref[0]];
    const int es = esize_of(r.dtype);
    F.p0 = space_ptr(c, r.space, r.slot) + r.base * es;
    F.rs0 = int32_t(r.stride[0] * es);
    F.dt0 = r.dtype;
  }
  if (ch.n_loads > 1) {
    const Ref& r = refs[ch.load_ref[1]];
    const int es = esize_of(r.dtype);
    F.p1 = space_ptr(c, r.space, r.slot) + r.base * es;
    F.rs1 = int32_t(r.stride[0] * es);
    F.dt1 = r.dtype;
  }
  F.r0 = ch.round0;
  F.r1 = ch.steps[0].round;
  F.r2 = ch.steps[1].round;
  F.a0 = ch.steps[0].imm;
  F.a1 = ch.steps[1].imm;
  F.c0 = ch.steps[0].cval;
  F.sub0 = ch.steps[0].op == OP_SUB;
  F.sub1 = ch.steps[1].op == OP_SUB;
  F.er = ch.steps[0].ext_round;
  F.out = space_ptr(c, t.out.space, t.out.slot) + t.out.base * esize_of(t.out.dtype);
  F.out_dt = t.out.dtype;
  return F;
}

template <int K>
struct FastTraits {
  static constexpr bool load0 = K != FK_E_ACC;
  static constexpr bool load1 = K == FK_E_BIAS_AXPY || K == FK_L_AXPY || K == FK_L_SCALE_AXPY;
};

// The same operations, in the same order and with the same roundings, as the
// chain the kind stands for.
// kLast = false leaves out the final rounding, for a caller that converts the
// result to the same 16-bit type right away (rounding twice to one format
// equals rounding once).
template <int K, bool kLast = true>
__device__ __forceinline__ void fast_apply(const Fast& F, const float (&l0)[8], const float (&l1)[8],
                                           const float (&acc)[8], float (&x)[8]) {
  if constexpr (K == FK_E_MOMENTUM) {
    // v' = round(round(v * mu) + a * round(acc))
    float m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      x[j] = acc[j];
      m[j] = __fmul_rn(l0[j], F.c0);
    }
    round_vec<8>(x, F.r0);
    round_vec<8>(m, F.er);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = __fadd_rn(m[j], __fmul_rn(F.a0, x[j]));
    if constexpr (kLast) round_vec<8>(x, F.r1);
  } else if constexpr (K == FK_E_UPDATE) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = acc[j];
    round_vec<8>(x, F.r0);
    if (F.sub0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = __fsub_rn(l0[j], __fmul_rn(F.a0, x[j]));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = __fadd_rn(l0[j], __fmul_rn(F.a0, x[j]));
    }
    if constexpr (kLast) round_vec<8>(x, F.r1);
  } else if constexpr (K >= FK_E_ACC && K <= FK_E_ACC_THRESH) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = (K == FK_E_ACC || K == FK_E_ACC_THRESH) ? acc[j] : __fadd_rn(acc[j], l0[j]);
    if (kLast || !(K == FK_E_ACC || K == FK_E_BIAS)) round_vec<8>(x, F.r0);  // r0 is the last rounding of these two
    if constexpr (K == FK_E_BIAS_RELU) {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = x[j] < 0.0f ? 0.0f : x[j];
      if constexpr (kLast) round_vec<8>(x, F.r1);
    } else if constexpr (K == FK_E_BIAS_AXPY) {
      if (F.sub0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = __fsub_rn(x[j], __fmul_rn(F.a0, l1[j]));
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = __fadd_rn(x[j], __fmul_rn(F.a0, l1[j]));
      }
      if constexpr (kLast) round_vec<8>(x, F.r1);
    } else if constexpr (K == FK_E_ACC_THRESH) {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = l0[j] <= F.a0 ? 0.0f : x[j];
      if constexpr (kLast) round_vec<8>(x, F.r1);
    }
  } else if constexpr (K == FK_L) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = l0[j];
  } else if constexpr (K == FK_L_MOV) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = l0[j];
    round_vec<8>(x, F.r1);
  } else if constexpr (K == FK_L_SQUARE) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = __fmul_rn(l0[j], l0[j]);
    round_vec<8>(x, F.r1);
  } else if constexpr (K == FK_L_SCALE || K == FK_L_SCALE_AXPY) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = __fmul_rn(l0[j], F.c0);
    round_vec<8>(x, F.r1);
    if constexpr (K == FK_L_SCALE_AXPY) {
      if (F.sub1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = __fsub_rn(x[j], __fmul_rn(F.a1, l1[j]));
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = __fadd_rn(x[j], __fmul_rn(F.a1, l1[j]));
      }
      round_vec<8>(x, F.r2);
    }
  } else if constexpr (K == FK_L_AXPY) {
    if (F.sub0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = __fsub_rn(l0[j], __fmul_rn(F.a0, l1[j]));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = __fadd_rn(l0[j], __fmul_rn(F.a0, l1[j]));
    }
    round_vec<8>(x, F.r1);
  }
}

// Dispatch a FastKind to a template taking the kind as its parameter.
#define TK_FAST_L_CASES(CALL)                 \
  case FK_L: CALL(FK_L); break;               \
  case FK_L_MOV: CALL(FK_L_MOV); break;       \
  case FK_L_SQUARE: CALL(FK_L_SQUARE); break; \
  case FK_L_SCALE: CALL(FK_L_SCALE); break;   \
  case FK_L_AXPY: CALL(FK_L_AXPY); break;     \
  case FK_L_SCALE_AXPY: CALL(FK_L_SCALE_AXPY); break;

// One vector of a task's expression, whichever form the planner chose.
template <int V>
__device__ __forceinline__ void eval_expr(const Ctx& c, const Task& t, const int64_t* crd, const float* acc,
                                          float (&out)[V]) {
  if (t.chain.valid) {
    float L[2][V];
    chain_load<V>(c, t, crd, L);
    chain_compute<V>(t.chain, L, acc, out);
  } else {
    vm_eval<V>(c, t, crd, acc, out);
  }
}

// ------------------------------------------------------------- barriers

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ void record_failure(const Ctx& c, int status, int stage) {
  if (atomicCAS(&c.hdr->status, 0, status) == 0) atomicExch(&c.hdr->stage, stage);
  atomicExch(&c.hdr->abort, 1);
}

// Grid barrier, in two halves so the block can stage the next stage's
// descriptors while thread 0 waits.  Barrier j of a run completes when the
// arrival counter reaches (j + 1) * gridDim.x: arriving is one fire-and-forget
// release reduction, waiting is a relaxed poll followed by one acquire fence.
// Thread 0 only.
__device__ __forceinline__ void barrier_arrive(const Ctx& c) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&c.hdr->count) : "memory");
}

__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Thread 0 only; false when the wait timed out or another block gave up.
__device__ __forceinline__ bool barrier_wait(const Ctx& c, unsigned target, int stage) {
  Header* h = c.hdr;
  unsigned spins = 0;
  long long t0 = 0;
  while (int(ld_relaxed(&h->count) - target) < 0) {
    if ((++spins & 31u) == 0u) {
      if (*reinterpret_cast<volatile int*>(&h->abort)) return false;
      const long long now = global_ns();
      if (t0 == 0) t0 = now;
      if (now - t0 > c.timeout_ns) {
        record_failure(c, TK_ERR_BARRIER_TIMEOUT, stage);
        return false;
      }
    }
  }
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  return true;
}

// Last block out resets the counters for the next run (also the folded
// finals' part counts, which a run that gave up may have left behind).
// Thread 0 only.
__device__ __forceinline__ void kernel_exit(const Ctx& c) {
  Header* h = c.hdr;
  if (atom_add_acq_rel(&h->exits, 1u) + 1u == gridDim.x) {
    for (int i = 0; i < kFoldCounters; ++i) h->fold[i] = 0u;
    atomicExch(&h->count, 0u);
    atomicExch(&h->exits, 0u);
  }
}

// ------------------------------------------------------------ block sums

// Deterministic block-wide sum; the result is valid in thread 0.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.0f;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];
  }
  __syncthreads();
  return s;
}

// A reduction's epilogue chain at output o (coordinates over post_shape).
__device__ __noinline__ float reduction_post(const Ctx c, const Task& t, int64_t o, float v) {
  int64_t crd[kMaxRank];
  int64_t f = o;
#pragma unroll
  for (int d = kMaxRank - 1; d >= 0; --d) {
    if (d < t.post_rank) {
      crd[d] = f % t.post_shape[d];
      f /= t.post_shape[d];
    } else {
      crd[d] = 0;
    }
  }
  const Ref* refs = c.refs + t.ref_begin;
  float L[2][1] = {{0.0f}, {0.0f}};
  if (t.post.n_loads > 0) load_ref<1>(c, t, refs[t.post.load_ref[0]], crd, L[0]);
  if (t.post.n_loads > 1) load_ref<1>(c, t, refs[t.post.load_ref[1]], crd, L[1]);
  const float a[1] = {v};
  float x[1];
  chain_compute<1>(t.post, L, a, x);
  return x[0];
}

// The operand of a compiled reduction epilogue (the parameter being updated)
// at output o, loaded before the reduction so its latency overlaps the sums.
__device__ __forceinline__ float post_operand(const Ctx& c, const Task& t, int64_t o) {
  if (t.post.fast != FK_E_UPDATE) return 0.0f;
  const Ref& r = c.refs[t.ref_begin + t.post.load_ref[0]];
  return load1(space_ptr(c, r.space, r.slot), r.dtype, r.base + o);
}

__device__ __forceinline__ void finish_reduction(const Ctx& c, const Task& t, int64_t o, float acc, float pre) {
  float v = t.red_mean ? __fdiv_rn(acc, t.size_f) : acc;
  if (t.post.fast == FK_E_UPDATE) {  // p -/+ a * round(v)
    const ChainStep st = t.post.steps[0];
    const float r = round_to(v, t.post.round0);
    v = round_to(st.op == OP_SUB ? __fsub_rn(pre, __fmul_rn(st.imm, r)) : __fadd_rn(pre, __fmul_rn(st.imm, r)), st.round);
  } else if (t.post.valid) {
    v = reduction_post(c, t, o, v);
  }
  store1(space_ptr(c, t.out.space, t.out.slot), t.out.dtype, t.out.base + o, v);
  if (t.has_side) {
    const float x[1] = {round_to(v, t.out.dtype)};  // the stored value
    store_side<1>(c, t, o, x);
  }
}

// ------------------------------------------------------------- work items

// Elements per pointwise work item: kThreads threads x V elements x U vectors.
template <int V>
__device__ __forceinline__ constexpr int pointwise_unroll() { return V == 8 ? kPointwiseUnroll : 1; }

// Vectors u = 0..U-1 of the item, software-pipelined: the loads of vector
// u+1 are in flight while vector u is computed and stored.
template <int V>
__device__ __noinline__ void pointwise_chain(const Ctx c, const Task& t, int item) {
  constexpr int U = pointwise_unroll<V>();
  const int64_t base = int64_t(item) * kThreads * V * U + int64_t(threadIdx.x) * V;
  constexpr int64_t step = int64_t(kThreads) * V;
  const int64_t numel = t.numel;
  if (base >= numel) return;
  Prep& P = c.prep[threadIdx.x >> 5];
  prepare(c, t, P);
  float cur[2][V], nxt[2][V];
  int32_t crd[kMaxRank];
  unravel32(t, uint32_t(base), crd);
  prep_load<V>(P, crd, cur);
#pragma unroll 1
  for (int u = 0; u < U; ++u) {
    const int64_t i0 = base + u * step;
    const bool more = u + 1 < U && i0 + step < numel;
    if (more) {
      unravel32(t, uint32_t(i0 + step), crd);
      prep_load<V>(P, crd, nxt);
    }
    float v[V];
    chain_compute<V>(P.ch, cur, nullptr, v);
    prep_store<V>(P, i0, v);
    if (!more) break;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      cur[0][j] = nxt[0][j];
      cur[1][j] = nxt[1][j];
    }
  }
}

template <int V>
__device__ __noinline__ void pointwise_vm(const Ctx c, const Task& t, int item) {
  constexpr int U = pointwise_unroll<V>();
  const int64_t base = int64_t(item) * kThreads * V * U;
  for (int u = 0; u < U; ++u) {
    const int64_t i0 = base + (int64_t(u) * kThreads + threadIdx.x) * V;
    if (i0 >= t.numel) return;
    int64_t crd[kMaxRank];
    unravel(t, i0, crd);
    float v[V];
    vm_eval<V>(c, t, crd, nullptr, v);
    store_out<V>(c, t.out, i0, v);
  }
}

// A FastKind pointwise item: operands and output at the flat index, all U
// vectors' loads issued before the first store.
// Operands and output all 16-bit: raw 16-byte vectors, twice as many in flight.
template <int K>
__device__ __noinline__ void pointwise_fast16(const Ctx c, const Task& t, int item) {
  constexpr int U = kPointwiseUnroll16;
  constexpr int64_t step = int64_t(kThreads) * 8;
  const int64_t base = int64_t(item) * kThreads * 8 * U + int64_t(threadIdx.x) * 8;
  const int64_t numel = t.numel;
  const Fast F = fast_params(c, t);
  uint4 q0[U], q1[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t i = base + u * step;
    if (i < numel) {
      q0[u] = *reinterpret_cast<const uint4*>(F.p0 + i * 2);
      if constexpr (FastTraits<K>::load1) q1[u] = *reinterpret_cast<const uint4*>(F.p1 + i * 2);
    }
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t i = base + u * step;
    if (i < numel) {
      float l0[8], l1[8], none[8], x[8];
      unpack8(q0[u], F.dt0, l0);
      if constexpr (FastTraits<K>::load1) unpack8(q1[u], F.dt1, l1);
      fast_apply<K>(F, l0, l1, none, x);
      *reinterpret_cast<uint4*>(F.out + i * 2) = pack8(x, F.out_dt);
    }
  }
}

template <int K>
__device__ __noinline__ void pointwise_fast(const Ctx c, const Task& t, int item) {
  constexpr int U = kPointwiseUnroll;
  constexpr int64_t step = int64_t(kThreads) * 8;
  const int64_t base = int64_t(item) * kThreads * 8 * U + int64_t(threadIdx.x) * 8;
  const int64_t numel = t.numel;
  const Fast F = fast_params(c, t);
  float l0[U][8], l1[U][8], none[8];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t i = base + u * step;
    if (i < numel) {
      load8(F.p0, F.dt0, i, l0[u]);
      if constexpr (FastTraits<K>::load1) load8(F.p1, F.dt1, i, l1[u]);
    }
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t i = base + u * step;
    if (i < numel) {
      float x[8];
      fast_apply<K>(F, l0[u], l1[u], none, x);
      store8(F.out, F.out_dt, i, x);
    }
  }
}

template <int V>
__device__ __forceinline__ void run_pointwise(const Ctx& c, const Task& t, int item) {
  if constexpr (V == 8) {
    if (t.pw_unroll == kPointwiseUnroll16) {
#define TK_CALL(k) pointwise_fast16<k>(c, t, item)
      switch (t.chain.fast) {
        TK_FAST_L_CASES(TK_CALL)
        default: break;
      }
#undef TK_CALL
    } else {
#define TK_CALL(k) pointwise_fast<k>(c, t, item)
      switch (t.chain.fast) {
        TK_FAST_L_CASES(TK_CALL)
        default: break;
      }
#undef TK_CALL
    }
    if (t.chain.fast != FK_NONE) return;
  }
  if (t.chain.valid)
    pointwise_chain<V>(c, t, item);
  else
    pointwise_vm<V>(c, t, item);
}

// This thread's share of one output row of a row reduction, in element order.
template <int V>
__device__ __noinline__ float row_sum_chain(const Ctx c, const Task& t, int64_t o, int64_t r0, int64_t r1) {
  constexpr int64_t step = int64_t(kThreads) * V;
  Prep& P = c.prep[threadIdx.x >> 5];
  prepare(c, t, P);
  const int64_t row0 = o * t.red_inner;
  float acc = 0.0f;
  for (int64_t r = r0 + int64_t(threadIdx.x) * V; r < r1; r += 2 * step) {
    // two vectors in flight: the second one's loads overlap the first
    const bool second = r + step < r1;
    float L0[2][V], L1[2][V], v[V];
    int32_t crd[kMaxRank];
    unravel32(t, uint32_t(row0 + r), crd);
    prep_load<V>(P, crd, L0);
    if (second) {
      unravel32(t, uint32_t(row0 + r + step), crd);
      prep_load<V>(P, crd, L1);
    }
    chain_compute<V>(P.ch, L0, nullptr, v);
#pragma unroll
    for (int j = 0; j < V; ++j) acc = __fadd_rn(acc, v[j]);
    if (second) {
      chain_compute<V>(P.ch, L1, nullptr, v);
#pragma unroll
      for (int j = 0; j < V; ++j) acc = __fadd_rn(acc, v[j]);
    }
  }
  return acc;
}

// row_sum_chain for a FastKind chain over flat-addressed operands.
template <int K>
__device__ __noinline__ float row_sum_fast(const Ctx c, const Task& t, int64_t o, int64_t r0, int64_t r1) {
  constexpr int64_t step = int64_t(kThreads) * 8;
  const Fast F = fast_params(c, t);
  const int64_t row0 = o * t.red_inner;
  float acc = 0.0f, none[8];
  for (int64_t r = r0 + int64_t(threadIdx.x) * 8; r < r1; r += 2 * step) {
    const bool second = r + step < r1;
    float a0[8], a1[8], b0[8], b1[8], x[8];
    load8(F.p0, F.dt0, row0 + r, a0);
    if constexpr (FastTraits<K>::load1) load8(F.p1, F.dt1, row0 + r, a1);
    if (second) {
      load8(F.p0, F.dt0, row0 + r + step, b0);
      if constexpr (FastTraits<K>::load1) load8(F.p1, F.dt1, row0 + r + step, b1);
    }
    fast_apply<K>(F, a0, a1, none, x);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc = __fadd_rn(acc, x[j]);
    if (second) {
      fast_apply<K>(F, b0, b1, none, x);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc = __fadd_rn(acc, x[j]);
    }
  }
  return acc;
}

template <int K>
__device__ __noinline__ float row_sum_bulk16(const Ctx c, const Task& t, int64_t o, int64_t r0, int64_t r1);
template <int K>
__device__ __noinline__ void run_reduce_col_bulk16(const Ctx c, const Task& t, int item, float* red);

// The same over 16-bit operands, streaming: eight raw 16-byte vectors per
// thread in flight (a reduction over a tensor much larger than one block's
// share must keep enough loads in flight to cover the memory latency).
template <int K>
__device__ __noinline__ float row_sum_fast16(const Ctx c, const Task& t, int64_t o, int64_t r0, int64_t r1) {
  constexpr int W = 8;
  constexpr int64_t step = int64_t(kThreads) * 8;
  const Fast F = fast_params(c, t);
  const char* p0 = F.p0 + o * t.red_inner * 2;
  const char* p1 = FastTraits<K>::load1 ? F.p1 + o * t.red_inner * 2 : nullptr;
  float acc = 0.0f, none[8];
  for (int64_t r = r0 + int64_t(threadIdx.x) * 8; r < r1; r += W * step) {
    uint4 q0[W], q1[W];
#pragma unroll
    for (int w = 0; w < W; ++w) {
      if (r + w * step < r1) {
        q0[w] = *reinterpret_cast<const uint4*>(p0 + (r + w * step) * 2);
        if constexpr (FastTraits<K>::load1) q1[w] = *reinterpret_cast<const uint4*>(p1 + (r + w * step) * 2);
      }
    }
#pragma unroll
    for (int w = 0; w < W; ++w) {
      if (r + w * step < r1) {
        float a[8], b[8], x[8];
        unpack8(q0[w], F.dt0, a);
        if constexpr (FastTraits<K>::load1) unpack8(q1[w], F.dt1, b);
        fast_apply<K>(F, a, b, none, x);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc = __fadd_rn(acc, x[j]);
      }
    }
  }
  return acc;
}

template <int V>
__device__ __noinline__ float row_sum_vm(const Ctx c, const Task& t, int64_t o, int64_t r0, int64_t r1) {
  float acc = 0.0f;
  for (int64_t r = r0 + int64_t(threadIdx.x) * V; r < r1; r += int64_t(kThreads) * V) {
    int64_t crd[kMaxRank];
    unravel(t, o * t.red_inner + r, crd);
    float v[V];
    vm_eval<V>(c, t, crd, nullptr, v);
#pragma unroll
    for (int j = 0; j < V; ++j) acc = __fadd_rn(acc, v[j]);
  }
  return acc;
}

template <int V>
__device__ __noinline__ void run_reduce_row(const Ctx c, const Task& t, int item, float* red) {
  const int64_t o = item / t.parts;
  const int p = item % t.parts;
  const int64_t r0 = int64_t(p) * t.part_len;
  const int64_t r1 = min(t.red_inner, r0 + t.part_len);
  const float pre = threadIdx.x == 0 && t.parts == 1 ? post_operand(c, t, o) : 0.0f;
  float acc;
  bool done = false;
  if constexpr (V == 8) {
    done = true;
    if (t.pw_unroll == kPointwiseUnroll16) {
#define TK_CALL(k) acc = row_sum_bulk16<k>(c, t, o, r0, r1)
      switch (t.chain.fast) {
        TK_FAST_L_CASES(TK_CALL)
        default: done = false; break;
      }
#undef TK_CALL
    } else {
#define TK_CALL(k) acc = row_sum_fast<k>(c, t, o, r0, r1)
      switch (t.chain.fast) {
        TK_FAST_L_CASES(TK_CALL)
        default: done = false; break;
      }
#undef TK_CALL
    }
  }
  if (!done) acc = t.chain.valid ? row_sum_chain<V>(c, t, o, r0, r1) : row_sum_vm<V>(c, t, o, r0, r1);
  acc = block_sum(acc, red);
  if (threadIdx.x == 0) {
    if (t.parts == 1)
      finish_reduction(c, t, o, acc, pre);
    else
      reinterpret_cast<float*>(c.ws)[t.scratch + o * t.parts + p] = acc;
  }
}

// Column reductions: warp w sums rows r0+w, r0+w+8, ... of 8*32 columns
// (lane l: columns 8l..8l+7), then the 8 warps' partial sums are added in warp
// order.
template <int V>
__device__ __forceinline__ void col_combine(const Ctx& c, const Task& t, int64_t ch, int p, const float (&acc)[V],
                                            float* red, float pre) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t Q = t.red_inner;
#pragma unroll
  for (int j = 0; j < V; ++j) red[warp * 32 * V + lane * V + j] = acc[j];
  __syncthreads();
  if (threadIdx.x < 32 * V) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) s = __fadd_rn(s, red[w * 32 * V + threadIdx.x]);
    const int64_t col = ch * 32 * V + threadIdx.x;
    if (col < Q) {
      if (t.parts == 1)
        finish_reduction(c, t, col, s, pre);
      else
        reinterpret_cast<float*>(c.ws)[t.scratch + col * t.parts + p] = s;
    }
  }
  __syncthreads();
}

template <int K>
__device__ __noinline__ void run_reduce_col_fast(const Ctx c, const Task& t, int item, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int64_t rstep = kThreads / 32;
  const int64_t ch = item / t.parts;
  const int p = item % t.parts;
  const int64_t Q = t.red_inner;
  const int64_t col0 = ch * 256 + lane * 8;
  const int64_t r0 = int64_t(p) * t.part_len;
  const int64_t r1 = min(t.red_outer, r0 + t.part_len);
  const int64_t my_col = ch * 256 + threadIdx.x;
  const float pre = t.parts == 1 && my_col < Q ? post_operand(c, t, my_col) : 0.0f;
  const Fast F = fast_params(c, t);
  float acc[8], none[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
  if (col0 < Q) {
    for (int64_t r = r0 + warp; r < r1; r += 2 * rstep) {
      const bool second = r + rstep < r1;
      float a0[8], a1[8], b0[8], b1[8], x[8];
      load8(F.p0, F.dt0, r * Q + col0, a0);
      if constexpr (FastTraits<K>::load1) load8(F.p1, F.dt1, r * Q + col0, a1);
      if (second) {
        load8(F.p0, F.dt0, (r + rstep) * Q + col0, b0);
        if constexpr (FastTraits<K>::load1) load8(F.p1, F.dt1, (r + rstep) * Q + col0, b1);
      }
      fast_apply<K>(F, a0, a1, none, x);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], x[j]);
      if (second) {
        fast_apply<K>(F, b0, b1, none, x);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], x[j]);
      }
    }
  }
  col_combine<8>(c, t, ch, p, acc, red, pre);
}

// Column sums over 16-bit operands, streaming: each warp keeps eight rows'
// 16-byte vectors in flight.
template <int K>
__device__ __noinline__ void run_reduce_col_fast16(const Ctx c, const Task& t, int item, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int W = 8;
  constexpr int64_t rstep = kThreads / 32;
  const int64_t ch = item / t.parts;
  const int p = item % t.parts;
  const int64_t Q = t.red_inner;
  const int64_t col0 = ch * 256 + lane * 8;
  const int64_t r0 = int64_t(p) * t.part_len;
  const int64_t r1 = min(t.red_outer, r0 + t.part_len);
  const int64_t my_col = ch * 256 + threadIdx.x;
  const float pre = t.parts == 1 && my_col < Q ? post_operand(c, t, my_col) : 0.0f;
  const Fast F = fast_params(c, t);
  float acc[8], none[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
  if (col0 < Q) {
    for (int64_t r = r0 + warp; r < r1; r += W * rstep) {
      uint4 q0[W], q1[W];
#pragma unroll
      for (int w = 0; w < W; ++w) {
        if (r + w * rstep < r1) {
          q0[w] = *reinterpret_cast<const uint4*>(F.p0 + ((r + w * rstep) * Q + col0) * 2);
          if constexpr (FastTraits<K>::load1)
            q1[w] = *reinterpret_cast<const uint4*>(F.p1 + ((r + w * rstep) * Q + col0) * 2);
        }
      }
#pragma unroll
      for (int w = 0; w < W; ++w) {
        if (r + w * rstep < r1) {
          float a[8], b[8], x[8];
          unpack8(q0[w], F.dt0, a);
          if constexpr (FastTraits<K>::load1) unpack8(q1[w], F.dt1, b);
          fast_apply<K>(F, a, b, none, x);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], x[j]);
        }
      }
    }
  }
  col_combine<8>(c, t, ch, p, acc, red, pre);
}

template <int V>
__device__ __noinline__ void run_reduce_col(const Ctx c, const Task& t, int item, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t ch = item / t.parts;
  const int p = item % t.parts;
  const int64_t Q = t.red_inner;
  const int64_t col0 = ch * 32 * V + lane * V;
  const int64_t r0 = int64_t(p) * t.part_len;
  const int64_t r1 = min(t.red_outer, r0 + t.part_len);
  const int64_t my_col = ch * 32 * V + threadIdx.x;
  const float pre = t.parts == 1 && threadIdx.x < 32 * V && my_col < Q ? post_operand(c, t, my_col) : 0.0f;
  float acc[V];
#pragma unroll
  for (int j = 0; j < V; ++j) acc[j] = 0.0f;
  if (col0 < Q) {
    for (int64_t r = r0 + warp; r < r1; r += kThreads / 32) {
      int64_t crd[kMaxRank];
      unravel(t, r * Q + col0, crd);
      float v[V];
      eval_expr<V>(c, t, crd, nullptr, v);
#pragma unroll
      for (int j = 0; j < V; ++j) acc[j] = __fadd_rn(acc[j], v[j]);
    }
  }
  col_combine<V>(c, t, ch, p, acc, red, pre);
}

__device__ __noinline__ void run_reduce_final(const Ctx c, const Task& t, int item, float* red) {
  const float* part = reinterpret_cast<const float*>(c.ws) + t.scratch;
  if (t.final_block) {
    const int64_t o = item;
    const float pre = threadIdx.x == 0 ? post_operand(c, t, o) : 0.0f;
    float acc = 0.0f;
    for (int q = threadIdx.x; q < t.parts; q += kThreads) acc = __fadd_rn(acc, part[o * t.parts + q]);
    acc = block_sum(acc, red);
    if (threadIdx.x == 0) finish_reduction(c, t, o, acc, pre);
  } else {
    const int64_t o = int64_t(item) * kThreads + threadIdx.x;
    if (o >= t.red_outer) return;
    const float pre = post_operand(c, t, o);
    float acc = 0.0f;
    for (int q = 0; q < t.parts; ++q) acc = __fadd_rn(acc, part[o * t.parts + q]);
    finish_reduction(c, t, o, acc, pre);
  }
}

// One-row GEMM: warp w of the item computes output n = 8 * item + w; lane l
// sums k = 8l + 256j, 8 elements at a time, in j order; the lanes' sums are
// added by a fixed butterfly; lane 0 applies the epilogue.
__device__ __noinline__ void run_gemv(const Ctx c, const Task& t, int item) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n = int64_t(item) * (kThreads / 32) + warp;
  if (n >= t.n) return;
  const char* pa = space_ptr(c, t.a.space, t.a.slot);
  const char* pb = space_ptr(c, t.b.space, t.b.slot);
  const int64_t brow = t.b.base + n * t.b.stride[1];
  float acc = 0.0f;
  for (int64_t k = int64_t(lane) * 8; k < t.k; k += 256) {
    float a[8], b[8];
    load8(pa, t.a.dtype, t.a.base + k, a);
    load8(pb, t.b.dtype, brow + k, b);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc = fmaf(a[j], b[j], acc);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
  if (lane == 0) {
    int64_t crd[kMaxRank] = {0, n, 0, 0};
    float v[1];
    const float a1[1] = {acc};
    eval_expr<1>(c, t, crd, a1, v);
    store_out<1>(c, t.out, n, v);
    if (t.has_side) store_side<1>(c, t, n, v);
  }
}

// CUDA-core GEMM tile: TM x TM outputs, 16 x 16 threads, (TM/16)^2 each;
// float32 fmaf accumulation in k order, then the epilogue expression.
template <int TM>
__device__ __noinline__ void run_gemm_simt(const Ctx c, const Task& t, int item, float* smem) {
  constexpr int KT = 16, P = TM + 4, R = TM / 16;
  float* As = smem;           // [KT][P]
  float* Bs = smem + KT * P;  // [KT][P]
  const int64_t m0 = int64_t(item / t.tiles_n) * TM, n0 = int64_t(item % t.tiles_n) * TM;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const char* pa = space_ptr(c, t.a.space, t.a.slot);
  const char* pb = space_ptr(c, t.b.space, t.b.slot);
  float acc[R][R];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int j = 0; j < R; ++j) acc[i][j] = 0.0f;
  for (int64_t k0 = 0; k0 < t.k; k0 += KT) {
    for (int q = threadIdx.x; q < TM * KT; q += kThreads) {
      int mm, kk;
      if (t.a_kcontig) {
        mm = q / KT;
        kk = q % KT;
      } else {
        kk = q / TM;
        mm = q % TM;
      }
      const int64_t gm = m0 + mm, gk = k0 + kk;
      As[kk * P + mm] = (gm < t.m && gk < t.k)
                            ? load1(pa, t.a.dtype, t.a.base + gm * t.a.stride[0] + gk * t.a.stride[1])
                            : 0.0f;
      int nn;
      if (t.b_ncontig) {
        kk = q / TM;
        nn = q % TM;
      } else {
        nn = q / KT;
        kk = q % KT;
      }
      const int64_t gn = n0 + nn, gk2 = k0 + kk;
      Bs[kk * P + nn] = (gn < t.n && gk2 < t.k)
                            ? load1(pb, t.b.dtype, t.b.base + gk2 * t.b.stride[0] + gn * t.b.stride[1])
                            : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      float a[R], b[R];
#pragma unroll
      for (int i = 0; i < R; ++i) a[i] = As[kk * P + ty * R + i];
#pragma unroll
      for (int j = 0; j < R; ++j) b[j] = Bs[kk * P + tx * R + j];
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int j = 0; j < R; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int64_t row = m0 + ty * R + i;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int64_t col = n0 + tx * R + j;
      if (row < t.m && col < t.n) {
        int64_t crd[kMaxRank] = {row, col, 0, 0};
        float v[1];
        const float a1[1] = {acc[i][j]};
        eval_expr<1>(c, t, crd, a1, v);
        store_out<1>(c, t.out, row * t.n + col, v);
        if (t.has_side) store_side<1>(c, t, row * t.n + col, v);
      }
    }
  }
}

// ---------------------------------------------------- tcgen05 tile path
//
// Warp roles while a stage's tensor-core tiles run (8 warps):
//   warp 0, lane 0: TMA producer -- waits for a free ring slot, arms its
//                   "full" mbarrier with the byte count and issues the A/B
//                   tile loads;
//   warp 1, lane 0: MMA issuer -- waits for a full slot, issues four
//                   tcgen05.mma (K = 16 each) into the TMEM accumulator and
//                   commits the slot back to "empty"; after the last K block
//                   it commits the accumulator to "acc_full";
//   warps 4..7:     epilogue -- each reads its 32 TMEM lanes (tile rows) with
//                   tcgen05.ld, runs the task's epilogue expression on 8
//                   columns at a time and stores; then frees the accumulator.
// Two accumulators (2 x 256 TMEM columns) let the epilogue of one tile
// overlap the MMAs of the next.  Ring and accumulator counters live in the
// role's registers for the whole kernel, so every stage continues the same
// phase sequence.

// An epilogue warp's staging ring: the task whose layout it currently holds,
// the chunks staged through it since that task began (chunk k uses buffer
// k % depth of each region) and the phase of each buffer's load mbarrier.
struct EpiRing {
  int32_t task;
  uint32_t k;
  uint32_t phases;
};

struct TcState {
  uint32_t ring;                  // shared address of the 1024-aligned ring
  uint32_t slot_bytes;            // bytes per ring slot (A tile, then B tile)
  uint32_t full, empty;           // shared addresses of kStages mbarriers each
  uint32_t acc_full, acc_empty;   // 2 mbarriers each
  uint32_t drain;                 // MMA completion after a failed wait (used once)
  uint32_t tmem;                  // TMEM base address
  uint32_t acc_cols;              // TMEM columns per accumulator buffer (half the allocation)
  uint32_t stg;                   // shared address of the epilogue staging area
  uint32_t stg_warp_bytes;        // staging bytes per epilogue warp
  uint32_t epi_bar;               // kEpiMaxDepth mbarriers per epilogue warp (staged-epilogue operand loads)
  const CUtensorMap* maps;        // the launch's TMA descriptors
  uint32_t p_it, m_it, m_tile, e_tile;
  EpiRing er;                      // this epilogue warp's staging ring
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long timeout_ns) {
  for (int i = 0; i < 256; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > timeout_ns) return false;
  return true;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// ------------------------------------------------- pairs of SMs (clusters of 2)
//
// A pair-tile launch runs in clusters of two blocks on two SMs.  The even
// block of a pair (its leader) issues the pair's MMAs (cta_group::2): A rows
// 0-127 of a 256-row tile come from the leader's shared memory and rows
// 128-255 from the peer's, at the same offset; B's columns are split in halves
// the same way; each block's TMEM holds the accumulator rows of its half.

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of `addr` (a shared::cta address of this block)
// in block `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive on an mbarrier of another block of the cluster (cluster-scope release).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// All threads of both blocks of the pair meet (cluster-scope release/acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// TMA loads into this block's shared memory whose completion is counted on an
// mbarrier of either block of the pair (cluster_bar: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                                 uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(cluster_bar)
      : "memory");
}

// TMA loads of a box into this block's and the other pair block's shared
// memory (same offset), completing on the mbarrier at `bar`'s offset in each.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_mc(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                               uint32_t bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "h"(mask)
      : "memory");
}

// Bounded wait with cluster-scope acquire (for phases completed by arrivals
// from the other block of the pair).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, long long timeout_ns) {
  for (int i = 0; i < 256; ++i)
    if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = global_ns();
  while (!mbar_try_wait_cluster(bar, parity))
    if (global_ns() - t0 > timeout_ns) return false;
  return true;
}

// One contiguous global -> shared bulk copy (both 16-byte aligned, size a
// multiple of 16) completing on mbarrier bar.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// ------------------------------------------- bulk-streamed reductions
//
// A long reduction over 16-bit operands keeps only 32 KB per SM in flight
// with register loads (eight 16-byte vectors per thread), far too little to
// cover the memory latency at full bandwidth with one block per SM.  In a
// tensor-core launch the TMA ring is idle during a stage's reductions, so
// these variants copy the operands into up to kBulkMaxSlots slots of it with
// bulk copies (16 KB per slot, all slots in flight) and sum from shared
// memory.  Each thread sums exactly the elements, in exactly the order, of
// the register-streaming variant, so the two give the same bits.

__device__ __forceinline__ uint4 lds128(uint32_t a);

// Slot k of the block's running slot sequence: its shared address and the
// parity of the phase that its copy completes.
struct BulkSlot {
  uint32_t addr, bar, parity;
};
__device__ __forceinline__ BulkSlot bulk_slot(const Ctx& c, uint32_t k) {
  const uint32_t s = k % uint32_t(c.bulk_slots);
  return {c.bulk + s * uint32_t(kBulkSlotBytes), c.bulk_bar + 8 * s, (k / uint32_t(c.bulk_slots)) & 1u};
}

// After a wait ran out at chunk ch (known to every thread): thread 0 waits,
// again with the time limit, for the copies still in flight (chunks ch up to
// ch + S - 1) so that none lands after the block has moved on, and records
// the failure.  Returns the number of chunks issued.
__device__ __noinline__ int bulk_abandon(const Ctx c, uint32_t it0, int ch, int nch) {
  const int issued = min(nch, ch + c.bulk_slots);
  if (threadIdx.x == 0) {
    for (int k = ch; k < issued; ++k) {
      const BulkSlot b = bulk_slot(c, it0 + uint32_t(k));
      mbar_wait(b.bar, b.parity, c.timeout_ns);
    }
    record_failure(c, TK_ERR_PIPELINE_TIMEOUT, c.stage);
  }
  __syncthreads();
  return issued;
}

template <int K>
__device__ __noinline__ float row_sum_bulk16(const Ctx c, const Task& t, int64_t o, int64_t r0, int64_t r1) {
  constexpr bool L1 = FastTraits<K>::load1;
  constexpr int64_t step = int64_t(kThreads) * 8;                         // elements per block-wide pass
  constexpr int64_t chunk = (L1 ? kBulkSlotBytes / 2 : kBulkSlotBytes) / 2;  // elements per slot and operand
  constexpr int passes = int(chunk / step);
  const Fast F = fast_params(c, t);
  const char* p0 = F.p0 + (o * t.red_inner + r0) * 2;
  const char* p1 = L1 ? F.p1 + (o * t.red_inner + r0) * 2 : nullptr;
  const int64_t n = r1 - r0;
  const bool aligned = (reinterpret_cast<uintptr_t>(p0) & 15) == 0 && (!L1 || (reinterpret_cast<uintptr_t>(p1) & 15) == 0);
  if (c.bulk_slots < 2 || n < 2 * chunk || n % 8 != 0 || !aligned) return row_sum_fast16<K>(c, t, o, r0, r1);
  const int S = c.bulk_slots;
  const int nch = int((n + chunk - 1) / chunk);
  const uint32_t it0 = *c.bulk_it;
  auto issue = [&](int ch) {
    const BulkSlot b = bulk_slot(c, it0 + uint32_t(ch));
    const int64_t e0 = int64_t(ch) * chunk;
    const uint32_t bytes = uint32_t(min(chunk, n - e0) * 2);
    mbar_expect_tx(b.bar, L1 ? 2 * bytes : bytes);
    bulk_g2s(b.addr, p0 + e0 * 2, bytes, b.bar);
    if constexpr (L1) bulk_g2s(b.addr + kBulkSlotBytes / 2, p1 + e0 * 2, bytes, b.bar);
  };
  if (threadIdx.x == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (int ch = 0; ch < min(S, nch); ++ch) issue(ch);
  }
  float acc = 0.0f, none[8];
  int done = nch;
#pragma unroll 1
  for (int ch = 0; ch < nch; ++ch) {
    const BulkSlot b = bulk_slot(c, it0 + uint32_t(ch));
    const bool ok = mbar_wait(b.bar, b.parity, c.timeout_ns);
    const uint32_t src = b.addr + threadIdx.x * 16;
    const int64_t e0 = int64_t(ch) * chunk + int64_t(threadIdx.x) * 8;
#pragma unroll
    for (int j = 0; j < passes; ++j) {
      if (ok && e0 + j * step < n) {
        float a[8], bb[8], x[8];
        unpack8(lds128(src + uint32_t(j * step * 2)), F.dt0, a);
        if constexpr (L1) unpack8(lds128(src + kBulkSlotBytes / 2 + uint32_t(j * step * 2)), F.dt1, bb);
        fast_apply<K>(F, a, bb, none, x);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc = __fadd_rn(acc, x[q]);
      }
    }
    // slot read by every thread before it is refilled; a wait that ran out
    // anywhere ends the loop everywhere
    if (__syncthreads_or(!ok)) {
      done = bulk_abandon(c, it0, ch, nch);
      break;
    }
    if (threadIdx.x == 0 && ch + S < nch) issue(ch + S);
  }
  if (threadIdx.x == 0) *c.bulk_it = it0 + uint32_t(done);
  return acc;
}

// Column sums: a slot holds consecutive rows of the item's 256 columns (one
// 512-byte line per row).  Rows of 512 bytes are too short for bulk copies,
// so every thread moves its 16-byte pieces with cp.async and a per-thread
// arrive-on on the slot's mbarrier (which counts all kThreads threads) marks
// them done; warp w sums rows r0 + w + 8i in increasing i as in the register
// variant.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src);
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

template <int K>
__device__ __noinline__ void run_reduce_col_bulk16(const Ctx c, const Task& t, int item, float* red) {
  constexpr bool L1 = FastTraits<K>::load1;
  constexpr int rows = (L1 ? kBulkSlotBytes / 2 : kBulkSlotBytes) / 512;  // rows per slot
  constexpr int pieces = rows * 32 / kThreads;                            // 16-byte pieces per thread
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t ch = item / t.parts;
  const int p = item % t.parts;
  const int64_t Q = t.red_inner;
  const int64_t r0 = int64_t(p) * t.part_len;
  const int64_t r1 = min(t.red_outer, r0 + t.part_len);
  const Fast F = fast_params(c, t);
  const bool aligned = (reinterpret_cast<uintptr_t>(F.p0) & 15) == 0 && (!L1 || (reinterpret_cast<uintptr_t>(F.p1) & 15) == 0);
  if (c.bulk_slots < 2 || r1 - r0 < 2 * rows || Q % 8 != 0 || !aligned) {
    run_reduce_col_fast16<K>(c, t, item, red);
    return;
  }
  const int64_t col0 = ch * 256 + lane * 8;
  const int64_t my_col = ch * 256 + threadIdx.x;
  const float pre = t.parts == 1 && my_col < Q ? post_operand(c, t, my_col) : 0.0f;
  const int seg = int(min(int64_t(256), Q - ch * 256) * 2);  // bytes per row
  const int S = c.bulk_slots;
  const int nch = int((r1 - r0 + rows - 1) / rows);
  const uint32_t it0 = *c.col_it;
  auto slot = [&](int i) {
    const uint32_t k = it0 + uint32_t(i), s = k % uint32_t(S);
    return BulkSlot{c.bulk + s * uint32_t(kBulkSlotBytes), c.col_bar + 8 * s, (k / uint32_t(S)) & 1u};
  };
  auto issue = [&](int i) {  // every thread
    const BulkSlot b = slot(i);
    const int64_t rr = r0 + int64_t(i) * rows;
#pragma unroll
    for (int m = 0; m < pieces; ++m) {
      const int q = int(threadIdx.x) + kThreads * m, row = q >> 5, pc = q & 31;
      if (rr + row < r1 && pc * 16 < seg) {
        const int64_t off = ((rr + row) * Q + ch * 256) * 2 + pc * 16;
        cp_async16(b.addr + uint32_t(row * 512 + pc * 16), F.p0 + off);
        if constexpr (L1) cp_async16(b.addr + kBulkSlotBytes / 2 + uint32_t(row * 512 + pc * 16), F.p1 + off);
      }
    }
    cp_async_arrive(b.bar);
  };
  for (int i = 0; i < min(S, nch); ++i) issue(i);
  float acc[8], none[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
  int done = nch;
#pragma unroll 1
  for (int i = 0; i < nch; ++i) {
    const BulkSlot b = slot(i);
    const bool ok = mbar_wait(b.bar, b.parity, c.timeout_ns);
    const int64_t rr = r0 + int64_t(i) * rows;
    if (ok && col0 < Q) {
      const uint32_t src = b.addr + uint32_t(lane) * 16;
#pragma unroll
      for (int w = 0; w < rows / 8; ++w) {
        const int rl = warp + 8 * w;
        if (rr + rl < r1) {
          float a[8], bb[8], x[8];
          unpack8(lds128(src + uint32_t(rl) * 512), F.dt0, a);
          if constexpr (L1) unpack8(lds128(src + kBulkSlotBytes / 2 + uint32_t(rl) * 512), F.dt1, bb);
          fast_apply<K>(F, a, bb, none, x);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], x[q]);
        }
      }
    }
    // slot read by every thread before it is refilled; a wait that ran out
    // anywhere ends the loop everywhere, after this thread's copies landed
    if (__syncthreads_or(!ok)) {
      asm volatile("cp.async.wait_all;" ::: "memory");
      __syncthreads();
      if (threadIdx.x == 0) record_failure(c, TK_ERR_PIPELINE_TIMEOUT, c.stage);
      done = min(nch, i + S);
      break;
    }
    if (i + S < nch) issue(i + S);
  }
  if (threadIdx.x == 0) *c.col_it = it0 + uint32_t(done);
  col_combine<8>(c, t, ch, p, acc, red, pre);
}

// Shared-memory matrix descriptor, 128-byte swizzle: start, leading and
// stride byte offsets in 16-byte units, descriptor version 1 (bit 46),
// layout SWIZZLE_128B (2 in bits 61-63).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((addr >> 4) & 0x3FFF) | (uint64_t((lbo >> 4) & 0x3FFF) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFF) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// The pair forms (every tcgen05 operation of a pair-tile launch uses
// cta_group::2): one MMA over both blocks' operands, and commits that arrive
// on the mbarrier at offset `bar` in the blocks of `mask` or in this block.
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               ::"r"(bar), "h"(mask)
               : "memory");
}
// A single block's commit arriving on the mbarrier at `bar`'s offset in the
// blocks of `mask` (a shared-B pair: both blocks' MMAs free a ring slot).
__device__ __forceinline__ void umma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               ::"r"(bar), "h"(mask)
               : "memory");
}
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]),
               "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
               "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
               "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]),
               "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])::"memory");
}

// 8 consecutive accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])::"memory");
}

// One tensor-core work item: a tile and, for split-K, its range of k blocks.
struct TileItem {
  int64_t m0, n0;
  int kb0, kb1, split;
};

// Walk this block's tensor-core items of a stage in order (all roles use the
// same sequence; in a pair-tile launch both blocks of a pair walk the pair's
// 256-row tiles, m0 being the tile's first row).  fn(task, item) returns
// false to stop.
template <bool PAIR, typename F>
__device__ __forceinline__ void for_my_tiles(const Ctx& c, const Stage& st, F&& fn) {
  int ti = st.task_begin, base = 0;
  const int g0 = PAIR ? int(blockIdx.x >> 1) : int(blockIdx.x), step = PAIR ? int(gridDim.x >> 1) : int(gridDim.x);
  for (int g = g0; g < st.n_tc_items; g += step) {
    while (g >= base + c.tasks[ti].n_items) {
      base += c.tasks[ti].n_items;
      ++ti;
    }
    const Task& t = c.tasks[ti];
    const int item = g - base, tile = item / t.k_splits, split = item - tile * t.k_splits;
    TileItem it;
    it.m0 = int64_t(tile / t.tiles_n) * (PAIR ? 2 * kTileM : kTileM);
    it.n0 = int64_t(tile % t.tiles_n) * t.tile_n;
    it.split = split;
    it.kb0 = split * t.kb_split;
    it.kb1 = min(t.k_blocks, it.kb0 + t.kb_split);
    if (!fn(t, it)) return;
  }
}

__device__ __noinline__ void tc_epilogue_tile_chain(const Ctx c, const Task& t, int64_t m0, int64_t n0,
                                                    uint32_t taddr) {
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const int64_t row = m0 + q * 32 + lane;
  const int64_t M = t.m, N = t.n;
  const int tile_n = t.tile_n;
  const bool live = row < M;
  Prep& P = c.prep[threadIdx.x >> 5];
  prepare(c, t, P);
  for (int cc = 0; cc < tile_n; cc += 32) {
    uint32_t r[32];
    __syncwarp();
    tmem_ld32(taddr + (uint32_t(q * 32) << 16) + uint32_t(cc), r);
    if (!live) continue;
    const int64_t col0 = n0 + cc;
    // operand loads two vectors at a time, issued before their arithmetic
#pragma unroll
    for (int v = 0; v < 4; v += 2) {
      float L[2][2][8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int32_t crd[kMaxRank] = {int32_t(row), int32_t(col0 + 8 * (v + h)), 0, 0};
        if (col0 + 8 * (v + h) < N) prep_load<8>(P, crd, L[h]);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t col = col0 + 8 * (v + h);
        if (col < N) {
          float a8[8], out[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) a8[j] = __uint_as_float(r[8 * (v + h) + j]);
          chain_compute<8>(P.ch, L[h], a8, out);
          prep_store<8>(P, row * N + col, out);
          if (t.has_side) store_side<8>(c, t, row * N + col, out);
        }
      }
    }
  }
}

// A FastKind epilogue: thread (q, lane) owns tile row q*32+lane; per 32-column
// chunk it reads its accumulator slice from TMEM, issues all operand loads,
// then computes and stores 4 vectors of 8.
template <int K>
__device__ __noinline__ void tc_epilogue_fast(const Ctx c, const Task& t, int64_t m0, int64_t n0, uint32_t taddr) {
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const int64_t row = m0 + q * 32 + lane;
  const int64_t N = t.n;
  const int tile_n = t.tile_n;
  const bool live = row < t.m;
  const Fast F = fast_params(c, t);
  const char* p0 = FastTraits<K>::load0 ? F.p0 + row * F.rs0 : nullptr;
  const char* p1 = FastTraits<K>::load1 ? F.p1 + row * F.rs1 : nullptr;
  const int64_t orow = row * N;
  for (int cc = 0; cc < tile_n; cc += 32) {
    uint32_t r[32];
    __syncwarp();
    tmem_ld32(taddr + (uint32_t(q * 32) << 16) + uint32_t(cc), r);
    if (!live) continue;
    const int64_t col0 = n0 + cc;
    float l0[4][8], l1[4][8];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int64_t col = col0 + 8 * v;
      if (col < N) {
        if constexpr (FastTraits<K>::load0) load8(p0, F.dt0, col, l0[v]);
        if constexpr (FastTraits<K>::load1) load8(p1, F.dt1, col, l1[v]);
      }
    }
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int64_t col = col0 + 8 * v;
      if (col < N) {
        float a8[8], x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a8[j] = __uint_as_float(r[8 * v + j]);
        fast_apply<K>(F, l0[v], l1[v], a8, x);
        store8(F.out, F.out_dt, orow + col, x);
        if (t.has_side) store_side<8>(c, t, orow + col, x);
      }
    }
  }
}

// ---------------------------------------------- staged GEMM epilogue
//
// TMEM gives each epilogue thread one row of the tile, so direct global
// accesses put 32 rows behind every warp instruction (32 L1 wavefronts).  The
// staged epilogue moves each 32 x 32 chunk through shared memory instead:
// per-row operands arrive by cp.async in row-contiguous order (issued a chunk
// ahead, the first before the accumulator is ready), each thread reads its
// row from shared memory, writes its results back there, and the warp stores
// the chunk with 4 threads per 64-byte row.
//
// Piece j (16 bytes, 0..3) of row r in a 32 x 64-byte buffer sits at a
// swizzled position so that both access patterns are free of bank conflicts.
__device__ __forceinline__ uint32_t stg_off(int r, int j) {
  return uint32_t(r * 64 + ((j ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// A GEMM's side output from a staged chunk: each lane turns its row of the
// stored (rounded) values in `buf` into the side values and writes them to
// `dst` (buf itself, a buffer of its own, or for a loaded side the buffer
// holding its operand, read from there).  Every value is of the 16-bit type
// DT.  The caller stores dst.
template <int DT>
__device__ __forceinline__ void stage_side(const Task& t, uint32_t buf, uint32_t dst) {
  const int lane = threadIdx.x & 31;
  const bool loaded = t.side.ext == EXT_LOAD1;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    float x[8], e[8];
    unpack8(lds128(buf + stg_off(lane, v)), DT, x);
    if (loaded) {
      unpack8(lds128(dst + stg_off(lane, v)), DT, e);
      const bool sub = t.side.op == OP_SUB, second = t.side.second;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float a = second ? e[j] : x[j], b = second ? x[j] : e[j];
        const float p = __fmul_rn(t.side.imm, b);
        x[j] = sub ? __fsub_rn(a, p) : __fadd_rn(a, p);
      }
    } else if (t.side.op == OP_MUL) {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = __fmul_rn(x[j], t.side.cval);
    } else if (t.side.op == OP_NEG) {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = -x[j];
    }
    sts128(dst + stg_off(lane, v), pack8(x, DT));  // rounds to the side's type
  }
}

// TMA store of a staged 32 x 32 chunk (64-byte swizzle) at (col, row) of the
// tensor behind `map`; rows and columns beyond the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed bulk store of this thread has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed bulk store of this thread has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Lane 0: every bulk store group this thread committed, except the `n` most
// recent ones, has finished reading shared memory (n above 7 waits as for 7).
__device__ __forceinline__ void bulk_wait_read_n(uint32_t n) {
  switch (n) {
    case 0: asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group.read 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group.read 6;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group.read 7;" ::: "memory"); break;
  }
}

// Returns false if a wait timed out.  The tile's 32-column chunks move through
// this warp's staging ring of D = t.epi_depth buffers per region: per-row
// operands (the target, the ReLU mask input, the parameter being updated, a
// loaded side's operand) arrive as 32 x 32 TMA boxes on the buffer's mbarrier,
// up to D - 1 chunks ahead (D - 2 from D = 4 on, so that a refill never waits
// for the stores of the chunk just finished); each lane turns its row of the
// chunk into outputs in shared memory (in place in the first per-row operand's
// buffer, else in the chunk's output buffer), and lane 0 stores the chunk with
// a TMA store, a side output the same way (from its own buffer, from the
// loaded side's buffer, or in place once the output's store has read it).
// Lane 0 commits one bulk group per chunk, so a buffer last used by ring chunk
// j is free once all but the groups of the chunks after j have been read.  An
// operand with one row for all tile rows (a bias) is copied once per tile by
// cp.async: its tile_n values.
template <int K, int DT>
__device__ __noinline__ bool tc_epilogue_staged(const Ctx c, const Task& t, int task_id, int64_t m0, int64_t n0,
                                                uint32_t taddr, uint32_t stg, uint32_t acc_bar, uint32_t phase,
                                                long long* stamp, const CUtensorMap* maps, uint32_t ebar,
                                                EpiRing* er) {
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const int row0 = int(m0) + q * 32;
  // 32-column chunks holding columns of the output (a 224-wide tile at the
  // right edge may hold only a few)
  const uint32_t nch = uint32_t((min(int64_t(t.tile_n), int64_t(t.n) - n0) + 31) / 32);
  const int mask = t.epi_stage;
  const uint32_t D = uint32_t(t.epi_depth), dmask = D - 1;  // 2, 4 or 8
  constexpr bool L0 = FastTraits<K>::load0, L1 = FastTraits<K>::load1;
  const bool st0 = L0 && (mask & 1), st1 = L1 && (mask & 2);
  const bool sl = t.has_side && t.side.ext == EXT_LOAD1 && (mask & 8);
  const bool su = t.has_side && !sl && (mask & 16);
  // every operand, rounding and output is of type DT: the conversions are
  // compiled for it, with no branch on a type read at run time
  Fast F = fast_params(c, t);
  F.dt0 = F.dt1 = F.out_dt = DT;
  F.r0 = F.r1 = F.r2 = F.er = DT;
  // per warp, regions of D buffers (each a multiple of 512 bytes, the 64-byte
  // swizzle's alignment): per-row operand 0, per-row operand 1, the outputs
  // when there is no per-row operand, a loaded side's operand, a unary side's
  // values; then one kBcastBytes row per one-row operand
  const uint32_t reg = D * kEpiBufBytes;
  const uint32_t b0 = stg, b1 = b0 + (st0 ? reg : 0);
  const uint32_t only = b1 + (st1 ? reg : 0);
  const uint32_t bs = only + (st0 || st1 ? 0 : reg);
  const uint32_t bu = bs + (sl ? reg : 0);
  const uint32_t r0 = bu + (su ? reg : 0);
  const uint32_t r1 = r0 + (L0 && !st0 ? kBcastBytes : 0);
  const bool loads = st0 || st1 || sl;
  const bool own_out = !(st0 || st1) || su;  // buffers written without a load first
  const uint32_t ld_bytes = uint32_t(int(st0) + int(st1) + int(sl)) * kEpiBufBytes;
  if (row0 >= t.m) {
    // no output row in this warp's lane quarter (a short GEMM): nothing to
    // load, compute or store; the accumulator is still waited for, so that
    // this warp's release of it follows the MMAs that wrote it
    const bool ok = mbar_wait(acc_bar, phase, c.timeout_ns);
    if (ok && stamp) *stamp = global_ns();
    return ok;
  }
  if (er->task != task_id) {
    // the staging area takes this task's layout: every earlier store has
    // finished reading it first
    if (lane == 0) bulk_wait_read();
    er->task = task_id;
    er->k = 0;
  }
  const uint32_t k = er->k;
  const uint32_t lag = D >= 4 ? 2u : 1u;
  // lane 0: before chunk j's buffers are refilled or rewritten, the stores of
  // ring chunk k + j - D (their last user) have read them; ring chunks before
  // `done` have committed their groups
  auto free_bufs = [&](uint32_t j, uint32_t done) {
    const uint32_t kk = k + j;
    if (kk >= D) bulk_wait_read_n(done - 1u - (kk - D));
  };
  auto load = [&](uint32_t j, uint32_t done) {  // lane 0
    free_bufs(j, done);
    const uint32_t b = (k + j) & dmask, bar = ebar + 8 * b, off = b * kEpiBufBytes;
    const int x = int(n0) + 32 * int(j);
    mbar_expect_tx(bar, ld_bytes);
    if (st0) tma_load_2d(b0 + off, &maps[t.tma_ld0], x, row0, bar);
    if (st1) tma_load_2d(b1 + off, &maps[t.tma_ld1], x, row0, bar);
    if (sl) tma_load_2d(bs + off, &maps[t.tma_sd], x, row0, bar);
  };

  // one-row operands: 8 values per lane, once per tile
  {
    const int64_t col = n0 + 8 * lane;
    if (8 * lane < t.tile_n && col < t.n) {
      if (L0 && !st0) cp_async16(r0 + 16 * lane, F.p0 + col * 2);
      if (L1 && !st1) cp_async16(r1 + 16 * lane, F.p1 + col * 2);
    }
  }
  cp_async_commit();
  uint32_t issued = 0;  // chunk loads issued (lane 0)
  if (loads && lane == 0)
    for (; issued < nch && issued + lag <= D; ++issued) load(issued, k);
  bool ok = mbar_wait(acc_bar, phase, c.timeout_ns);
  if (ok && stamp) *stamp = global_ns();
  tc_fence_after();
  cp_async_wait<0>();
  __syncwarp();
  uint32_t phases = er->phases;
  const uint32_t tlane = taddr + (uint32_t(q * 32) << 16);
  uint32_t ch = 0;
#pragma unroll 1
  for (; ok && ch < nch; ++ch) {
    const uint32_t kk = k + ch, b = kk & dmask, off = b * kEpiBufBytes;
    const int col0 = int(n0) + 32 * int(ch);
    if (lane == 0) {
      if (loads)
        for (; issued < nch && issued + lag <= ch + D; ++issued) load(issued, kk);
      if (own_out) free_bufs(ch, kk);
    }
    if (loads) {
      if (!mbar_wait(ebar + 8 * b, (phases >> b) & 1u, c.timeout_ns)) {
        ok = false;
        break;
      }
      phases ^= 1u << b;
    }
    __syncwarp();
    const uint32_t ob = st0 ? b0 + off : (st1 ? b1 + off : only + off);
    uint32_t rv[32];
    tmem_ld32(tlane + 32 * ch, rv);
    // one 8-wide vector at a time: this thread's row, read and written in place
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      float l0[8], l1[8], a8[8], x[8];
      if constexpr (L0) unpack8(lds128(st0 ? b0 + off + stg_off(lane, v) : r0 + 64 * ch + 16 * v), F.dt0, l0);
      if constexpr (L1) unpack8(lds128(st1 ? b1 + off + stg_off(lane, v) : r1 + 64 * ch + 16 * v), F.dt1, l1);
#pragma unroll
      for (int j = 0; j < 8; ++j) a8[j] = __uint_as_float(rv[8 * v + j]);
      fast_apply<K, false>(F, l0, l1, a8, x);
      sts128(ob + stg_off(lane, v), pack8(x, F.out_dt));
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) tma_store_2d(&maps[t.tma_out], ob, col0, row0);
    if (t.has_side) {
      uint32_t dst = sl ? bs + off : bu + off;
      if (!sl && !su) {  // in place: the side values replace the outputs once their store has read them
        if (lane == 0) {
          bulk_commit();
          bulk_wait_read();
        }
        __syncwarp();
        dst = ob;
      }
      stage_side<DT>(t, ob, dst);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) tma_store_2d(&maps[t.tma_out2], dst, col0, row0);
    }
    if (lane == 0) bulk_commit();
  }
  if (!ok && lane == 0) {
    // a wait gave up: the loads already issued land, and the stores already
    // issued finish, before the block moves on
    for (uint32_t j = ch; j < issued; ++j) {
      const uint32_t b = (k + j) & dmask;
      mbar_wait(ebar + 8 * b, (phases >> b) & 1u, c.timeout_ns);
      phases ^= 1u << b;
    }
    bulk_wait_all();
  }
  __syncwarp();
  er->k = k + nch;
  er->phases = phases;
  return ok;
}

__device__ __noinline__ bool tc_epilogue_staged_any(const Ctx c, const Task& t, int task_id, int64_t m0, int64_t n0,
                                                    uint32_t taddr, uint32_t stg, uint32_t acc_bar, uint32_t phase,
                                                    long long* stamp, const CUtensorMap* maps, uint32_t ebar,
                                                    EpiRing* er) {
#define TK_STAGED(KIND, DT) \
  tc_epilogue_staged<KIND, DT>(c, t, task_id, m0, n0, taddr, stg, acc_bar, phase, stamp, maps, ebar, er)
#define TK_STAGED_KINDS(DT)                                       \
  switch (t.chain.fast) {                                         \
    case FK_E_ACC: return TK_STAGED(FK_E_ACC, DT);                \
    case FK_E_BIAS: return TK_STAGED(FK_E_BIAS, DT);              \
    case FK_E_BIAS_RELU: return TK_STAGED(FK_E_BIAS_RELU, DT);    \
    case FK_E_BIAS_AXPY: return TK_STAGED(FK_E_BIAS_AXPY, DT);    \
    case FK_E_ACC_THRESH: return TK_STAGED(FK_E_ACC_THRESH, DT);  \
    case FK_E_MOMENTUM: return TK_STAGED(FK_E_MOMENTUM, DT);      \
    default: return TK_STAGED(FK_E_UPDATE, DT);                   \
  }
  if (t.epi_dtype == TK_BF16) TK_STAGED_KINDS(TK_BF16)
  TK_STAGED_KINDS(TK_F16)
#undef TK_STAGED_KINDS
#undef TK_STAGED
}

// Split-K: this split's float32 accumulator, as is, to its scratch plane.
__device__ __noinline__ void tc_epilogue_partial(const Ctx c, const Task& t, int64_t m0, int64_t n0, int split,
                                                 uint32_t taddr) {
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const int64_t row = m0 + q * 32 + lane, M = t.m, N = t.n;
  float* plane = reinterpret_cast<float*>(c.ws) + t.scratch + int64_t(split) * M * N;
#pragma unroll 1
  for (int cc = 0; cc < t.tile_n; cc += 32) {
    uint32_t r[32];
    __syncwarp();
    tmem_ld32(taddr + (uint32_t(q * 32) << 16) + uint32_t(cc), r);
    if (row >= M) continue;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const int64_t col = n0 + cc + 4 * v;
      if (col < N)
        *reinterpret_cast<float4*>(plane + row * N + col) =
            make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]), __uint_as_float(r[4 * v + 2]),
                        __uint_as_float(r[4 * v + 3]));
    }
  }
}

// Split-K: the splits' partial accumulators summed in split order, then the
// GEMM's epilogue (V elements per thread, flat index over [M, N]).
template <int V>
__device__ __noinline__ void run_splitk_final(const Ctx c, const Task& t, int item) {
  const int64_t i0 = (int64_t(item) * kThreads + threadIdx.x) * V;
  const int64_t numel = t.numel;
  if (i0 >= numel) return;
  const float* part = reinterpret_cast<const float*>(c.ws) + t.scratch;
  float acc[V];
#pragma unroll
  for (int j = 0; j < V; ++j) acc[j] = 0.0f;
  for (int s = 0; s < t.k_splits; ++s) {
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = __fadd_rn(acc[j], part[int64_t(s) * numel + i0 + j]);
  }
  int64_t crd[kMaxRank];
  unravel(t, i0, crd);
  float out[V];
  eval_expr<V>(c, t, crd, acc, out);
  store_out<V>(c, t.out, i0, out);
  if (t.has_side) store_side<V>(c, t, i0, out);
}

__device__ __noinline__ void tc_epilogue_tile_any(const Ctx c, const Task& t, int64_t m0, int64_t n0,
                                                  uint32_t taddr) {
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const int64_t row = m0 + q * 32 + lane;
  for (int cc = 0; cc < t.tile_n; cc += 32) {
    uint32_t r[32];
    __syncwarp();
    tmem_ld32(taddr + (uint32_t(q * 32) << 16) + uint32_t(cc), r);
    if (row >= t.m) continue;
    if (t.vec == 8) {
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int64_t col = n0 + cc + 8 * v;
        if (col < t.n) {
          float a8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) a8[j] = __uint_as_float(r[8 * v + j]);
          int64_t crd[kMaxRank] = {row, col, 0, 0};
          float out[8];
          vm_eval<8>(c, t, crd, a8, out);
          store_out<8>(c, t.out, row * t.n + col, out);
          if (t.has_side) store_side<8>(c, t, row * t.n + col, out);
        }
      }
    } else {
      for (int j = 0; j < 32; ++j) {
        const int64_t col = n0 + cc + j;
        if (col < t.n) {
          const float a1[1] = {__uint_as_float(r[j])};
          int64_t crd[kMaxRank] = {row, col, 0, 0};
          float out[1];
          eval_expr<1>(c, t, crd, a1, out);
          store_out<1>(c, t.out, row * t.n + col, out);
          if (t.has_side) store_side<1>(c, t, row * t.n + col, out);
        }
      }
    }
  }
}

__device__ __forceinline__ void tc_epilogue_tile(const Ctx& c, const Task& t, int64_t m0, int64_t n0, uint32_t taddr) {
  switch (t.chain.fast) {
    case FK_E_ACC: tc_epilogue_fast<FK_E_ACC>(c, t, m0, n0, taddr); return;
    case FK_E_BIAS: tc_epilogue_fast<FK_E_BIAS>(c, t, m0, n0, taddr); return;
    case FK_E_BIAS_RELU: tc_epilogue_fast<FK_E_BIAS_RELU>(c, t, m0, n0, taddr); return;
    case FK_E_BIAS_AXPY: tc_epilogue_fast<FK_E_BIAS_AXPY>(c, t, m0, n0, taddr); return;
    case FK_E_ACC_THRESH: tc_epilogue_fast<FK_E_ACC_THRESH>(c, t, m0, n0, taddr); return;
    case FK_E_UPDATE: tc_epilogue_fast<FK_E_UPDATE>(c, t, m0, n0, taddr); return;
    case FK_E_MOMENTUM: tc_epilogue_fast<FK_E_MOMENTUM>(c, t, m0, n0, taddr); return;
    default: break;
  }
  if (t.vec == 8 && t.chain.valid)
    tc_epilogue_tile_chain(c, t, m0, n0, taddr);
  else
    tc_epilogue_tile_any(c, t, m0, n0, taddr);
}

// Each role returns its updated ring/accumulator counter in the low 32 bits
// and 1 << 32 if all its waits completed.
//
// After a wait gave up, a role still owns asynchronous work it started: TMA
// copies into the ring (producer) and MMAs writing TMEM (MMA issuer).  Each
// waits, again with the time limit, for that work to land before returning,
// so that nothing arrives in shared memory or TMEM after the block has freed
// them and exited.
// PM: 0 one block per tile; 1 a pair of blocks per 256-row tile with
// cta_group::2 MMAs; 2 a pair per 256-row tile, each block its own 128-row
// MMAs, B's halves multicast to both blocks.
template <int PM>
__device__ __noinline__ uint64_t tc_producer(const Ctx c, const Stage st, const CUtensorMap* maps, const TcState ts,
                                             uint32_t p_it) {
  constexpr bool PAIR = PM == 1, MC = PM == 2, CL = PM != 0;
  constexpr uint32_t NS = PAIR ? kPairStages : kStages;
  bool ok = true;
  const uint32_t p_it0 = p_it;
  // pairs: this block loads its 128 rows of A and its half of B's columns;
  // PM 1: both blocks' copies complete on the leader's "full" mbarrier;
  // PM 2: the B half goes to both blocks, each counting the whole tile
  const uint32_t rank = CL ? cluster_rank() & 1u : 0u;
  const uint32_t leader = CL ? cluster_rank() & ~1u : 0u;
  const uint16_t mask = uint16_t(3u << leader);
  asm volatile("fence.proxy.async.global;" ::: "memory");
  for_my_tiles<CL>(c, st, [&](const Task& t, const TileItem& it) {
    const int half = CL ? t.tile_n / 2 : t.tile_n;  // B columns this block loads
    const uint32_t bytes = uint32_t(kStageBytesA + half * kTileK * 2);
    const uint32_t tile_bytes = uint32_t(kStageBytesA + t.tile_n * kTileK * 2);
    const int tma_a = t.tma_a, tma_b = t.tma_b;
    const int a_mn = t.a_mn_major, b_mn = t.b_mn_major;
    const int64_t m0 = it.m0 + int64_t(rank) * kTileM, n0 = it.n0 + int64_t(rank) * half;
    for (int kb = it.kb0; kb < it.kb1; ++kb) {
      const uint32_t slot = p_it % NS, ph = ((p_it / NS) & 1u) ^ 1u;
      if (!mbar_wait(ts.empty + 8 * slot, ph, c.timeout_ns)) return ok = false;
      const uint32_t full = ts.full + 8 * slot;
      const uint32_t a_dst = ts.ring + slot * ts.slot_bytes, b_dst = a_dst + kStageBytesA;
      const int k0 = kb * kTileK;
      if constexpr (PAIR) {
        if (rank == 0) mbar_expect_tx(full, 2 * bytes);  // the leader counts both blocks' bytes
        const uint32_t bar = cluster_addr(full, leader);
        if (!a_mn) {
          tma_load_2d_pair(a_dst, &maps[tma_a], k0, int(m0), bar);
        } else if (a_mn == 2) {
          tma_load_3d_pair(a_dst, &maps[tma_a], 0, k0, int(m0 >> 6), bar);
        } else {
          tma_load_2d_pair(a_dst, &maps[tma_a], int(m0), k0, bar);
          tma_load_2d_pair(a_dst + 8192, &maps[tma_a], int(m0) + 64, k0, bar);
        }
        if (!b_mn) {
          tma_load_2d_pair(b_dst, &maps[tma_b], k0, int(n0), bar);
        } else if (b_mn == 2) {
          tma_load_3d_pair(b_dst, &maps[tma_b], 0, k0, int(n0 >> 6), bar);
        } else {
          for (int j = 0; j < half / 64; ++j) tma_load_2d_pair(b_dst + 8192 * j, &maps[tma_b], int(n0) + 64 * j, k0, bar);
        }
      } else if constexpr (MC) {
        mbar_expect_tx(full, tile_bytes);  // own A, both B halves
        if (!a_mn) {
          tma_load_2d(a_dst, &maps[tma_a], k0, int(m0), full);
        } else if (a_mn == 2) {
          tma_load_3d(a_dst, &maps[tma_a], 0, k0, int(m0 >> 6), full);
        } else {
          tma_load_2d(a_dst, &maps[tma_a], int(m0), k0, full);
          tma_load_2d(a_dst + 8192, &maps[tma_a], int(m0) + 64, k0, full);
        }
        const uint32_t bh = b_dst + rank * uint32_t(half) * kTileK * 2;  // this block's half of the tile
        if (!b_mn) {
          tma_load_2d_mc(bh, &maps[tma_b], k0, int(n0), full, mask);
        } else if (b_mn == 2) {
          tma_load_3d_mc(bh, &maps[tma_b], 0, k0, int(n0 >> 6), full, mask);
        } else {
          for (int j = 0; j < half / 64; ++j) tma_load_2d_mc(bh + 8192 * j, &maps[tma_b], int(n0) + 64 * j, k0, full, mask);
        }
      } else {
        mbar_expect_tx(full, bytes);
        if (!a_mn) {
          tma_load_2d(a_dst, &maps[tma_a], k0, int(m0), full);
        } else if (a_mn == 2) {
          tma_load_3d(a_dst, &maps[tma_a], 0, k0, int(m0 >> 6), full);
        } else {
          tma_load_2d(a_dst, &maps[tma_a], int(m0), k0, full);
          tma_load_2d(a_dst + 8192, &maps[tma_a], int(m0) + 64, k0, full);
        }
        if (!b_mn) {
          tma_load_2d(b_dst, &maps[tma_b], k0, int(n0), full);
        } else if (b_mn == 2) {
          tma_load_3d(b_dst, &maps[tma_b], 0, k0, int(n0 >> 6), full);
        } else {
          for (int j = 0; j < half / 64; ++j) tma_load_2d(b_dst + 8192 * j, &maps[tma_b], int(n0) + 64 * j, k0, full);
        }
      }
      ++p_it;
    }
    return true;
  });
  if (!ok && (!PAIR || rank == 0)) {
    // the copies of the last (up to) NS slots this stage armed: each
    // completes its slot's current "full" phase (a slot is re-armed only
    // after its previous phase was consumed, so that phase is still the one
    // with this parity; in a pair the leader's phases count the peer's
    // copies too)
    const uint32_t first = p_it - min(p_it - p_it0, NS);
    for (uint32_t i = first; i < p_it; ++i) mbar_wait(ts.full + 8 * (i % NS), (i / NS) & 1u, c.timeout_ns);
  }
  return (uint64_t(ok) << 32) | p_it;
}

template <int PM>
__device__ __noinline__ uint64_t tc_mma(const Ctx c, const Stage st, const TcState ts, uint32_t m_it,
                                        uint32_t* m_tile_io, long long* prof) {
  constexpr bool PAIR = PM == 1, MC = PM == 2, CL = PM != 0;
  constexpr uint32_t NS = PAIR ? kPairStages : kStages;
  // pair: the leader issues the pair's MMAs; its commits arrive on the
  // "empty" and accumulator mbarriers of both blocks
  if (PAIR && (cluster_rank() & 1u)) return uint64_t(1) << 32 | m_it;
  // (shared B: a slot is free once both blocks' MMAs have read it)
  const uint16_t pair_mask = CL ? uint16_t(3u << (cluster_rank() & ~1u)) : uint16_t(0);
  bool ok = true;
  bool first = true;
  uint32_t m_tile = *m_tile_io;
  for_my_tiles<CL>(c, st, [&](const Task& t, const TileItem& it) {
    const uint32_t acc = m_tile & 1u, ph = ((m_tile >> 1) & 1u) ^ 1u;
    // pair: the epilogue warps of both blocks release the accumulator
    const bool freed = PAIR ? mbar_wait_cluster(ts.acc_empty + 8 * acc, ph, c.timeout_ns)
                            : mbar_wait(ts.acc_empty + 8 * acc, ph, c.timeout_ns);
    if (!freed) return ok = false;
    tc_fence_after();
    const uint32_t d_tmem = ts.tmem + acc * ts.acc_cols;
    const uint32_t idesc = t.idesc;
    const bool a_mn = t.a_mn_major, b_mn = t.b_mn_major;
    for (int kb = it.kb0; kb < it.kb1; ++kb) {
      const uint32_t slot = m_it % NS, fph = (m_it / NS) & 1u;
      if (!mbar_wait(ts.full + 8 * slot, fph, c.timeout_ns)) return ok = false;
      if (prof && first) prof[3] = global_ns();
      first = false;
      tc_fence_after();
      const uint32_t a_base = ts.ring + slot * ts.slot_bytes, b_base = a_base + kStageBytesA;
#pragma unroll
      for (int k = 0; k < kTileK / 16; ++k) {
        const uint64_t ad = a_mn ? smem_desc(a_base + 2048 * k, 8192, 1024) : smem_desc(a_base + 32 * k, 16, 1024);
        const uint64_t bd = b_mn ? smem_desc(b_base + 2048 * k, 8192, 1024) : smem_desc(b_base + 32 * k, 16, 1024);
        if constexpr (PAIR)
          umma_f16_pair(d_tmem, ad, bd, idesc, uint32_t((kb - it.kb0) | k));
        else
          umma_f16(d_tmem, ad, bd, idesc, uint32_t((kb - it.kb0) | k));
      }
      if constexpr (PAIR)
        umma_commit_pair_mc(ts.empty + 8 * slot, pair_mask);
      else if constexpr (MC)
        umma_commit_mc(ts.empty + 8 * slot, pair_mask);
      else
        umma_commit(ts.empty + 8 * slot);
      ++m_it;
    }
    if constexpr (PAIR)
      umma_commit_pair_mc(ts.acc_full + 8 * acc, pair_mask);
    else
      umma_commit(ts.acc_full + 8 * acc);
    ++m_tile;
    return true;
  });
  if (!ok) {
    // every MMA this thread issued completes before the drain barrier's phase
    if constexpr (PAIR)
      umma_commit_pair(ts.drain);
    else
      umma_commit(ts.drain);
    mbar_wait(ts.drain, 0, c.timeout_ns);
  }
  *m_tile_io = m_tile;
  return (uint64_t(ok) << 32) | m_it;
}

template <int PM>
__device__ __noinline__ uint64_t tc_epilogue(const Ctx c, const Stage st, const TcState ts, uint32_t e_tile,
                                             long long* prof, EpiRing* er) {
  constexpr bool PAIR = PM == 1, CL = PM != 0;
  bool ok = true;
  bool first = true;
  const int lane = threadIdx.x & 31;
  const uint32_t ew = uint32_t(threadIdx.x >> 5) - 4;
  const uint32_t stg = ts.stg + ew * ts.stg_warp_bytes, ebar = ts.epi_bar + 8 * kEpiMaxDepth * ew;
  // pair: this block's accumulator rows are the tile's half `rank`; the
  // accumulator is released on the leader's mbarrier
  const uint32_t rank = CL ? cluster_rank() & 1u : 0u;
  const uint32_t acc_empty_leader = PAIR ? cluster_addr(ts.acc_empty, cluster_rank() & ~1u) : 0u;
  for_my_tiles<CL>(c, st, [&](const Task& t, const TileItem& it) {
    const int64_t m0 = it.m0 + int64_t(rank) * kTileM, n0 = it.n0;
    const uint32_t acc = e_tile & 1u, ph = (e_tile >> 1) & 1u;
    long long* stamp = prof && first && threadIdx.x == 128 ? prof + 5 : nullptr;
    first = false;
    if (t.k_splits > 1) {
      if (!mbar_wait(ts.acc_full + 8 * acc, ph, c.timeout_ns)) return ok = false;
      if (stamp) *stamp = global_ns();
      tc_fence_after();
      tc_epilogue_partial(c, t, m0, n0, it.split, ts.tmem + acc * ts.acc_cols);
    } else if (t.epi_stage) {
      if (!tc_epilogue_staged_any(c, t, int(&t - c.tasks), m0, n0, ts.tmem + acc * ts.acc_cols, stg,
                                  ts.acc_full + 8 * acc, ph, stamp, ts.maps, ebar, er))
        return ok = false;
    } else {
      if (!mbar_wait(ts.acc_full + 8 * acc, ph, c.timeout_ns)) return ok = false;
      if (stamp) *stamp = global_ns();
      tc_fence_after();
      tc_epilogue_tile(c, t, m0, n0, ts.tmem + acc * ts.acc_cols);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if constexpr (PAIR)
        mbar_arrive_cluster(acc_empty_leader + 8 * acc);
      else
        mbar_arrive(ts.acc_empty + 8 * acc);
    }
    ++e_tile;
    return true;
  });
  // the stage's TMA stores complete before the block reaches the grid barrier
  if (prof && threadIdx.x == 128) prof[8] = global_ns();
  if (lane == 0) bulk_wait_all();
  __syncwarp();
  return (uint64_t(ok) << 32) | e_tile;
}

// ------------------------------------ reductions beside the tensor-core tiles
//
// During a stage's tensor-core phase warps 2 and 3 have no role.  Reductions
// the planner marks `bg` run there instead of after the tiles: one warp per
// work item, emulating the eight warps of the 256-thread routines so that
// every output gets exactly the same additions in exactly the same order
// (per virtual thread the same elements in sequence; the same butterfly per
// virtual warp; the warps' totals added in warp order), hence the same bits.

// Row reduction item (output o, part p): virtual thread vt = 32 w + lane sums
// elements r0 + 8 vt + k * 2048 (k = 0, 1, ...), eight at a time in order.
template <int K, int DT>
__device__ __forceinline__ void bg_row_item(const Ctx& c, const Task& t, int item) {
  constexpr int64_t step = int64_t(kThreads) * 8;
  constexpr int VW = kThreads / 32;  // virtual warps
  const int lane = threadIdx.x & 31;
  const int64_t o = item / t.parts;
  const int p = item % t.parts;
  const int64_t r0 = int64_t(p) * t.part_len;
  const int64_t r1 = min(t.red_inner, r0 + t.part_len);
  const float pre = lane == 0 && t.parts == 1 ? post_operand(c, t, o) : 0.0f;
  const Fast F = fast_params(c, t);
  const int64_t row0 = o * t.red_inner;
  float acc[VW], none[8];
#pragma unroll
  for (int w = 0; w < VW; ++w) acc[w] = 0.0f;
  // all eight virtual warps' vectors in flight at a time
  for (int64_t base = r0; base < r1; base += step) {
#pragma unroll
    for (int h = 0; h < VW; h += 8) {
      uint4 qa[8], qb[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t r = base + int64_t(32 * (h + u) + lane) * 8;
        if (r < r1) {
          qa[u] = *reinterpret_cast<const uint4*>(F.p0 + (row0 + r) * 2);
          if constexpr (FastTraits<K>::load1) qb[u] = *reinterpret_cast<const uint4*>(F.p1 + (row0 + r) * 2);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t r = base + int64_t(32 * (h + u) + lane) * 8;
        if (r < r1) {
          float a[8], b[8], x[8];
          unpack8(qa[u], DT, a);
          if constexpr (FastTraits<K>::load1) unpack8(qb[u], DT, b);
          fast_apply<K>(F, a, b, none, x);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[h + u] = __fadd_rn(acc[h + u], x[j]);
        }
      }
    }
  }
  float s = 0.0f;
#pragma unroll
  for (int w = 0; w < VW; ++w) {
    float v = acc[w];
#pragma unroll
    for (int d = 16; d; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    s += v;
  }
  if (lane == 0) {
    if (t.parts == 1)
      finish_reduction(c, t, o, s, pre);
    else
      reinterpret_cast<float*>(c.ws)[t.scratch + o * t.parts + p] = s;
  }
}

// Column reduction item (256-column chunk, part p): virtual warp w sums rows
// r0 + w + 8 i (i = 0, 1, ...) of the lane's eight columns; then the eight
// virtual warps' sums are added in warp order.
template <int K, int DT>
__device__ __forceinline__ void bg_col_item(const Ctx& c, const Task& t, int item) {
  constexpr int VW = kThreads / 32;
  const int lane = threadIdx.x & 31;
  const int64_t ch = item / t.parts;
  const int p = item % t.parts;
  const int64_t Q = t.red_inner;
  const int64_t col0 = ch * 256 + lane * 8;
  const int64_t r0 = int64_t(p) * t.part_len;
  const int64_t r1 = min(t.red_outer, r0 + t.part_len);
  const Fast F = fast_params(c, t);
  float acc[VW][8], none[8];
#pragma unroll
  for (int w = 0; w < VW; ++w)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[w][j] = 0.0f;
  if (col0 < Q) {
    // four rows' vectors in flight at a time
    for (int64_t i0 = r0; i0 < r1; i0 += VW) {
#pragma unroll
      for (int h = 0; h < VW; h += 4) {
        uint4 qa[4], qb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (i0 + h + u < r1) {
            qa[u] = *reinterpret_cast<const uint4*>(F.p0 + ((i0 + h + u) * Q + col0) * 2);
            if constexpr (FastTraits<K>::load1) qb[u] = *reinterpret_cast<const uint4*>(F.p1 + ((i0 + h + u) * Q + col0) * 2);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (i0 + h + u < r1) {
            float a[8], b[8], x[8];
            unpack8(qa[u], DT, a);
            if constexpr (FastTraits<K>::load1) unpack8(qb[u], DT, b);
            fast_apply<K>(F, a, b, none, x);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[h + u][j] = __fadd_rn(acc[h + u][j], x[j]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < VW; ++w) s = __fadd_rn(s, acc[w][j]);
    const int64_t col = col0 + j;
    if (col < Q) {
      if (t.parts == 1)
        finish_reduction(c, t, col, s, post_operand(c, t, col));
      else
        reinterpret_cast<float*>(c.ws)[t.scratch + col * t.parts + p] = s;
    }
  }
}

// The kinds run beside the tiles: sums of a 16-bit operand (FK_L, a bias
// gradient) and of its squares (FK_L_SQUARE, a squared-error loss), all
// operand of the type t.bg says (the planner marks only those).
__device__ __noinline__ void fold_arrive(const Ctx c, const Task& t, int item);
__device__ __noinline__ void bg_item(const Ctx& c, const Task& t, int item) {
  const bool row = t.kind == T_REDUCE_ROW, bf = t.bg == TK_BF16;
  if (t.chain.fast == FK_L) {
    if (row)
      bf ? bg_row_item<FK_L, TK_BF16>(c, t, item) : bg_row_item<FK_L, TK_F16>(c, t, item);
    else
      bf ? bg_col_item<FK_L, TK_BF16>(c, t, item) : bg_col_item<FK_L, TK_F16>(c, t, item);
  } else {
    if (row)
      bf ? bg_row_item<FK_L_SQUARE, TK_BF16>(c, t, item) : bg_row_item<FK_L_SQUARE, TK_F16>(c, t, item);
    else
      bf ? bg_col_item<FK_L_SQUARE, TK_BF16>(c, t, item) : bg_col_item<FK_L_SQUARE, TK_F16>(c, t, item);
  }
  if (t.fold) fold_arrive(c, t, item);
}

// A folded final pass (Task::fold): after a warp has written part p of
// 256-column chunk ch, it counts the part; the warp that counts the chunk's
// last part sums the chunk's parts and applies the final's chain, output by
// output with the same additions in the same order as the final pass's
// threads (lane l takes outputs 256 ch + 32 v + l, v = 0..7).  The parts are
// read from L2: other blocks wrote them, each before a release of its count.
__device__ __noinline__ void fold_arrive(const Ctx c, const Task& t, int item) {
  const int lane = threadIdx.x & 31;
  const int ch = item / t.parts;
  __threadfence();
  __syncwarp();
  unsigned last = 0;
  if (lane == 0) last = atom_add_acq_rel(&c.hdr->fold[t.fold_ctr + ch], 1u) + 1u == unsigned(t.parts);
  last = __shfl_sync(0xffffffffu, last, 0);
  __syncwarp();
  if (!last) return;
  const Task& f = c.tasks[t.fold - 1];
  const float* part = reinterpret_cast<const float*>(c.ws) + f.scratch;
  for (int v = 0; v < kThreads / 32; ++v) {
    const int64_t o = int64_t(ch) * kThreads + v * 32 + lane;
    if (o >= f.red_outer) break;
    const float pre = post_operand(c, f, o);
    const float* q = part + o * f.parts;
    float acc = 0.0f;
    for (int q0 = 0; q0 < f.parts; q0 += 8) {
      float x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = q0 + u < f.parts ? __ldcg(q + q0 + u) : 0.0f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (q0 + u < f.parts) acc = __fadd_rn(acc, x[u]);
    }
    finish_reduction(c, f, o, acc, pre);
  }
}

// Warp 2 or 3: this block's `bg` items of the stage (item g of a bg task goes
// to block g mod grid; the block's items alternate between the two warps).
__device__ __noinline__ void run_bg_items(const Ctx& c, const Stage& st) {
  const int w = (threadIdx.x >> 5) - 2;
  int k = 0;
  for (int ti = st.task_begin; ti < st.task_end; ++ti) {
    const Task& t = c.tasks[ti];
    if (!t.bg) continue;
    for (int g = blockIdx.x; g < t.n_items; g += gridDim.x, ++k)
      if ((k & 1) == w) bg_item(c, t, g);
  }
}

// Run this block's tensor-core tiles of one stage; false after a wait timed out.
template <int PM>
__device__ bool run_tc_phase(const Ctx& c, const Stage& st, const CUtensorMap* maps, TcState& ts, int stage,
                             int* s_flag, long long* prof) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bool ok = true;
  if (warp == 0 && lane == 0) {
    const uint64_t r = tc_producer<PM>(c, st, maps, ts, ts.p_it);
    ts.p_it = uint32_t(r);
    ok = (r >> 32) != 0;
    if (prof) prof[2] = global_ns();
  } else if (warp == 1 && lane == 0) {
    uint32_t m_tile = ts.m_tile;
    const uint64_t r = tc_mma<PM>(c, st, ts, ts.m_it, &m_tile, prof);
    ts.m_it = uint32_t(r);
    ts.m_tile = m_tile;
    ok = (r >> 32) != 0;
    if (prof) prof[4] = global_ns();
  } else if (warp == 2 || warp == 3) {
    if (st.has_bg) run_bg_items(c, st);
  } else if (warp >= 4) {
    EpiRing er = ts.er;
    const uint64_t r = tc_epilogue<PM>(c, st, ts, ts.e_tile, prof, &er);
    ts.e_tile = uint32_t(r);
    ts.er = er;
    ok = (r >> 32) != 0;
    if (prof && threadIdx.x == 128) prof[6] = global_ns();
  }
  if (!ok) record_failure(c, TK_ERR_PIPELINE_TIMEOUT, stage);
  if (threadIdx.x == 0) *s_flag = 1;
  __syncthreads();
  if (!ok) *s_flag = 0;
  __syncthreads();
  return *s_flag != 0;
}

__device__ void run_item(const Ctx& c, const Task& t, int item, float* smem) {
  switch (t.kind) {
    case T_POINTWISE:
      if (t.vec == 8)
        run_pointwise<8>(c, t, item);
      else
        run_pointwise<1>(c, t, item);
      break;
    case T_GEMV:
      run_gemv(c, t, item);
      break;
    case T_SPLITK_FINAL:
      if (t.vec == 8)
        run_splitk_final<8>(c, t, item);
      else
        run_splitk_final<1>(c, t, item);
      break;
    case T_REDUCE_ROW:
      if (t.vec == 8)
        run_reduce_row<8>(c, t, item, smem);
      else
        run_reduce_row<1>(c, t, item, smem);
      break;
    case T_REDUCE_COL:
      if (t.vec == 8)
        if (t.pw_unroll == kPointwiseUnroll16) {
          switch (t.chain.fast) {
#define TK_CALL(k) run_reduce_col_bulk16<k>(c, t, item, smem)
            TK_FAST_L_CASES(TK_CALL)
#undef TK_CALL
            default: run_reduce_col<8>(c, t, item, smem); break;
          }
        } else {
          switch (t.chain.fast) {
#define TK_CALL(k) run_reduce_col_fast<k>(c, t, item, smem)
            TK_FAST_L_CASES(TK_CALL)
#undef TK_CALL
            default: run_reduce_col<8>(c, t, item, smem); break;
          }
        }
      else
        run_reduce_col<1>(c, t, item, smem);
      break;
    case T_REDUCE_FINAL:
      run_reduce_final(c, t, item, smem);
      break;
    case T_GEMM_SIMT:
      if (t.tile_m == 64)
        run_gemm_simt<64>(c, t, item, smem);
      else if (t.tile_m == 32)
        run_gemm_simt<32>(c, t, item, smem);
      else
        run_gemm_simt<16>(c, t, item, smem);
      break;
    default:
      break;
  }
}


__device__ __forceinline__ void copy_words(void* dst, const void* src, int bytes, int tid, int n) {
  uint64_t* d = static_cast<uint64_t*>(dst);
  const uint64_t* q = static_cast<const uint64_t*>(src);
  for (int i = tid; i < bytes / 8; i += n) d[i] = q[i];
}

// Copy stage s's tasks, instructions and refs into shared memory (threads
// first..kThreads-1 take part); ranges that do not fit stay in global memory.
__device__ __forceinline__ void stage_in(const Program* prog, int s, Stage* s_stage, Task* s_tasks, Instr* s_code,
                                         Ref* s_refs, int first) {
  if (int(threadIdx.x) < first) return;
  const int tid = threadIdx.x - first, n = kThreads - first;
  const Stage st = prog->stages[s];
  if (tid == 0) *s_stage = st;
  if (st.task_end - st.task_begin <= kStageTasks)
    copy_words(s_tasks, prog->tasks + st.task_begin, (st.task_end - st.task_begin) * int(sizeof(Task)), tid, n);
  if (st.code_hi - st.code_lo <= kStageCode)
    copy_words(s_code, prog->code + st.code_lo, (st.code_hi - st.code_lo) * int(sizeof(Instr)), tid, n);
  if (st.ref_hi - st.ref_lo <= kStageRefs)
    copy_words(s_refs, prog->refs + st.ref_lo, (st.ref_hi - st.ref_lo) * int(sizeof(Ref)), tid, n);
}

// PM: 0 one block per tile; a pair-tile launch (clusters of two blocks, every
// tensor-core GEMM on 256-row tiles) with 1 cta_group::2 MMAs and kPairStages
// ring slots, or 2 each block's own MMAs on B tiles shared by multicast.
template <int PM>
__device__ __forceinline__ void persistent_body(const Params& p, const CUtensorMap* maps) {
  constexpr bool PAIR = PM == 1, MC = PM == 2;
  constexpr int NS = PAIR ? kPairStages : kStages;
  __shared__ void* s_io[2 * kMaxIO];
  __shared__ Task s_tasks[kStageTasks];
  __shared__ __align__(16) Instr s_code[kStageCode];
  __shared__ __align__(16) Ref s_refs[kStageRefs];
  __shared__ Stage s_stage;
  __shared__ Prep s_prep[kThreads / 32];
  __shared__ __align__(8) uint64_t s_bar[2 * NS + 5];
  __shared__ __align__(8) uint64_t s_epi_bar[4 * kEpiMaxDepth];
  __shared__ __align__(8) uint64_t s_bulk_bar[kBulkMaxSlots];
  __shared__ uint32_t s_bulk_it;
  __shared__ __align__(8) uint64_t s_col_bar[kBulkMaxSlots];
  __shared__ uint32_t s_col_it;
  __shared__ uint32_t s_tmem;
  __shared__ int s_flag;
  extern __shared__ __align__(1024) unsigned char s_dyn[];
  const bool tc = maps != nullptr;
  // pair: the launch must have formed clusters of two (else no cluster or
  // pair operation runs and the kernel reports TK_ERR_PAIR_TMEM)
  const bool paired = PM != 0 && cluster_size() == 2;
  // scratch for reductions and CUDA-core GEMMs at the start of the dynamic
  // region; in a tensor-core launch it overlays the (then idle) ring
  float* s_work = reinterpret_cast<float*>(s_dyn + ((1024u - (smem_u32(s_dyn) & 1023u)) & 1023u));
  const int warp = threadIdx.x >> 5;
  const Program* prog = p.prog;
  const long long entry_ns = global_ns();
  for (int i = threadIdx.x; i < p.n_in; i += kThreads) s_io[i] = p.io[i];
  for (int i = threadIdx.x; i < p.n_out; i += kThreads) s_io[kMaxIO + i] = p.io[kMaxIO + i];
  stage_in(prog, 0, &s_stage, s_tasks, s_code, s_refs, 0);
  TcState ts{};
  if (tc) {
    ts.ring = (smem_u32(s_dyn) + 1023u) & ~1023u;
    ts.slot_bytes = uint32_t(p.ring_stage_bytes);
    ts.stg = ts.ring + uint32_t(NS) * ts.slot_bytes;
    ts.stg_warp_bytes = uint32_t(p.epi_warp_bytes);
    ts.full = smem_u32(&s_bar[0]);
    ts.empty = smem_u32(&s_bar[NS]);
    ts.acc_full = smem_u32(&s_bar[2 * NS]);
    ts.acc_empty = smem_u32(&s_bar[2 * NS + 2]);
    ts.drain = smem_u32(&s_bar[2 * NS + 4]);
    ts.epi_bar = smem_u32(&s_epi_bar[0]);
    ts.maps = maps;
    ts.er.task = -1;
    if (threadIdx.x == 0) {
      for (int i = 0; i < NS; ++i) {
        mbar_init(ts.full + 8 * i, 1);
        mbar_init(ts.empty + 8 * i, MC ? 2 : 1);  // shared B: both blocks' MMAs free a slot
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(ts.acc_full + 8 * i, 1);
        mbar_init(ts.acc_empty + 8 * i, PAIR ? 8 : 4);  // pair: both blocks' epilogue warps (leader's copy)
      }
      mbar_init(ts.drain, 1);
      for (int i = 0; i < 4 * kEpiMaxDepth; ++i) mbar_init(ts.epi_bar + 8 * i, 1);
      for (int i = 0; i < kBulkMaxSlots; ++i) {
        mbar_init(smem_u32(&s_bulk_bar[i]), 1);
        mbar_init(smem_u32(&s_col_bar[i]), kThreads);
      }
      s_bulk_it = 0;
      s_col_it = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (threadIdx.x == 0)
      for (int i = 0; i < p.n_maps; ++i)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps[i])) : "memory");
    if (warp == 1 && (PM == 0 || paired)) {
      // pair: one warp of each block of the pair allocates, together
      if constexpr (PAIR) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(p.tmem_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
      } else {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(p.tmem_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  // pair: neither block signals the other's mbarriers before both have
  // initialised them
  if (paired) cluster_sync();
  bool pair_ok = PM == 0 || paired;
  if (tc) {
    tc_fence_after();
    ts.tmem = s_tmem;
    ts.acc_cols = uint32_t(p.tmem_cols) / 2;
    // pair: an MMA of the pair writes the same TMEM columns in both blocks,
    // so both must have been given the same address
    if (PAIR && paired) {
      uint32_t other;
      asm volatile("ld.shared::cluster.u32 %0, [%1];"
                   : "=r"(other)
                   : "r"(cluster_addr(smem_u32(&s_tmem), cluster_rank() ^ 1u))
                   : "memory");
      pair_ok = other == ts.tmem;
    }
  }
  if (warp == 2) {
    // L2 prefetch of the op table and the inputs, spread over blocks and lanes
    const int n_pf = prog->n_prefetch;
    for (int g = blockIdx.x + gridDim.x * (threadIdx.x & 31); g < n_pf; g += 32 * gridDim.x) {
      const Prefetch f = prog->prefetch[g];
      const char* base = f.space == SP_TABLE ? reinterpret_cast<const char*>(prog)
                                              : static_cast<const char*>(s_io[f.space == SP_IN ? f.slot : kMaxIO + f.slot]);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + f.offset), "r"(uint32_t(f.bytes))
                   : "memory");
    }
  }
  Ctx c{nullptr, nullptr, nullptr, p.ws, reinterpret_cast<Header*>(p.ws), s_io, p.timeout_ns, s_prep};
  if (tc) {
    c.bulk = ts.ring + kBulkOffset;
    c.bulk_bar = smem_u32(&s_bulk_bar[0]);
    c.bulk_slots = max(0, min(kBulkMaxSlots, (NS * p.ring_stage_bytes - kBulkOffset) / kBulkSlotBytes));
    c.bulk_it = &s_bulk_it;
    c.col_bar = smem_u32(&s_col_bar[0]);
    c.col_it = &s_col_it;
  }
  long long* prof = p.prof ? p.prof + kProfStamps * int64_t(blockIdx.x) : nullptr;
  const int64_t prof_step = kProfStamps * int64_t(gridDim.x);
  if (!pair_ok && threadIdx.x == 0) record_failure(c, TK_ERR_PAIR_TMEM, 0);
  const int n_stages = pair_ok ? prog->n_stages : 0;
  if (prof) {
    // stamps a stage may leave unwritten read as 0
    if (threadIdx.x == 0) {
      for (int s = 0; s < n_stages; ++s)
        for (int k = 2; k < kProfStamps; ++k) prof[s * prof_step + k] = 0;
      prof[7] = entry_ns;
    }
    __syncthreads();
  }
  for (int s = 0; s < n_stages; ++s) {
    const Stage st = s_stage;
    c.stage = s;
    if (prof && threadIdx.x == 0) prof[s * prof_step] = global_ns();
    c.tasks = st.task_end - st.task_begin <= kStageTasks ? s_tasks - st.task_begin : prog->tasks;
    c.code = st.code_hi - st.code_lo <= kStageCode ? s_code - st.code_lo : prog->code;
    c.refs = st.ref_hi - st.ref_lo <= kStageRefs ? s_refs - st.ref_lo : prog->refs;
    if (tc && st.n_tc_items > 0 &&
        !run_tc_phase<PM>(c, st, maps, ts, s, &s_flag, prof ? prof + s * prof_step : nullptr))
      break;
    // the stage's other items after its tiles: blocks with one tile fewer
    // than the busiest (the first r blocks have one more: r = tiles mod grid,
    // or twice tiles mod pairs when tiles go to pairs of blocks) first take
    // up to light_items each, the rest go round-robin from block r on
    {
      const int G = gridDim.x, b = blockIdx.x, T = st.n_tc_items, n_rest = st.n_items - T;
      const int r = PM ? 2 * (T % (G / 2)) : T % G, n_light = r ? G - r : 0;
      const int extra = min(n_rest, n_light * st.light_items);
      // this block's first-round items j = b - r + k * n_light (k < n1), then
      // j = extra + (b - r) mod G + k' * G
      const int n1 = b >= r && extra > b - r ? (extra - (b - r) + n_light - 1) / n_light : 0;
      int ti = st.task_begin, base = 0;
      for (int k = 0;; ++k) {
        const int j = k < n1 ? b - r + k * n_light : extra + (b - r + G) % G + (k - n1) * G;
        if (j >= n_rest) break;
        const int g = T + j;
        while (ti < st.task_end && g >= base + c.tasks[ti].n_items) {
          base += c.tasks[ti].n_items;
          ++ti;
        }
        // (a bg task ran beside the tiles; without tiles it runs here)
        if (!(c.tasks[ti].bg && st.n_tc_items > 0 && tc)) run_item(c, c.tasks[ti], g - base, s_work);
      }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncthreads();
    if (prof && threadIdx.x == 0) prof[s * prof_step + 1] = global_ns();
    if (s + 1 == n_stages) break;
    if (threadIdx.x == 0) barrier_arrive(c);
    stage_in(prog, s + 1, &s_stage, s_tasks, s_code, s_refs, 32);
    if (threadIdx.x == 0) s_flag = barrier_wait(c, unsigned(s + 1) * gridDim.x, s) ? 1 : 0;
    __syncthreads();
    if (!s_flag) break;
  }
  __syncthreads();
  if (threadIdx.x == 0) kernel_exit(c);
  if (tc) {
    tc_fence_before();
    __syncthreads();
    // pair: no block leaves while the other may still signal its mbarriers;
    // both free the TMEM together
    if (paired) cluster_sync();
    tc_fence_after();
    if (warp == 1 && (PM == 0 || paired)) {
      if constexpr (PAIR)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(ts.tmem), "r"(p.tmem_cols));
      else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(ts.tmem), "r"(p.tmem_cols));
    }
  }
}

}  // namespace
}  // namespace tkk
