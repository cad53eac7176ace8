// The persistent training-step kernel for sm_103a (GB300).
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
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/tk.h"
#include "tk_device.h"
#include "tk_kernel.h"

namespace tkk {

using namespace tkd;

struct Ctx {
  const Program* prog;
  char* ws;
  Header* hdr;
  void* const* io;  // shared-memory copy of Params::io
  long long timeout_ns;
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

// 8 consecutive elements from a 16-byte aligned address.
__device__ __forceinline__ void load8(const char* p, int dt, int64_t i, float (&v)[8]) {
  if (dt == TK_F32) {
    const float4* q = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i);
    float4 x = q[0], y = q[1];
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
  } else {
    uint4 raw = *reinterpret_cast<const uint4*>(p + i * 2);
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
}

__device__ __forceinline__ void store8(char* p, int dt, int64_t i, const float (&v)[8]) {
  if (dt == TK_F32) {
    float4* q = reinterpret_cast<float4*>(reinterpret_cast<float*>(p) + i);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
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
    *reinterpret_cast<uint4*>(p + i * 2) = make_uint4(w[0], w[1], w[2], w[3]);
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

__device__ __forceinline__ void unravel(const Task& t, int64_t f, int64_t* crd) {
#pragma unroll
  for (int d = kMaxRank - 1; d >= 0; --d) {
    if (d < t.rank) {
      int64_t n = t.shape[d];
      crd[d] = f % n;
      f /= n;
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
      TK_GET(0) TK_GET(1) TK_GET(2) TK_GET(3) TK_GET(4) TK_GET(5)
#undef TK_GET
    }
  }
  __device__ __forceinline__ void set(int i, const float (&in)[V]) {
    switch (i) {
#define TK_SET(k)                                        \
  case k:                                                \
    _Pragma("unroll") for (int j = 0; j < V; ++j) r[k][j] = in[j]; \
    break;
      TK_SET(0) TK_SET(1) TK_SET(2) TK_SET(3) TK_SET(4) TK_SET(5)
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
  const Instr* code = c.prog->code + t.code_begin;
  const Ref* refs = c.prog->refs + t.ref_begin;
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

// ------------------------------------------------------------- barriers

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

// All blocks meet here; returns false if the kernel must stop.
__device__ bool grid_barrier(const Ctx& c, int stage, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    Header* h = c.hdr;
    unsigned gen = ld_acquire(&h->gen);
    unsigned arrived = atom_add_acq_rel(&h->count, 1u) + 1u;
    if (arrived == gridDim.x) {
      atomicExch(&h->count, 0u);
      st_release(&h->gen, gen + 1u);
    } else {
      long long t0 = global_ns();
      unsigned spins = 0;
      while (ld_acquire(&h->gen) == gen) {
        if ((++spins & 31u) == 0u) {
          if (*reinterpret_cast<volatile int*>(&h->abort)) {
            ok = 0;
            break;
          }
          if (global_ns() - t0 > c.timeout_ns) {
            record_failure(c, TK_ERR_BARRIER_TIMEOUT, stage);
            ok = 0;
            break;
          }
        }
      }
    }
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
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

__device__ __forceinline__ void finish_reduction(const Ctx& c, const Task& t, int64_t o, float acc) {
  float v = t.red_mean ? __fdiv_rn(acc, t.size_f) : acc;
  store1(space_ptr(c, t.out.space, t.out.slot), t.out.dtype, t.out.base + o, v);
}

// ------------------------------------------------------------- work items

template <int V>
__device__ void run_pointwise(const Ctx& c, const Task& t, int item) {
  int64_t i0 = (int64_t(item) * kThreads + threadIdx.x) * V;
  if (i0 >= t.numel) return;
  int64_t crd[kMaxRank];
  unravel(t, i0, crd);
  float v[V];
  vm_eval<V>(c, t, crd, nullptr, v);
  store_out<V>(c, t.out, i0, v);
}

template <int V>
__device__ void run_reduce_row(const Ctx& c, const Task& t, int item, float* red) {
  const int64_t o = item / t.parts;
  const int p = item % t.parts;
  const int64_t r0 = int64_t(p) * t.part_len;
  const int64_t r1 = min(t.red_inner, r0 + t.part_len);
  float acc = 0.0f;
  for (int64_t r = r0 + int64_t(threadIdx.x) * V; r < r1; r += int64_t(kThreads) * V) {
    int64_t crd[kMaxRank];
    unravel(t, o * t.red_inner + r, crd);
    float v[V];
    vm_eval<V>(c, t, crd, nullptr, v);
#pragma unroll
    for (int j = 0; j < V; ++j) acc = __fadd_rn(acc, v[j]);
  }
  acc = block_sum(acc, red);
  if (threadIdx.x == 0) {
    if (t.parts == 1)
      finish_reduction(c, t, o, acc);
    else
      reinterpret_cast<float*>(c.ws)[t.scratch + o * t.parts + p] = acc;
  }
}

template <int V>
__device__ void run_reduce_col(const Ctx& c, const Task& t, int item, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t ch = item / t.parts;
  const int p = item % t.parts;
  const int64_t Q = t.red_inner;
  const int64_t col0 = ch * 32 * V + lane * V;
  const int64_t r0 = int64_t(p) * t.part_len;
  const int64_t r1 = min(t.red_outer, r0 + t.part_len);
  float acc[V];
#pragma unroll
  for (int j = 0; j < V; ++j) acc[j] = 0.0f;
  if (col0 < Q) {
    for (int64_t r = r0 + warp; r < r1; r += kThreads / 32) {
      int64_t crd[kMaxRank];
      unravel(t, r * Q + col0, crd);
      float v[V];
      vm_eval<V>(c, t, crd, nullptr, v);
#pragma unroll
      for (int j = 0; j < V; ++j) acc[j] = __fadd_rn(acc[j], v[j]);
    }
  }
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
        finish_reduction(c, t, col, s);
      else
        reinterpret_cast<float*>(c.ws)[t.scratch + col * t.parts + p] = s;
    }
  }
  __syncthreads();
}

__device__ void run_reduce_final(const Ctx& c, const Task& t, int item, float* red) {
  const float* part = reinterpret_cast<const float*>(c.ws) + t.scratch;
  if (t.final_block) {
    const int64_t o = item;
    float acc = 0.0f;
    for (int q = threadIdx.x; q < t.parts; q += kThreads) acc = __fadd_rn(acc, part[o * t.parts + q]);
    acc = block_sum(acc, red);
    if (threadIdx.x == 0) finish_reduction(c, t, o, acc);
  } else {
    const int64_t o = int64_t(item) * kThreads + threadIdx.x;
    if (o >= t.red_outer) return;
    float acc = 0.0f;
    for (int q = 0; q < t.parts; ++q) acc = __fadd_rn(acc, part[o * t.parts + q]);
    finish_reduction(c, t, o, acc);
  }
}

// CUDA-core GEMM tile: TM x TM outputs, 16 x 16 threads, (TM/16)^2 each;
// float32 fmaf accumulation in k order, then the epilogue expression.
template <int TM>
__device__ void run_gemm_simt(const Ctx& c, const Task& t, int item, float* smem) {
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
        vm_eval<1>(c, t, crd, a1, v);
        store_out<1>(c, t.out, row * t.n + col, v);
      }
    }
  }
}

__device__ void run_item(const Ctx& c, const Task& t, int item, float* smem) {
  switch (t.kind) {
    case T_POINTWISE:
      if (t.vec == 8)
        run_pointwise<8>(c, t, item);
      else
        run_pointwise<1>(c, t, item);
      break;
    case T_REDUCE_ROW:
      if (t.vec == 8)
        run_reduce_row<8>(c, t, item, smem);
      else
        run_reduce_row<1>(c, t, item, smem);
      break;
    case T_REDUCE_COL:
      if (t.vec == 8)
        run_reduce_col<8>(c, t, item, smem);
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

constexpr int kSmemFloats = 2 * 16 * (64 + 4) > 8 * 256 ? 2 * 16 * (64 + 4) : 8 * 256;

__global__ void __launch_bounds__(kThreads, 1) tk_persistent(const __grid_constant__ Params p) {
  __shared__ void* s_io[2 * kMaxIO];
  __shared__ __align__(16) float s_work[kSmemFloats];
  __shared__ int s_flag;
  for (int i = threadIdx.x; i < 2 * kMaxIO; i += kThreads) s_io[i] = p.io[i];
  __syncthreads();
  Ctx c{p.prog, p.ws, reinterpret_cast<Header*>(p.ws), s_io, p.timeout_ns};
  const Program* prog = p.prog;
  const int n_stages = prog->n_stages;
  for (int s = 0; s < n_stages; ++s) {
    const Stage st = prog->stages[s];
    int ti = st.task_begin, base = 0;
    for (int g = blockIdx.x; g < st.n_items; g += gridDim.x) {
      while (ti < st.task_end && g >= base + prog->tasks[ti].n_items) {
        base += prog->tasks[ti].n_items;
        ++ti;
      }
      run_item(c, prog->tasks[ti], g - base, s_work);
    }
    if (s + 1 < n_stages && !grid_barrier(c, s, &s_flag)) return;
  }
}

}  // namespace tkk

// ------------------------------------------------------------ host side

cudaError_t tk_kernel_launch(const tkd::Params& params, int grid, size_t dyn_smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(tkd::kThreads);
  cfg.dynamicSmemBytes = dyn_smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tkk::tk_persistent, params);
}

cudaError_t tk_kernel_occupancy(int* blocks_per_sm, size_t dyn_smem) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, tkk::tk_persistent, tkd::kThreads, dyn_smem);
}

cudaError_t tk_kernel_attributes(cudaFuncAttributes* attr) {
  return cudaFuncGetAttributes(attr, tkk::tk_persistent);
}
