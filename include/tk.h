/*
 * tk.h -- C ABI of the GB300 persistent training-step kernel (libtk.so).
 *
 * One functional training step (forward addmm/relu, loss, explicit backward
 * mm/threshold_backward, bias column sums, in-place parameter update) is given
 * as a static op list in topological order.  tk_program_create plans it once
 * (op order, inlining of single-use pointwise values, GEMM epilogue chains,
 * workspace arena, grid-barrier placement) and uploads a device op table;
 * tk_run launches ONE cooperative persistent kernel that walks the op table
 * stage by stage with a grid-wide barrier between dependent stages.
 *
 * The statement of the problem follows trainkernel (pages "trainkernel 0.1.0 --
 * trainkernel/codegen.py" and "trainkernel/runtime.py"):
 *   - tensors are TensorSpec views (buffer, shape, element strides, element
 *     offset, dtype) -- codegen.py, `_Generator.read` / `coords`;
 *   - the op set is the pointwise set {add, sub, mul, div, neg, relu, pow,
 *     threshold_backward, full, cast}, mm/addmm and sum/mean -- codegen.py
 *     `_POINTWISE`, `emit_mm`, `emit_reduction`;
 *   - every op computes in float32 and rounds its result to its output dtype
 *     (round to nearest even) -- codegen.py `_round`, `store`;
 *   - `allocate` sizes a float32 workspace and binds in-place outputs to their
 *     inputs; `run_into` checks buffers and launches -- runtime.py
 *     `CompiledProgram.allocate` / `run_into` / `ExecutionBuffers`;
 *   - in-place outputs map an output slot to the input it overwrites --
 *     codegen.py `generate(..., inplace_outputs=...)`.
 *
 * Conventions for every entry point:
 *   - Device memory is owned by the caller (inputs, outputs, workspace).  The
 *     library owns the plan and its device op table.
 *   - Every pointer argument documented as "device" must be a device address on
 *     the program's device, 16-byte aligned when non-NULL.
 *   - `stream` is a cudaStream_t (CUstream) handle passed as void*; NULL means
 *     the legacy default stream.  Calls that take a stream are asynchronous.
 *   - A non-zero tk_status means nothing was launched; tk_last_error() then
 *     returns a "tk: ..." message (thread-local, valid until the next call).
 */
#ifndef TK_H
#define TK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TK_MAX_RANK 4
#define TK_MAX_OPERANDS 3
#define TK_MAX_IO 256

typedef enum {
  TK_OK = 0,
  TK_ERR_INVALID = 1,          /* malformed program, argument or buffer */
  TK_ERR_UNSUPPORTED = 2,      /* well-formed but outside the supported subset */
  TK_ERR_WORKSPACE = 3,        /* workspace missing or smaller than tk_allocate says */
  TK_ERR_ALIAS = 4,            /* outputs/workspace overlap inputs or each other */
  TK_ERR_CUDA = 5,             /* a CUDA runtime call failed */
  TK_ERR_DEVICE = 6,           /* no usable device (or a plan-only program was run) */
  TK_ERR_BARRIER_TIMEOUT = 7,  /* device status: a grid barrier wait ran out */
  TK_ERR_PIPELINE_TIMEOUT = 8, /* device status: a tensor-core pipeline wait ran out */
  TK_ERR_PAIR_TMEM = 9         /* device status: the two blocks of a pair-tile launch were given
                                  different tensor-memory addresses (no tile was run) */
} tk_status;

typedef enum { TK_F32 = 0, TK_F16 = 1, TK_BF16 = 2 } tk_dtype;

typedef enum {
  TK_OP_ADD = 0,                /* in0 + alpha*in1            (codegen.py point_expr) */
  TK_OP_SUB = 1,                /* in0 - alpha*in1 */
  TK_OP_MUL = 2,                /* in0 * in1 */
  TK_OP_DIV = 3,                /* in0 / in1 (IEEE) */
  TK_OP_NEG = 4,                /* -in0 */
  TK_OP_RELU = 5,               /* in0 < 0 ? 0 : in0 */
  TK_OP_POW = 6,                /* in0 ^ exponent (exponent: scalar in1, else attr) */
  TK_OP_THRESHOLD_BACKWARD = 7, /* in1 <= threshold ? 0 : in0 */
  TK_OP_FULL = 8,               /* the value attribute when given, else scalar in0, else 0 */
  TK_OP_CAST = 9,               /* in0, rounded to the output dtype */
  TK_OP_MM = 10,                /* in0[m,k] @ in1[k,n]        (codegen.py emit_mm) */
  TK_OP_ADDMM = 11,             /* alpha*(in1 @ in2) + beta*in0 (bias broadcast) */
  TK_OP_SUM = 12,               /* sum of in0 over dims       (codegen.py emit_reduction) */
  TK_OP_MEAN = 13               /* sum / float32(size); empty -> NaN */
} tk_op_kind;

/* A strided view of a buffer.  buffer_id names the buffer: a program input
 * defines one, an op output defines one.  shape/strides/offset count elements;
 * only the first `rank` entries are read.  An op's output view must be
 * contiguous with offset 0 (it is the buffer). */
typedef struct {
  int32_t buffer_id;
  int32_t rank;
  int64_t shape[TK_MAX_RANK];
  int64_t strides[TK_MAX_RANK];
  int64_t offset;
  int32_t dtype;               /* tk_dtype */
  int32_t reserved;
} tk_tensor_spec;

/* One operation.  Operand i is scalars[i] (a float32 literal once rounded) when
 * bit i of scalar_mask is set, else the view inputs[i].  Attributes the op does
 * not use are ignored.  Reductions: n_dims == -1 reduces every dim, otherwise
 * dims[0..n_dims) (negative dims count from the end). */
typedef struct {
  int32_t kind;                /* tk_op_kind */
  int32_t n_inputs;
  tk_tensor_spec inputs[TK_MAX_OPERANDS];
  double scalars[TK_MAX_OPERANDS];
  uint32_t scalar_mask;
  int32_t n_dims;
  int32_t dims[TK_MAX_RANK];
  tk_tensor_spec output;
  double alpha, beta, threshold, exponent, value;
  int32_t value_given;         /* 1: the value attribute is given; full then uses it over a scalar
                                  operand (codegen.py point_expr: attrs value, else inputs[0], else 0) */
  int32_t reserved;            /* 0 */
} tk_op;

/* A whole program.  inplace holds n_inplace pairs {output_slot, input_index}:
 * that output overwrites that input's storage (transactionally: every read of
 * the old value happens first). */
typedef struct {
  int32_t n_inputs;
  const tk_tensor_spec* inputs;
  int32_t n_outputs;
  const tk_tensor_spec* outputs;
  int32_t n_ops;
  const tk_op* ops;
  int32_t n_inplace;
  const int32_t* inplace;
} tk_program_desc;

/* Planner and launch options (codegen.py `generate` keyword knobs). */
typedef struct {
  int32_t blocks_per_sm;       /* upper bound on resident blocks per SM, 1..8 (default 1) */
  int32_t max_blocks;          /* cap on the grid; <= 0: none */
  int32_t fuse_pointwise;      /* inline single-use pointwise values (default 1) */
  int32_t fuse_epilogues;      /* fuse pointwise chains into GEMM epilogues (default 1) */
  int32_t inline_input_casts;  /* inline casts of program inputs (default 1) */
  int32_t tensor_cores;        /* 1: tcgen05 path for eligible bf16/fp16 GEMMs (default 1) */
  int32_t sm_count;            /* 0: query the device; > 0: SM count for a plan-only program */
  int32_t profile;             /* 1: record per-stage globaltimer stamps (see tk_profile_read) */
  double barrier_timeout_s;    /* limit of every in-kernel wait (default 2.0) */
  int32_t expr_forms;          /* expression evaluators the planner may pick: 0 all (compiled
                                  loops of fixed shapes, else generic chains, else instructions;
                                  default), 1 no compiled loops, 2 instructions only.  All give
                                  bit-identical results; 1 and 2 exist for testing. */
  int32_t split_k;             /* 1: split the K loop of under-filled tensor-core GEMMs over more
                                  SMs (partial sums, then a pass that adds them; default 1) */
  int32_t tile_n;              /* N width of every tensor-core tile: 0 (default) picks 64, 128,
                                  224 or 256 per GEMM from its tile count and the SM count; 64,
                                  128, 224 or 256 forces that width (224 only where the B operand
                                  is K-major, else 256; used by tests to reach each tile path) */
  int32_t epi_stage_bytes;     /* cap on the shared-memory staging bytes of each epilogue warp
                                  (0, default: what the SM has left beside the operand ring).
                                  Smaller caps give shallower staging rings; results are
                                  identical (used by tests to reach each staging layout) */
  int32_t cta_pairs;           /* every tensor-core GEMM on pairs of SMs: 256-row tiles, one
                                  cluster of two blocks per tile, each block loading its 128 rows
                                  of A and half of B's columns; 1: cta_group::2 MMAs over both
                                  blocks' shared memory; 2: each block runs its own 128-row MMAs,
                                  the B halves multicast to both blocks.  Programs with no
                                  tensor-core GEMM ignore it; 0 (default): one SM per 128-row tile */
  int32_t overlap_reductions;  /* 1 (default): a stage's compiled row and column reductions of
                                  16-bit operands run on the warps the tensor-core tiles leave idle,
                                  while the tiles run, where the planner estimates they fit in the
                                  tiles' time; 2: every such reduction (tests); 0: after the tiles.
                                  Results are identical */
} tk_options;

/* What the planner decided (codegen.py `GeneratedKernel` counters). */
typedef struct {
  int32_t materialized_ops;    /* scheduled ops (a fused GEMM+chain counts once) */
  int32_t inlined_ops;         /* pointwise values evaluated at their consumer */
  int32_t fused_epilogues;     /* GEMMs carrying a pointwise chain */
  int32_t tensor_core_ops;     /* GEMMs on the tcgen05 path */
  int32_t stages;              /* barrier-separated stages */
  int32_t grid_barriers;       /* = stages - 1 */
  int32_t direct_outputs;      /* outputs written in place by their producer */
  int32_t direct_state_commits;/* in-place outputs written directly (no commit copy) */
  int32_t max_work_items;      /* largest stage, in work items */
  int32_t grid_blocks;         /* blocks tk_run launches */
  int32_t output_copies;       /* end-of-kernel copies and transactional commits */
  int32_t split_reductions;    /* reductions done as partials + a final pass */
  int64_t workspace_elements;  /* float32 elements tk_allocate reports */
  int64_t arena_elements;      /* of which: intermediate-value arena */
  int32_t compiled_tasks;      /* tasks whose expression runs as a compiled loop of a fixed shape */
  int32_t chain_tasks;         /* tasks evaluating a generic linear chain (the rest use instructions) */
  int32_t tasks;               /* device tasks (see tk_plan_task) */
  int32_t tma_descriptors;     /* TMA descriptors a launch passes (GEMM operand tiles, epilogue chunks) */
  int32_t cta_pairs;           /* 1 or 2: a pair-tile launch (clusters of two blocks; see tk_options) */
} tk_plan_stats;

/* One device task of a plan: a scheduled op (with whatever the planner fused
 * into its expression), one half of a split reduction, or an end-of-kernel
 * output copy.  Tasks are listed stage by stage. */
typedef struct {
  int32_t stage;               /* barrier-separated stage the task runs in */
  int32_t kind;                /* 0 pointwise, 1 row reduction, 2 column reduction, 3 partials sum,
                                  4 CUDA-core GEMM, 5 tensor-core GEMM, 6 split-K sum + epilogue,
                                  7 one-row GEMM (batch 1) */
  int32_t op_index;            /* index into tk_program_desc.ops; -1 for an output copy or commit */
  int32_t n_items;             /* work items (GEMM tiles, element blocks, reduction outputs x parts) */
  int32_t form;                /* expression evaluator: 0 instructions, 1 generic chain, 2 compiled loop */
  int32_t compiled_shape;      /* which compiled loop (1..11) when form == 2, else 0 */
  int32_t m, n, k;             /* GEMM extents (0 otherwise) */
  int32_t tile_m, tile_n;      /* GEMM tile (0 otherwise) */
  int32_t parts;               /* reduction parts (1 = not split) */
  int32_t staged_epilogue;     /* tensor-core GEMM whose epilogue moves tiles through shared memory */
  int32_t side_output;         /* GEMM that also writes a second value (a side output) from its tile */
  int32_t staged_depth;        /* staged epilogue: 32-column chunks in flight per epilogue warp
                                  (2, 4 or 8; +16 when a side output has buffers of its own); 0 */
  int32_t beside_tiles;        /* reduction run while the stage's tensor-core tiles run */
  int32_t folded;              /* partials sum run in the stage of its partials, by the warp that
                                  adds a 256-column chunk's last part (n_items 0) */
  int64_t numel;               /* elements of the task's index space */
} tk_task_info;

typedef struct tk_program tk_program;

/* Fill *opt with the defaults above. */
void tk_options_default(tk_options* opt);

/* Validate and plan `desc` for `device` (a CUDA ordinal; -1 = plan only: no
 * CUDA call is made and tk_run refuses the program).  `opt` may be NULL.  The
 * descriptor is copied; the caller may free it on return.  On success *out owns
 * the plan and must be released with tk_program_destroy. */
tk_status tk_program_create(const tk_program_desc* desc, const tk_options* opt, int device,
                            tk_program** out);

/* Free a program and its device op table (NULL is ignored).  No run using it
 * may still be pending. */
void tk_program_destroy(tk_program* program);

/* Size of the float32 workspace tk_run needs, in elements (>= 1).  Sizing
 * only: the caller allocates (runtime.py `allocate`). */
tk_status tk_allocate(const tk_program* program, size_t* workspace_elements);

/* Zero the workspace header (barrier counter and status word) on `stream`.
 * Required once for each new workspace and again after a run whose device
 * status was not TK_OK; every successful run leaves the header ready for the
 * next one. */
tk_status tk_workspace_init(const tk_program* program, float* workspace, size_t workspace_elements,
                            void* stream);

/* Launch one step on `stream`.  inputs[i] / outputs[j] are device base
 * addresses of the program's inputs / outputs (element (c) of a view lives at
 * base + offset + sum(c*stride)).  An in-place output must be given exactly its
 * input's pointer; otherwise outputs must not overlap each other, the
 * workspace or any input, and the workspace must not overlap an input
 * (runtime.py `run_into`).  workspace: device, >= tk_allocate elements,
 * header initialised by tk_workspace_init.  Asynchronous; errors found on the
 * host return before anything is launched. */
tk_status tk_run(tk_program* program, const void* const* inputs, int32_t n_inputs,
                 void* const* outputs, int32_t n_outputs, float* workspace,
                 size_t workspace_elements, void* stream);

/* Synchronise `stream` and read the device status word a run left in the
 * workspace header: TK_OK, TK_ERR_BARRIER_TIMEOUT or TK_ERR_PIPELINE_TIMEOUT,
 * with the stage where the wait gave up in *stage (may be NULL). */
tk_status tk_run_status(const tk_program* program, const float* workspace, void* stream,
                        int32_t* device_status, int32_t* stage);

/* Kernel resources (codegen.py `resource_usage`): out[0] registers per thread,
 * out[1] local bytes per thread, out[2] shared bytes per block (static +
 * dynamic), out[3] resident blocks per SM. */
tk_status tk_resource_usage(const tk_program* program, int64_t out[4]);

/* Per-stage timing of the last run of a program created with profile = 1.
 * Synchronises `stream`, then copies stages * grid_blocks groups of 9
 * %globaltimer stamps (ns) into stamps[(s*grid+b)*9 + i]: i = 0 block b starts
 * stage s, 1 it reaches the barrier after it, 2 its TMA producer is done,
 * 3 its first operand tile has landed, 4 its MMA issue is done, 5 its first
 * accumulator is ready, 6 its epilogue is done (its stores complete), 8 its
 * epilogue has issued its last store (2-6 and 8 are 0 when the block has no
 * tensor-core tile in that stage), 7 kernel entry (stage 0 only).
 * n_stamps must be >= 9 * stages * grid_blocks (see tk_plan_stats). */
tk_status tk_profile_read(const tk_program* program, const float* workspace, void* stream, int64_t* stamps,
                          size_t n_stamps);

/* Planner decisions for tests and reports. */
tk_status tk_plan_stats_get(const tk_program* program, tk_plan_stats* stats);

/* Task `index` (0 <= index < stats.tasks) of the plan; TK_ERR_INVALID if out of
 * range.  Plan-only programs (device -1) answer too. */
tk_status tk_plan_task(const tk_program* program, int32_t index, tk_task_info* info);

/* ---- Built-in workspace (no allocation) ---------------------------------
 * The pages this library follows have no counterpart for this entry point.
 *
 * tk_run_static runs one step exactly like tk_run, but its workspace is an
 * array compiled into this library instead of memory the caller allocates.
 * It is for callers that cannot allocate device memory where they run a step:
 * code inside a CUDA stream capture that must not add allocation calls,
 * runtimes whose device memory is entirely reserved by another allocator, and
 * embedders that only receive input/output pointers from a framework that
 * owns every allocation.  The caller still passes inputs and outputs (same
 * rules as tk_run, including in-place outputs bound to their inputs).
 *
 * Limits and behaviour:
 *   - the array holds TK_STATIC_WORKSPACE_ELEMENTS float32 elements (8 MiB);
 *     a program whose tk_allocate size is larger is rejected with
 *     TK_ERR_WORKSPACE and a message naming both sizes -- use tk_run then;
 *   - every GPU on which this library's device code is loaded keeps the 8 MiB
 *     array until the process exits;
 *   - the first call for a program's device performs set-up: it looks up the
 *     array's device address with that device current (which also makes the
 *     CUDA runtime load this library's device code there).  Make that first
 *     call before any stream capture.  The address is kept with the device's
 *     context; after a device reset the next call looks it up again (so make
 *     that call outside a capture too);
 *   - every call shares the one array, which keeps the previous call's
 *     contents; each call clears the header (barrier counter, status word)
 *     with an asynchronous memset on `stream` before launching;
 *   - calls that can overlap on the GPU (different streams, or different
 *     programs on the same device without ordering) race on the array: order
 *     them on one stream;
 *   - nothing is allocated: no cudaMalloc/cudaFree or allocating library call;
 *   - tk_run_status and tk_profile_read do not apply (no workspace pointer is
 *     exposed to the caller). */
#define TK_STATIC_WORKSPACE_ELEMENTS 2097152

tk_status tk_run_static(tk_program* program, const void* const* inputs, int32_t n_inputs,
                        void* const* outputs, int32_t n_outputs, void* stream);

/* ---- Steps fed from host memory ------------------------------------------
 * The pages time steps on batches already resident on the GPU; a training
 * loop fed by a host-side loader also moves each batch to the device.  This
 * entry point keeps that copy off the critical path.
 *
 * tk_run_host enqueues n_steps steps, each exactly like tk_run, where the
 * batch inputs of step s are copied from host memory first and chosen outputs
 * of step s are copied to host memory after it.  The host-to-device copies run
 * on a second stream the program owns, into two device buffers per batch
 * input used alternately (step s reads buffer s mod 2), so the copy of step
 * s+1's batch overlaps step s; step s waits for its own copy, and the copy
 * into a buffer waits for the step that last read it.
 *
 *   batch[b], b < n_batch: the index of the b-th batch input.  A batch input
 *     is not the target of an in-place output.  Its two device buffers are
 *     inputs[batch[b]] (even steps) and batch_alt[b] (odd steps): each holds
 *     the input's bytes (its tk_run extent), is 16-byte aligned and overlaps
 *     no other buffer of the call.
 *   host_batches[s * n_batch + b]: host address of step s's value of batch
 *     input b, the same bytes as the device buffer.  Page-locked memory lets
 *     the copy overlap the previous step; pageable memory also works, without
 *     the overlap.
 *   results[r], r < n_results: an output index; after step s the output's
 *     bytes are copied to host_results[s * n_results + r] (on `stream`).
 *   Every other argument as tk_run; in-place outputs carry the state from
 *   step to step.
 *
 * Ownership: the caller owns every buffer; the program owns the copy stream
 * and its events (released by tk_program_destroy).  Asynchronous on `stream`:
 * the call returns once everything is enqueued, and the host buffers must
 * stay valid and host_batches unchanged until `stream` has completed.  The
 * copies into the first buffer wait for the work enqueued on `stream` before
 * the call.  Errors found on the host (counts, NULL or misaligned pointers,
 * aliasing, a batch input that is an in-place target) return before anything
 * is enqueued; a CUDA error part-way returns TK_ERR_CUDA with earlier steps
 * enqueued. */
tk_status tk_run_host(tk_program* program, int32_t n_steps, const void* const* inputs, int32_t n_inputs,
                      void* const* outputs, int32_t n_outputs, const int32_t* batch, int32_t n_batch,
                      void* const* batch_alt, const void* const* host_batches, const int32_t* results,
                      int32_t n_results, void* const* host_results, float* workspace,
                      size_t workspace_elements, void* stream);

/* Message of the last failing call on this thread ("" if none). */
const char* tk_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TK_H */
