// Device op table: the plan as the persistent kernel reads it.
//
// The host planner lowers every scheduled operation into a Task (a kind, an
// index space, a small expression program and operand references) and groups
// tasks into Stages; a grid barrier separates consecutive stages.  Each task
// is cut into independent work items that blocks take round-robin.
//
// This header is plain data shared by planner.cpp and the kernel (megakernel.cuh).
#pragma once

#include <stdint.h>

namespace tkd {

constexpr int kThreads = 256;      // threads per block (8 warps)
constexpr int kMaxRank = 4;
constexpr int kVmRegs = 4;         // expression registers per element
constexpr int kPointwiseUnroll = 4; // 8-element vectors per thread in a pointwise item
constexpr int kPointwiseUnroll16 = 8; // the same for compiled loops over 16-bit values only
constexpr int kHeaderUnits = 64;   // workspace header: 64 floats = 256 bytes
constexpr int kMaxIO = 256;        // program inputs (and outputs) per launch

// tcgen05 tile path: a 128 x BN output tile (BN = 64, 128 or 256) accumulates
// in TMEM over K blocks of 64 bf16/fp16 elements (one 128-byte swizzle row)
// staged by TMA through a kStages-deep shared-memory ring.
constexpr int kTileM = 128;
constexpr int kTileK = 64;
constexpr int kMaxTileN = 256;
constexpr int kStages = 4;
// Pair-tile launches (clusters of two blocks, 256-row tiles of cta_group::2
// MMAs) stage half of B per block: 16 KB of A + 16 KB of B per slot at
// 256-wide tiles, so six slots fit where four did.
constexpr int kPairStages = 6;
constexpr int kStageBytesA = kTileM * kTileK * 2;       // 16 KB
constexpr int kStageBytesB = kMaxTileN * kTileK * 2;    // 32 KB
// Dynamic shared memory of a tensor-core launch: 1 KB alignment slack, the
// TMA ring, then each epilogue warp's staging buffers.  The planner keeps the
// total within kDynSmemBudget (the 227 KB per-block limit minus the kernel's
// static shared memory, with margin).
constexpr int kDynSmemBudget = 211 * 1024;
// Scratch floats for reductions and CUDA-core GEMM tiles; at the start of the
// dynamic region (in a tensor-core launch it overlays the ring, which is idle
// outside the tensor-core phase of a stage).
constexpr int kWorkFloats = 2 * 16 * (64 + 4) > 8 * 256 ? 2 * 16 * (64 + 4) : 8 * 256;
// Epilogue staging: a 32-row x 32-column chunk of 16-bit values (64-byte rows).
// Long 16-bit reductions in a tensor-core launch stream their operands
// through the (then idle) TMA ring with bulk copies: slots of kBulkSlotBytes
// from kBulkOffset on (the first bytes hold the reduction scratch).
constexpr int kBulkOffset = 16 * 1024;
constexpr int kBulkSlotBytes = 16 * 1024;
constexpr int kBulkMaxSlots = 12;
constexpr int kEpiBufBytes = 32 * 64;
constexpr int kEpiMaxDepth = 8;                         // chunk buffers (and mbarriers) per epilogue warp
constexpr int kBcastBytes = kMaxTileN * 2;   // one 16-bit row of a tile
constexpr int kTmemCols = 2 * kMaxTileN;                // double-buffered accumulator (at most)
constexpr int kMaxMaps = 192;                           // TMA descriptors per launch

// Where a referenced tensor lives.
enum Space : int32_t { SP_IN = 0, SP_OUT = 1, SP_WS = 2 };

// How V consecutive index-space elements map to memory.
enum VMode : int32_t {
  VM_GATHER = 0,   // per-element address
  VM_CONTIG = 1,   // unit stride along the innermost index dim, vector-aligned
  VM_BCAST = 2     // stride 0 along the innermost index dim
};

// A tensor operand seen from a task's index space: element (c) is at
// base + sum_d c[d] * stride[d] in units of its dtype.
struct Ref {
  int32_t space, slot, dtype, vmode;
  int64_t base;
  int64_t stride[kMaxRank];
};

// Expression instructions; every result is rounded to `round` (a tk_dtype).
enum Opcode : uint8_t {
  OP_LOAD = 0,    // dst <- ref[ref]
  OP_CONST = 1,   // dst <- imm
  OP_ACC = 2,     // dst <- value supplied by the task (GEMM accumulator)
  OP_MOV = 3,     // dst <- a
  OP_ADD = 4,     // dst <- a + fl(imm * b)
  OP_SUB = 5,     // dst <- a - fl(imm * b)
  OP_MUL = 6,     // dst <- a * b
  OP_DIV = 7,     // dst <- a / b
  OP_NEG = 8,     // dst <- -a
  OP_RELU = 9,    // dst <- a < 0 ? 0 : a
  OP_SQUARE = 10, // dst <- a * a
  OP_POW = 11,    // dst <- powf(a, imm)
  OP_THRESH = 12  // dst <- b <= imm ? 0 : a
};

struct Instr {
  uint8_t op, dst, a, b;
  uint8_t round;
  uint8_t pad[3];
  float imm;
  int32_t ref;
};

// Linear-chain form of an expression, evaluated by compiled code instead of
// the instruction loop: a start value (the GEMM accumulator through the addmm
// formula, a load, or a constant), then up to kChainSteps ops, each combining
// the running value with nothing, a loaded operand or a constant.  At most two
// operand loads per element, which the kernel issues before any arithmetic.
constexpr int kChainSteps = 4;

enum ChainStart : int32_t { CH_ACC = 0, CH_LOAD = 1, CH_CONST = 2 };
enum ChainExt : uint8_t { EXT_NONE = 0, EXT_LOAD0 = 1, EXT_LOAD1 = 2, EXT_CONST = 3 };
enum AddmmMode : int32_t { AM_ACC = 0, AM_FULL = 1, AM_ZERO = 2, AM_ALPHA = 3, AM_BETA = 4, AM_SUM = 5 };

struct ChainStep {
  uint8_t op;       // Opcode (OP_ADD ... OP_THRESH, OP_MOV for a cast)
  uint8_t round;    // tk_dtype of the result
  uint8_t ext;      // ChainExt
  uint8_t second;   // 1: the running value is the op's second operand
  uint8_t ext_mul;  // 1: a loaded operand is first scaled: round(load * cval, ext_round)
  uint8_t ext_round;
  uint8_t pad[2];
  float imm;        // alpha (add/sub), threshold, exponent
  float cval;       // constant operand (EXT_CONST), or the scale of a loaded one
};

// Chains of these shapes run as compiled loops with their parameters hoisted
// out of the element loop (no per-element decoding).  E_*: GEMM epilogues on
// a [M,N] tile, operands contiguous along N; L_*: a load of operand slot 0
// addressed by the flat index, then the listed steps.
enum FastKind : int32_t {
  FK_NONE = 0,
  FK_E_ACC = 1,          // round(acc)
  FK_E_BIAS = 2,         // round(acc + l0)
  FK_E_BIAS_RELU = 3,    // round(relu(round(acc + l0)))
  FK_E_BIAS_AXPY = 4,    // round(round(acc + l0) +/- a*l1)
  FK_E_ACC_THRESH = 5,   // round(l0 <= a ? 0 : round(acc))
  FK_L = 6,              // l0
  FK_L_MOV = 7,          // round(l0)
  FK_L_SQUARE = 8,       // round(l0 * l0)
  FK_L_SCALE = 9,        // round(l0 * c)
  FK_L_AXPY = 10,        // round(l0 +/- a*l1)
  FK_L_SCALE_AXPY = 11,  // round(round(l0 * c) +/- a*l1)
  FK_E_UPDATE = 12,      // round(l0 +/- a*round(acc))   (SGD step in a weight-gradient epilogue)
  FK_E_MOMENTUM = 13     // round(round(l0*c) + a*round(acc))   (momentum buffer update)
};

struct Chain {
  int32_t valid;
  int32_t fast;          // FastKind
  int32_t n_loads;
  int32_t load_ref[2];   // task-relative refs of the two load slots
  int32_t start;         // ChainStart; CH_LOAD reads slot 0
  float start_const;
  int32_t bias;          // addmm bias: -1 none, 0/1 load slot, 2 constant
  float bias_const;
  float alpha, beta;
  int32_t addmm_mode;    // AddmmMode
  int32_t round0;        // dtype of the start value
  int32_t n_steps;
  ChainStep steps[kChainSteps];
};

enum TaskKind : int32_t {
  T_POINTWISE = 0,     // out[i] = expr(i)
  T_REDUCE_ROW = 1,    // reduce the innermost index dims; item = (output, part)
  T_REDUCE_COL = 2,    // reduce the outer index dims; item = (column chunk, part)
  T_REDUCE_FINAL = 3,  // sum the partials of a split reduction
  T_GEMM_SIMT = 4,     // CUDA-core tiled GEMM + epilogue expression
  T_GEMM_TC = 5,       // tcgen05 GEMM + epilogue expression
  T_SPLITK_FINAL = 6,  // sum of a split-K GEMM's partial accumulators + its epilogue
  T_GEMV = 7           // one-row GEMM (batch 1) with K-contiguous B: a warp per output
};

struct alignas(16) Task {
  int32_t kind;
  int32_t n_items;
  int32_t op_index;          // program op this task computes (-1: an output copy or commit)
  int32_t stage;             // stage the task runs in
  int32_t rank;              // index-space rank (0..4)
  int32_t vec;               // elements per thread-vector: 8 or 1
  int64_t shape[kMaxRank];   // index space
  int64_t numel;
  int32_t code_begin, code_len;
  int32_t ref_begin, n_refs;
  Chain chain;               // used instead of the instructions when valid
  Ref out;                   // contiguous output, addressed by flat output index
  // reductions
  int32_t red_mean;          // 1: divide by size_f
  int32_t parts;             // > 1: partials then a T_REDUCE_FINAL task
  int64_t red_outer;         // ROW: outputs;      COL: reduced rows
  int64_t red_inner;         // ROW: reduced size; COL: outputs (columns)
  int64_t part_len;          // ROW: elements per part; COL: rows per part
  int64_t scratch;           // float offset of the partials in the workspace
  float size_f;              // float32(reduced size)
  int32_t final_block;       // FINAL: 1 block per output (else 1 thread per output)
  // GEMM (A[m,k] strides: a.stride[0], a.stride[1]; B[k,n]: b.stride[0], b.stride[1])
  int32_t m, n, k;
  int32_t tile_m, tile_n, tiles_n;
  int32_t a_kcontig, b_ncontig;
  Ref a, b;
  // tcgen05 path
  int32_t tma_a, tma_b;
  uint32_t idesc;
  int32_t a_mn_major, b_mn_major;  // 0 K-major; 1 MN-major, 64-wide boxes; 2 MN-major, one box of slabs
  int32_t k_blocks;
  // Reductions: a pointwise chain applied to each finished output (e.g. the
  // SGD step of a bias right after its gradient's column sum).  Its start is
  // the reduced value (after the mean division) rounded to round0; its loads
  // are indexed by the output's coordinates in post_shape.
  Chain post;
  int64_t post_shape[kMaxRank];
  int32_t post_rank;
  // GEMMs and reductions: a side output, one more pointwise op on the stored
  // (rounded) final value, written to out2 (same shape, contiguous) from the
  // same tile.  side.ext: EXT_NONE / EXT_CONST (x*c, -x, a cast), or
  // EXT_LOAD1: an add/sub with the operand side_ld (contiguous, the output's
  // shape) read at the output's flat index; side.second as in a chain step.
  int32_t has_side;
  ChainStep side;
  Ref out2;
  Ref side_ld;
  // Staged epilogue (compiled GEMM epilogues with 16-bit output): bit s set =
  // load slot s is read per row and copied through shared memory; bit 2 =
  // the staged path is on; bit 3 = the side output's operand (side_ld) is
  // copied through shared memory too; bit 4 = a unary side output has chunk
  // buffers of its own.  0 = operands and output accessed directly.
  // epi_depth: chunk buffers per operand in each epilogue warp's ring
  // (2, 4 or 8; at most the tile's 32-column chunks); epi_dtype: the one
  // 16-bit type of all the staged epilogue's operands, roundings and outputs.
  int32_t epi_stage;
  int32_t epi_depth;
  int32_t epi_dtype;
  // TMA descriptors of a staged epilogue's 32 x 32 chunks (64-byte swizzle,
  // the staging layout): the output, the side output, the per-row operands
  // of load slots 0 and 1 and the loaded side's operand (-1: none).
  int32_t tma_out, tma_out2, tma_ld0, tma_ld1, tma_sd;
  int32_t pw_unroll;         // pointwise items: vectors per thread (kPointwiseUnroll or kPointwiseUnroll16)
  // Split-K (under-filled tensor-core GEMMs): item = tile * k_splits + split;
  // split s covers k blocks [s * kb_split, (s + 1) * kb_split) and writes its
  // float32 accumulator to scratch + s * m * n; the T_SPLITK_FINAL task sums
  // the splits in order and applies the epilogue.
  int32_t k_splits;
  int32_t kb_split;
  // A reduction run by warps 2 and 3 while the stage's tensor-core tiles run
  // (same additions in the same order as after the tiles): the 16-bit type
  // of its operand (TK_BF16 or TK_F16); 0: after the tiles.
  int32_t bg;
  // A split column reduction run beside the tiles whose final pass runs in
  // the same stage: fold = 1 + the index of that T_REDUCE_FINAL task (which
  // has folded = 1 and no items of its own), 0: none.  The warp that adds
  // the last part of a 256-column chunk (counter fold_ctr + chunk of the
  // workspace header) sums the chunk's parts and applies the final's chain.
  int32_t fold;
  int32_t fold_ctr;
  int32_t folded;
};

struct Stage {
  int32_t task_begin, task_end;
  int32_t n_items;           // all items of the stage (tensor-core tiles first)
  int32_t n_tc_items;
  int32_t code_lo, code_hi;  // instructions the stage's tasks use
  int32_t ref_lo, ref_hi;    // operand refs the stage's tasks use
  // Other items a block with one tensor-core tile fewer than the busiest
  // blocks takes before the rest are dealt round-robin over all blocks (the
  // planner's estimate of one tile's time in items of the stage; 0: plain
  // round-robin after the tiles).
  int32_t light_items;
  int32_t has_bg;            // some task runs beside the tiles (Task::bg)
};

// A stage whose descriptors fit these bounds is copied into shared memory
// while the previous grid barrier completes.
constexpr int kStageTasks = 6;
constexpr int kStageCode = 96;
constexpr int kStageRefs = 48;

// A byte range the kernel asks L2 to fetch at entry, so that the first reads
// of program inputs and of the op table in later stages hit L2.  `space` is a
// Space or SP_TABLE (the op table itself); offset and bytes are multiples of 16.
constexpr int32_t SP_TABLE = 3;
constexpr int64_t kPrefetchPiece = 64 * 1024;            // bytes per prefetch instruction
constexpr int64_t kPrefetchInputBudget = 48ll << 20;     // inputs larger in total are not prefetched

struct Prefetch {
  int32_t space, slot;
  int64_t offset, bytes;
};

struct Program {
  int32_t n_stages, n_tasks, n_code, n_refs;
  const Stage* stages;
  const Task* tasks;
  const Instr* code;
  const Ref* refs;
  int32_t n_prefetch, pad;
  const Prefetch* prefetch;
};

// Workspace header (offset 0, 256 bytes).  `count` only grows during a run
// (barrier j completes when it reaches (j+1) * gridDim.x); the last block to
// leave the kernel sets `count` and `exits` back to 0, so a run that
// completes leaves the header ready for the next run.
struct Header {
  unsigned int count;   // barrier arrivals in this run
  unsigned int exits;   // blocks that have left the kernel
  int status;           // 0, or the tk_status of the first failure
  int stage;            // stage of the first failure
  int abort;            // nonzero once any block gives up
  // parts added so far per 256-column chunk of the split reductions whose
  // final pass is folded into their own stage (Task::fold_ctr); zero between
  // runs (the last block to leave clears them)
  unsigned int fold[59];
};
constexpr int kFoldCounters = 59;
static_assert(sizeof(Header) == kHeaderUnits * 4, "the workspace header is kHeaderUnits floats");

// Kernel arguments: io[i] is input i, io[kMaxIO + j] is output j.
// Profile stamps per (stage, block): 0 stage begin, 1 barrier arrival,
// 2 producer done, 3 first operand tile ready, 4 MMA issue done, 5 first
// accumulator ready, 6 epilogue done, 7 kernel entry (stage 0 only), 8 the
// epilogue's last store issued.
constexpr int kProfStamps = 9;

struct Params {
  const Program* prog;
  char* ws;
  long long timeout_ns;
  long long* prof;      // optional stamps, [stage][block][kProfStamps]
  int n_in, n_out, n_maps;
  int ring_stage_bytes; // bytes per TMA ring slot (A tile + widest B tile)
  int tmem_cols;        // TMEM columns allocated: two accumulators of the widest tile (a power of 2)
  int epi_warp_bytes;   // staging bytes per epilogue warp (after the ring)
  void* io[2 * kMaxIO];
};

}  // namespace tkd
