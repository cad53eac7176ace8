"""ctypes binding of libtk's C ABI (declared in include/tk.h).

Functions keep the C names; this module only marshals arguments.  Every step
of the training step runs in the CUDA kernel behind ``tk_run``; nothing here
computes.  Loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .ir import Program, TensorSpec

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libtk.so")
_lock = threading.Lock()
_lib = None

MAX_RANK = 4
DTYPE = {"float32": 0, "float16": 1, "bfloat16": 2}
OP_KIND = {"add": 0, "sub": 1, "mul": 2, "div": 3, "neg": 4, "relu": 5, "pow": 6,
           "threshold_backward": 7, "full": 8, "cast": 9, "mm": 10, "addmm": 11, "sum": 12, "mean": 13}
STATUS = {0: "TK_OK", 1: "TK_ERR_INVALID", 2: "TK_ERR_UNSUPPORTED", 3: "TK_ERR_WORKSPACE", 4: "TK_ERR_ALIAS",
          5: "TK_ERR_CUDA", 6: "TK_ERR_DEVICE", 7: "TK_ERR_BARRIER_TIMEOUT", 8: "TK_ERR_PIPELINE_TIMEOUT",
          9: "TK_ERR_PAIR_TMEM"}


class tk_tensor_spec(ctypes.Structure):
    _fields_ = [("buffer_id", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("shape", ctypes.c_int64 * MAX_RANK), ("strides", ctypes.c_int64 * MAX_RANK),
                ("offset", ctypes.c_int64), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class tk_op(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("n_inputs", ctypes.c_int32),
                ("inputs", tk_tensor_spec * 3), ("scalars", ctypes.c_double * 3),
                ("scalar_mask", ctypes.c_uint32), ("n_dims", ctypes.c_int32), ("dims", ctypes.c_int32 * MAX_RANK),
                ("output", tk_tensor_spec),
                ("alpha", ctypes.c_double), ("beta", ctypes.c_double), ("threshold", ctypes.c_double),
                ("exponent", ctypes.c_double), ("value", ctypes.c_double),
                ("value_given", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class tk_program_desc(ctypes.Structure):
    _fields_ = [("n_inputs", ctypes.c_int32), ("inputs", ctypes.POINTER(tk_tensor_spec)),
                ("n_outputs", ctypes.c_int32), ("outputs", ctypes.POINTER(tk_tensor_spec)),
                ("n_ops", ctypes.c_int32), ("ops", ctypes.POINTER(tk_op)),
                ("n_inplace", ctypes.c_int32), ("inplace", ctypes.POINTER(ctypes.c_int32))]


class tk_options(ctypes.Structure):
    _fields_ = [("blocks_per_sm", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("fuse_pointwise", ctypes.c_int32), ("fuse_epilogues", ctypes.c_int32),
                ("inline_input_casts", ctypes.c_int32), ("tensor_cores", ctypes.c_int32),
                ("sm_count", ctypes.c_int32), ("profile", ctypes.c_int32),
                ("barrier_timeout_s", ctypes.c_double), ("expr_forms", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("epi_stage_bytes", ctypes.c_int32), ("cta_pairs", ctypes.c_int32),
                ("overlap_reductions", ctypes.c_int32)]


class tk_plan_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "materialized_ops", "inlined_ops", "fused_epilogues", "tensor_core_ops", "stages", "grid_barriers",
        "direct_outputs", "direct_state_commits", "max_work_items", "grid_blocks", "output_copies",
        "split_reductions")] + [("workspace_elements", ctypes.c_int64), ("arena_elements", ctypes.c_int64),
        ("compiled_tasks", ctypes.c_int32), ("chain_tasks", ctypes.c_int32), ("tasks", ctypes.c_int32),
        ("tma_descriptors", ctypes.c_int32), ("cta_pairs", ctypes.c_int32)]


class tk_task_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "stage", "kind", "op_index", "n_items", "form", "compiled_shape", "m", "n", "k", "tile_m", "tile_n",
        "parts", "staged_epilogue", "side_output", "staged_depth", "beside_tiles", "folded")] + [("numel", ctypes.c_int64)]


# (name, restype, argtypes) for every entry point of include/tk.h
SIGNATURES = [
    ("tk_options_default", None, [ctypes.POINTER(tk_options)]),
    ("tk_program_create", ctypes.c_int, [ctypes.POINTER(tk_program_desc), ctypes.POINTER(tk_options), ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_void_p)]),
    ("tk_program_destroy", None, [ctypes.c_void_p]),
    ("tk_allocate", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)]),
    ("tk_workspace_init", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    ("tk_run", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32,
                              ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                              ctypes.c_void_p]),
    ("tk_run_status", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    ("tk_resource_usage", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64 * 4]),
    ("tk_profile_read", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.POINTER(ctypes.c_int64), ctypes.c_size_t]),
    ("tk_plan_stats_get", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(tk_plan_stats)]),
    ("tk_plan_task", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(tk_task_info)]),
    ("tk_run_static", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32,
                                     ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32, ctypes.c_void_p]),
    ("tk_run_host", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32,
                                   ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                   ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
                                   ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p),
                                   ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    ("tk_last_error", ctypes.c_char_p, []),
]

STATIC_WORKSPACE_ELEMENTS = 2097152


class TkError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def lib():
    """The loaded libtk; raises if the shared library is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libtk.so is not built ({LIB_PATH}); call __graft_entry__.build() "
                                   "or persistent_step_megakernel_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, res, args in SIGNATURES:
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def check(status: int) -> None:
    if status != 0:
        raise TkError(status, lib().tk_last_error().decode())


# ----------------------------------------------------------- marshalling

def _spec(s: TensorSpec, ids: dict) -> tk_tensor_spec:
    c = tk_tensor_spec()
    c.buffer_id = ids[s.buffer]
    c.rank = len(s.shape)
    if c.rank > MAX_RANK:
        raise ValueError("tensor rank must be 0..4")
    for d, (n, st) in enumerate(zip(s.shape, s.strides)):
        c.shape[d] = int(n)
        c.strides[d] = int(st)
    c.offset = int(s.offset)
    c.dtype = DTYPE.get(s.dtype, 99)
    return c


class Described:
    """A program as C structs (keeps the arrays alive while in use)."""

    def __init__(self, program: Program):
        ids = {}
        for s in program.inputs:
            ids.setdefault(s.buffer, len(ids))
        for op in program.operations:
            ids.setdefault(op.output.buffer, len(ids))
        for s in program.outputs:
            ids.setdefault(s.buffer, len(ids))
        self.ids = ids
        self.inputs = (tk_tensor_spec * max(1, len(program.inputs)))(*[_spec(s, ids) for s in program.inputs])
        self.outputs = (tk_tensor_spec * max(1, len(program.outputs)))(*[_spec(s, ids) for s in program.outputs])
        ops = []
        for op in program.operations:
            c = tk_op()
            c.kind = OP_KIND.get(op.op, 99)
            c.n_inputs = len(op.inputs)
            for j, x in enumerate(op.inputs):
                if isinstance(x, TensorSpec):
                    c.inputs[j] = _spec(x, ids)
                else:
                    c.scalars[j] = float(x)
                    c.scalar_mask |= 1 << j
            c.output = _spec(op.output, ids)
            a = op.attrs
            c.alpha = float(a.get("alpha", 1.0))
            c.beta = float(a.get("beta", 1.0))
            c.threshold = float(a.get("threshold", 0.0))
            c.exponent = float(a.get("exponent", 2.0))
            c.value = float(a.get("value", 0.0))
            c.value_given = int("value" in a)
            dims = a.get("dims")
            c.n_dims = -1 if dims is None else len(tuple(dims))
            for j, d in enumerate(tuple(dims or ())):
                c.dims[j] = int(d)
            ops.append(c)
        self.ops = (tk_op * max(1, len(ops)))(*ops)
        pairs = [v for kv in sorted(program.inplace.items()) for v in kv]
        self.inplace = (ctypes.c_int32 * max(1, len(pairs)))(*pairs)
        self.desc = tk_program_desc(len(program.inputs), self.inputs, len(program.outputs), self.outputs,
                                    len(ops), self.ops, len(program.inplace), self.inplace)


def options(**kw) -> tk_options:
    o = tk_options()
    lib().tk_options_default(ctypes.byref(o))
    for k, v in kw.items():
        setattr(o, k, v)
    return o


# ----------------------------------------------------------- entry points

def tk_options_default() -> tk_options:
    return options()


def tk_program_create(program: Program, opts: tk_options | None = None, device: int = 0) -> ctypes.c_void_p:
    d = Described(program)
    h = ctypes.c_void_p()
    check(lib().tk_program_create(ctypes.byref(d.desc), ctypes.byref(opts) if opts is not None else None,
                                  device, ctypes.byref(h)))
    return h


def tk_program_destroy(handle) -> None:
    lib().tk_program_destroy(handle)


def tk_allocate(handle) -> int:
    n = ctypes.c_size_t()
    check(lib().tk_allocate(handle, ctypes.byref(n)))
    return n.value


def tk_workspace_init(handle, workspace_ptr: int, workspace_elements: int, stream: int = 0) -> None:
    check(lib().tk_workspace_init(handle, ctypes.c_void_p(workspace_ptr), workspace_elements, ctypes.c_void_p(stream)))


def tk_run(handle, input_ptrs, output_ptrs, workspace_ptr: int, workspace_elements: int, stream: int = 0) -> None:
    ins = (ctypes.c_void_p * max(1, len(input_ptrs)))(*input_ptrs)
    outs = (ctypes.c_void_p * max(1, len(output_ptrs)))(*output_ptrs)
    check(lib().tk_run(handle, ins, len(input_ptrs), outs, len(output_ptrs), ctypes.c_void_p(workspace_ptr),
                       workspace_elements, ctypes.c_void_p(stream)))


def tk_run_prepared(handle, input_ptrs, output_ptrs, workspace_ptr: int, workspace_elements: int, stream: int = 0):
    """tk_run with its arguments marshalled once: returns a callable that
    launches one step per call (for loops that launch the same buffers)."""
    ins = (ctypes.c_void_p * max(1, len(input_ptrs)))(*input_ptrs)
    outs = (ctypes.c_void_p * max(1, len(output_ptrs)))(*output_ptrs)
    args = (handle, ins, len(input_ptrs), outs, len(output_ptrs), ctypes.c_void_p(workspace_ptr), workspace_elements,
            ctypes.c_void_p(stream))
    fn = lib().tk_run

    def launch() -> None:
        rc = fn(*args)
        if rc != 0:
            check(rc)
    return launch


def tk_run_status(handle, workspace_ptr: int, stream: int = 0):
    st, stage = ctypes.c_int32(), ctypes.c_int32()
    check(lib().tk_run_status(handle, ctypes.c_void_p(workspace_ptr), ctypes.c_void_p(stream),
                              ctypes.byref(st), ctypes.byref(stage)))
    return st.value, stage.value


def tk_resource_usage(handle) -> dict:
    out = (ctypes.c_int64 * 4)()
    check(lib().tk_resource_usage(handle, out))
    return dict(zip(("registers_per_thread", "local_bytes_per_thread", "shared_bytes_per_block",
                     "resident_blocks_per_sm"), list(out)))


PROFILE_STAMPS = 9


def tk_profile_read(handle, workspace_ptr: int, stages: int, grid: int, stream: int = 0):
    """Stamps as a list [stage][block] of 9-tuples (see tk_profile_read in tk.h)."""
    n = PROFILE_STAMPS * stages * grid
    buf = (ctypes.c_int64 * n)()
    check(lib().tk_profile_read(handle, ctypes.c_void_p(workspace_ptr), ctypes.c_void_p(stream), buf, n))
    k = PROFILE_STAMPS
    return [[tuple(buf[(s * grid + b) * k:(s * grid + b + 1) * k]) for b in range(grid)] for s in range(stages)]


def tk_plan_stats_get(handle) -> dict:
    s = tk_plan_stats()
    check(lib().tk_plan_stats_get(handle, ctypes.byref(s)))
    return {name: getattr(s, name) for name, _ in tk_plan_stats._fields_}


TASK_KINDS = ("pointwise", "reduce_row", "reduce_col", "reduce_final", "gemm_simt", "gemm_tc", "splitk_final",
              "gemv")
EXPR_FORMS = ("instructions", "chain", "compiled")


def tk_plan_task(handle, index: int) -> dict:
    t = tk_task_info()
    check(lib().tk_plan_task(handle, index, ctypes.byref(t)))
    d = {name: getattr(t, name) for name, _ in tk_task_info._fields_}
    d["kind"] = TASK_KINDS[d["kind"]]
    d["form"] = EXPR_FORMS[d["form"]]
    return d


def tk_run_static(handle, input_ptrs, output_ptrs, stream: int = 0) -> None:
    """tk_run with the library's built-in 8 MiB workspace: allocates nothing.

    For callers that cannot allocate device memory where they run a step (see
    tk_run_static in include/tk.h).  The first call per device does set-up and
    should happen before any stream capture; calls share one array, so order
    them on one stream.
    """
    ins = (ctypes.c_void_p * max(1, len(input_ptrs)))(*input_ptrs)
    outs = (ctypes.c_void_p * max(1, len(output_ptrs)))(*output_ptrs)
    check(lib().tk_run_static(handle, ins, len(input_ptrs), outs, len(output_ptrs), ctypes.c_void_p(stream)))


def tk_run_host(handle, n_steps: int, input_ptrs, output_ptrs, batch, batch_alt_ptrs, host_batch_ptrs,
                results, host_result_ptrs, workspace_ptr: int, workspace_elements: int, stream: int = 0) -> None:
    """n_steps steps fed from host memory (tk_run_host in include/tk.h):
    host_batch_ptrs[s * len(batch) + b] is step s's host copy of input
    batch[b], host_result_ptrs[s * len(results) + r] receives output
    results[r] after step s."""
    P = ctypes.c_void_p
    ins = (P * max(1, len(input_ptrs)))(*input_ptrs)
    outs = (P * max(1, len(output_ptrs)))(*output_ptrs)
    bt = (ctypes.c_int32 * max(1, len(batch)))(*batch)
    alt = (P * max(1, len(batch_alt_ptrs)))(*batch_alt_ptrs)
    hb = (P * max(1, len(host_batch_ptrs)))(*host_batch_ptrs)
    rs = (ctypes.c_int32 * max(1, len(results)))(*results)
    hr = (P * max(1, len(host_result_ptrs)))(*host_result_ptrs)
    check(lib().tk_run_host(handle, n_steps, ins, len(input_ptrs), outs, len(output_ptrs), bt, len(batch), alt, hb,
                            rs, len(results), hr, P(workspace_ptr), workspace_elements, P(stream)))


def tk_last_error() -> str:
    return lib().tk_last_error().decode()
