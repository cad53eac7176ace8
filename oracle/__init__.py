"""Python access to the CPU oracle (``oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the product path never imports it.

The oracle takes its own text serialisation of a program (written here from
any object with the ``inputs``/``outputs``/``operations`` shape of the
training-step IR) and exchanges tensor values as float64 arrays holding the
values already rounded to each tensor's dtype.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODE = {"float32": 0, "float16": 1, "bfloat16": 2, "float64": 3}


def build(force: bool = False) -> str:
    """Compile liboracle.so with strict IEEE float semantics (no contraction)."""
    src = os.path.join(_HERE, "oracle.cpp")
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
                        "-fopenmp", "-fPIC", "-shared", "-o", tmp, src], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, cp, i64, dp = ctypes.c_void_p, ctypes.c_char_p, ctypes.c_int64, ctypes.POINTER(ctypes.c_double)
            L.oracle_load.restype = vp
            L.oracle_load.argtypes = [cp]
            L.oracle_free.argtypes = [vp]
            L.oracle_set.argtypes = [vp, cp, dp, i64]
            L.oracle_size.restype = i64
            L.oracle_size.argtypes = [vp, cp]
            L.oracle_get.argtypes = [vp, cp, dp, i64]
            L.oracle_run.argtypes = [vp]
            L.oracle_eval_op.argtypes = [vp, ctypes.c_int]
            L.oracle_eval_op_sampled.argtypes = [vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int64), i64, dp, dp]
            L.oracle_output.argtypes = [vp, ctypes.c_int, dp, i64]
            L.oracle_round.argtypes = [ctypes.c_int, dp, dp, i64]
            L.oracle_last_error.restype = cp
            _lib = L
    return _lib


def _spec_text(s) -> str:
    shape = " ".join(str(int(v)) for v in s.shape)
    strides = " ".join(str(int(v)) for v in s.strides)
    return f"{s.buffer} {s.dtype} {len(s.shape)} {shape} {strides} {int(s.offset)}"


def serialize(program) -> str:
    lines = ["TKORACLE 1", f"INPUTS {len(program.inputs)}"]
    lines += [_spec_text(s) for s in program.inputs]
    lines.append(f"OPS {len(program.operations)}")
    for op in program.operations:
        lines.append(f"OP {op.op} {op.name} {len(op.inputs)}")
        for x in op.inputs:
            if hasattr(x, "buffer"):
                lines.append("T " + _spec_text(x))
            else:
                lines.append("S " + repr(float(x)))
        lines.append("OUT " + _spec_text(op.output))
        a = op.attrs
        dims = a.get("dims")
        dims_txt = "-1" if dims is None else " ".join([str(len(tuple(dims)))] + [str(int(d)) for d in dims])
        lines.append("ATTR {} {} {} {} {} {} {} {}".format(
            repr(float(a.get("alpha", 1))), repr(float(a.get("beta", 1))),
            repr(float(a.get("threshold", 0))), repr(float(a.get("exponent", 2))),
            repr(float(a.get("value", 0))), int("exponent" in a), int("value" in a), dims_txt))
    lines.append(f"OUTPUTS {len(program.outputs)}")
    lines += [_spec_text(s) for s in program.outputs]
    lines.append("END")
    return "\n".join(lines) + "\n"


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(rc: int):
    if rc != 0:
        raise RuntimeError(lib().oracle_last_error().decode())


class Oracle:
    """One loaded program; buffers hold float64 values rounded to their dtype."""

    def __init__(self, program):
        self.program = program
        self._h = lib().oracle_load(serialize(program).encode())
        if not self._h:
            raise ValueError(lib().oracle_last_error().decode())

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().oracle_free(h)
            self._h = None

    def set(self, buffer: str, values) -> None:
        a = np.ascontiguousarray(np.asarray(values, dtype=np.float64).reshape(-1))
        _check(lib().oracle_set(self._h, buffer.encode(), _dp(a), a.size))

    def set_inputs(self, values) -> None:
        for spec, v in zip(self.program.inputs, values):
            self.set(spec.buffer, v)

    def get(self, buffer: str) -> np.ndarray:
        n = lib().oracle_size(self._h, buffer.encode())
        if n < 0:
            raise KeyError(buffer)
        out = np.empty(n, dtype=np.float64)
        _check(lib().oracle_get(self._h, buffer.encode(), _dp(out), n))
        return out

    def run(self) -> None:
        _check(lib().oracle_run(self._h))

    def eval_op(self, index: int) -> np.ndarray:
        _check(lib().oracle_eval_op(self._h, index))
        op = self.program.operations[index]
        return self.get(op.output.buffer).reshape(op.output.shape)

    def eval_op_sampled(self, index: int, flat_indices):
        idx = np.ascontiguousarray(np.asarray(flat_indices, dtype=np.int64))
        out = np.empty(idx.size, dtype=np.float64)
        bound = np.empty(idx.size, dtype=np.float64)
        _check(lib().oracle_eval_op_sampled(self._h, index, idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                            idx.size, _dp(out), _dp(bound)))
        return out, bound

    def output(self, slot: int) -> np.ndarray:
        spec = self.program.outputs[slot]
        n = int(np.prod(spec.shape)) if spec.shape else 1
        out = np.empty(n, dtype=np.float64)
        _check(lib().oracle_output(self._h, slot, _dp(out), n))
        return out.reshape(spec.shape)

    def outputs(self) -> list:
        return [self.output(i) for i in range(len(self.program.outputs))]


def run_program(program, input_values) -> list:
    """Evaluate a whole program on float64 input values; returns every output."""
    o = Oracle(program)
    o.set_inputs(input_values)
    o.run()
    return o.outputs()


def round_values(values, dtype: str) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(values, dtype=np.float64).reshape(-1))
    out = np.empty_like(a)
    _check(lib().oracle_round(DTYPE_CODE[dtype], _dp(a), _dp(out), a.size))
    return out.reshape(np.shape(values))


def threads() -> int:
    return int(lib().oracle_threads())
