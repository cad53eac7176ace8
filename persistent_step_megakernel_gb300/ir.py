"""Static program description: tensors, operations and the training-step program.

The shape of this description follows trainkernel's IR as it is used by
trainkernel/codegen.py (page "trainkernel 0.1.0 -- trainkernel/codegen.py",
the ``TensorSpec``/``Operation``/``Program`` uses in ``_Generator``): a tensor
is a (buffer, shape, strides, element offset, dtype) view, an operation names
its kind, its tensor-or-scalar inputs, its output view and its attributes, and a
program lists its inputs, its outputs and its operations in topological order.

This module holds data only: no arithmetic of the method lives here, so that the
CPU oracle and the CUDA path can both be handed the same program.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math
from typing import Union

DTYPES = ("float32", "float16", "bfloat16")
POINTWISE = ("add", "sub", "mul", "div", "neg", "relu", "pow",
             "threshold_backward", "full", "cast")
MATMUL = ("mm", "addmm")
REDUCTIONS = ("sum", "mean")
OPS = POINTWISE + MATMUL + REDUCTIONS


def numel(shape) -> int:
    return int(math.prod(shape))


def contiguous_strides(shape) -> tuple:
    return tuple(int(math.prod(shape[i + 1:])) for i in range(len(shape)))


@dataclass(frozen=True)
class TensorSpec:
    """A strided view of a named buffer; strides and offset count elements."""
    buffer: str
    shape: tuple
    strides: tuple
    offset: int = 0
    dtype: str = "float32"

    @staticmethod
    def contiguous(buffer: str, shape, dtype: str) -> "TensorSpec":
        shape = tuple(int(s) for s in shape)
        return TensorSpec(buffer, shape, contiguous_strides(shape), 0, dtype)

    @property
    def T(self) -> "TensorSpec":
        """Transposed view of a rank-2 tensor (no data movement)."""
        if len(self.shape) != 2:
            raise ValueError("transpose needs a rank-2 view")
        return TensorSpec(self.buffer, (self.shape[1], self.shape[0]),
                          (self.strides[1], self.strides[0]), self.offset, self.dtype)

    @property
    def is_contiguous(self) -> bool:
        return self.strides == contiguous_strides(self.shape) and self.offset == 0


Operand = Union[TensorSpec, float, int]


@dataclass(frozen=True)
class Operation:
    name: str
    op: str
    inputs: tuple
    output: TensorSpec
    attrs: dict = field(default_factory=dict)


@dataclass
class Program:
    """Inputs, outputs and operations in topological order.

    ``inplace`` maps an output slot to the input index whose storage it
    overwrites (the in-place state update of a training step).
    """
    inputs: list
    outputs: list
    operations: list
    inplace: dict = field(default_factory=dict)

    def producer(self, buffer: str):
        for op in self.operations:
            if op.output.buffer == buffer:
                return op
        return None
