"""GB300-native persistent training-step kernel.

One functional training step of a small MLP -- forward addmm/relu, loss, explicit
backward mm/threshold_backward, bias column sums and the in-place parameter
update -- runs as a static op list inside a single cooperative persistent
kernel written for sm_103a.  The kernel sits behind the C ABI declared in
``include/tk.h`` (``libtk.so``); :mod:`.binding` is a thin ctypes layer over it.

Importing this package loads nothing native; :func:`binding.lib` loads the
shared library on first use and raises if it has not been built.
"""
from .ir import Operation, Program, TensorSpec  # noqa: F401

__all__ = ["Operation", "Program", "TensorSpec"]
