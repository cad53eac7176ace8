"""The C-ABI library builds, loads without a GPU and exports every symbol
include/tk.h declares; the Python binding covers the same names."""
import ctypes
import os
import re
import subprocess

from persistent_step_megakernel_gb300 import binding as B
from persistent_step_megakernel_gb300.build import LIB, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared():
    text = open(os.path.join(ROOT, "include", "tk.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(tk_[a-z_]+)\s*\(", text))


def test_library_exports_every_declared_symbol():
    build()
    names = declared()
    assert {"tk_program_create", "tk_allocate", "tk_run", "tk_run_status"} <= names
    lib = ctypes.CDLL(LIB)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(tk_[a-z_]+)\b", out))
    assert names <= exported, names - exported


def test_binding_covers_the_header():
    assert {n for n, _, _ in B.SIGNATURES} == declared()


def test_options_defaults():
    o = B.tk_options_default()
    assert (o.blocks_per_sm, o.fuse_pointwise, o.fuse_epilogues, o.inline_input_casts, o.tensor_cores) == (1, 1, 1, 1, 1)
    assert o.barrier_timeout_s == 2.0


def test_struct_sizes_match_the_header():
    assert ctypes.sizeof(B.tk_tensor_spec) == 88
    assert ctypes.sizeof(B.tk_op) == 448
    assert ctypes.sizeof(B.tk_options) == 48
