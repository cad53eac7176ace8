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


STRUCTS = ("tk_tensor_spec", "tk_op", "tk_program_desc", "tk_options", "tk_plan_stats", "tk_task_info")


def test_struct_layouts_match_the_header(tmp_path):
    # a C compiler's view of the header: size of every struct and offset of every field
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "tk.h"', "int main(void) {"]
    for name in STRUCTS:
        lines.append(f'  printf("{name} %zu\\n", sizeof({name}));')
        for field, _ in getattr(B, name)._fields_:
            lines.append(f'  printf("{name}.{field} %zu\\n", offsetof({name}, {field}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    c = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines())
    for name in STRUCTS:
        cls = getattr(B, name)
        assert int(c[name]) == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert int(c[f"{name}.{field}"]) == getattr(cls, field).offset, f"{name}.{field}"
