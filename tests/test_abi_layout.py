"""The Python binding agrees with include/grs.h, checked on the host (no
GPU): every #define and enum constant of the header has the same value in
the binding, and every struct the binding declares has the C compiler's
size and field offsets (a small C program built with the host compiler
prints them)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "grs.h")


@pytest.fixture(scope="module")
def grs():
    from gradient_reduction_sharded_gb300 import _build
    _build.build()
    from gradient_reduction_sharded_gb300 import grs as g
    return g


def header_constants() -> dict:
    """#define GRS_X <int expr> and enumerators GRS_X = <int> of the header."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    out = {}
    for name, expr in re.findall(r"^#define\s+(GRS_[A-Z0-9_]+)\s+(.+)$", text, flags=re.M):
        expr = re.sub(r"(\d+)[uU]", r"\1", expr.strip())
        if re.fullmatch(r"[\d\s()<<+*]+", expr):
            out[name] = int(eval(expr, {"__builtins__": {}}))  # digits, parentheses and shifts only
    for name, val in re.findall(r"\b(GRS_[A-Z0-9_]+)\s*=\s*(\d+)", text):
        out[name] = int(val)
    return out


def test_every_header_constant_matches_the_binding(grs):
    consts = header_constants()
    assert len(consts) >= 20, consts
    for name, val in consts.items():
        assert hasattr(grs, name), f"{name} is in grs.h but not in the binding"
        assert getattr(grs, name) == val, (name, getattr(grs, name), val)


STRUCTS = ("grs_plan_info", "grs_bucket_desc", "grs_segment_desc", "grs_tensor_desc", "grs_adamw")


def test_struct_layouts_match_the_c_compiler(grs, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "grs.h"', "int main(void) {"]
    for s in STRUCTS:
        lines.append(f'  printf("{s} sizeof %zu\\n", sizeof({s}));')
        for field, _ in getattr(grs, s)._fields_:
            lines.append(f'  printf("{s} {field} %zu\\n", offsetof({s}, {field}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        s, field, val = line.split()
        got[(s, field)] = int(val)
    for s in STRUCTS:
        cls = getattr(grs, s)
        assert got[(s, "sizeof")] == ctypes.sizeof(cls), (s, got[(s, "sizeof")], ctypes.sizeof(cls))
        for field, _ in cls._fields_:
            assert got[(s, field)] == getattr(cls, field).offset, (s, field)
