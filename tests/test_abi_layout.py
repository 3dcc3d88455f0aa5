"""The ctypes binding's structs have the C header's layout (CPU; gcc).

A small C program compiled against include/tfl.h prints sizeof of every struct
and the offset and size of every field; the binding's ctypes structures must agree, or
every call through them would hand the library misplaced arguments.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

import attention_qkv_gemm_gb300 as pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

STRUCTS = {
    "tfl_shape": pkg.TflShape,
    "tfl_layer_weights": pkg.TflLayerWeights,
    "tfl_weights": pkg.TflWeights,
    "tfl_options": pkg.TflOptions,
}


def _c_layout():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "tfl.h"', "int main(void) {"]
    for cname, cls in STRUCTS.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'  printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
            lines.append(f'  printf("{cname} {f}.size %zu\\n", sizeof((({cname}*)0)->{f}));')
    lines += ["  return 0;", "}"]
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        with open(src, "w") as fh:
            fh.write("\n".join(lines))
        subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True,
                       capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    got = {}
    for line in out.splitlines():
        name, field, val = line.split()
        got[(name, field)] = int(val)
    return got


def test_struct_sizes_and_offsets_match_the_header():
    c = _c_layout()
    for cname, cls in STRUCTS.items():
        assert c[(cname, "size")] == ctypes_sizeof(cls), cname
        for f, _ in cls._fields_:
            assert c[(cname, f)] == getattr(cls, f).offset, f"{cname}.{f} offset"
            assert c[(cname, f + ".size")] == getattr(cls, f).size, f"{cname}.{f} size"


def ctypes_sizeof(cls):
    import ctypes
    return ctypes.sizeof(cls)
