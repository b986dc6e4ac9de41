"""The binding's ctypes mirrors of the structs in include/lmoe.h have the C
layout: a small C program built with gcc against the header prints every
field's offset and size and each struct's size, which must equal what ctypes
computes.  A field missing on either side, a reordered field or a wrong type
fails here (no GPU: only the header and the CUDA runtime's type headers are
compiled)."""
import ctypes
import os
import shutil
import subprocess

import pytest

from sparse_moe_layer_bias_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INCLUDE = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")

STRUCTS = {
    "lmoe_config": binding.LmoeConfig,
    "lmoe_weights": binding.LmoeWeights,
    "lmoe_grads": binding.LmoeGrads,
    "lmoe_ws_layout": binding.LmoeWsLayout,
}


def c_layout(tmp_path):
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "lmoe.h"', "int main(void) {"]
    for cname, py in STRUCTS.items():
        lines.append(f'    printf("{cname} . %zu %zu\\n", (size_t)0, sizeof({cname}));')
        for field, _ in py._fields_:
            lines.append(f'    printf("{cname} {field} %zu %zu\\n", offsetof({cname}, {field}), '
                         f"sizeof((({cname} *)0)->{field}));")
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    exe = tmp_path / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", CUDA_INCLUDE, str(src), "-o", str(exe)], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    table = {}
    for row in out.split("\n"):
        if row:
            s, f, off, size = row.split()
            table[(s, f)] = (int(off), int(size))
    return table


@pytest.mark.skipif(shutil.which("gcc") is None or not os.path.isdir(CUDA_INCLUDE),
                    reason="needs gcc and the CUDA headers")
def test_ctypes_structs_match_the_header(tmp_path):
    table = c_layout(tmp_path)
    for cname, py in STRUCTS.items():
        assert table[(cname, ".")][1] == ctypes.sizeof(py), cname
        for field, ctype in py._fields_:
            got = (getattr(py, field).offset, ctypes.sizeof(ctype))
            assert table[(cname, field)] == got, (cname, field, table[(cname, field)], got)
