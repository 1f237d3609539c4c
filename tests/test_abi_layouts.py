"""The ctypes mirrors of the C ABI's structs have the header's layout.

A small C program, compiled with the host compiler against include/kvev.h,
prints sizeof and offsetof of every field that the Python binding declares.
Each must equal the ctypes figure, and a field name the header lacks fails the
compile.  This needs no GPU and no CUDA library."""
import ctypes
import os
import shutil
import subprocess

import pytest

from decoding_kv_cache_split_gb300 import kvev

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = [kvev.kvev_layout, kvev.kvev_cache, kvev.kvev_state, kvev.kvev_region_table,
           kvev.kvev_paged_cache, kvev.kvev_block_state, kvev.kvev_tier_cache,
           kvev.kvev_tier_state]


@pytest.fixture(scope="module")
def c_layouts(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "kvev.h"', "int main(void) {"]
    for T in STRUCTS:
        n = T.__name__
        lines.append(f'    printf("{n} . %zu\\n", sizeof({n}));')
        for f in T._fields_:
            lines.append(f'    printf("{n} {f[0]} %zu\\n", offsetof({n}, {f[0]}));')
    lines += ["    return 0;", "}"]
    d = tmp_path_factory.mktemp("abi_layout")
    src, exe = d / "layout.c", d / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-o", str(exe), str(src)], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {}
    for line in out.splitlines():
        struct, field, value = line.split()
        got[(struct, field)] = int(value)
    return got


@pytest.mark.parametrize("T", STRUCTS, ids=[T.__name__ for T in STRUCTS])
def test_ctypes_mirror_matches_the_header(c_layouts, T):
    n = T.__name__
    assert ctypes.sizeof(T) == c_layouts[(n, ".")], f"sizeof({n})"
    for f in T._fields_:
        assert getattr(T, f[0]).offset == c_layouts[(n, f[0])], f"offsetof({n}, {f[0]})"
