"""The ctypes structs of the binding have the C header's layout: a small C program compiled
against include/sparse_mla.h prints every struct's size and field offsets (no GPU needed)."""

import ctypes
import os
import shutil
import subprocess

import pytest

import sparse_mla_attention_decode_gb300 as smla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = [smla.smla_dims, smla.smla_decode_opts, smla.smla_topk_dims, smla.smla_indexer_dims]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_struct_layouts_match_the_header(tmp_path):
    lines = ['#include <stdio.h>', '#include "sparse_mla.h"', "int main(void) {"]
    for s in STRUCTS:
        n = s.__name__
        lines.append(f'  printf("{n} size %zu\\n", sizeof({n}));')
        for f, _ in s._fields_:
            lines.append(f'  printf("{n} {f} %zu\\n", offsetof({n}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = dict(line.rsplit(" ", 1) for line in subprocess.run([str(exe)], check=True,
                                                                capture_output=True,
                                                                text=True).stdout.splitlines())
    for s in STRUCTS:
        n = s.__name__
        assert int(got[f"{n} size"]) == ctypes.sizeof(s), n
        for f, _ in s._fields_:
            assert int(got[f"{n} {f}"]) == getattr(s, f).offset, (n, f)
