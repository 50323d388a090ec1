"""The ctypes mirrors of the C parameter blocks (kda_fwd_params, kda_bwd_params) against the
layout a C compiler gives the headers: a small C program built with gcc prints every field's
offset and each struct's size.  Host only."""
import ctypes
import os
import shutil
import subprocess

import pytest

from kimi_delta_attention_gate_gb300 import _binding as kb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _c_layout(tmp_path, struct, fields):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    src = tmp_path / f"{struct}.c"
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "kda_bwd.h"', "int main(void) {",
             f'  printf("sizeof %zu\\n", sizeof({struct}));']
    lines += [f'  printf("{f} %zu\\n", offsetof({struct}, {f}));' for f in fields]
    lines += ["  return 0;", "}"]
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / struct
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.splitlines())}


@pytest.mark.parametrize("cls,struct", [(kb.kda_fwd_params, "kda_fwd_params"),
                                        (kb.kda_bwd_params, "kda_bwd_params")])
def test_ctypes_mirror_matches_the_c_layout(tmp_path, cls, struct):
    fields = [name for name, _ in cls._fields_]
    c = _c_layout(tmp_path, struct, fields)
    assert c["sizeof"] == ctypes.sizeof(cls)
    for name in fields:
        assert c[name] == getattr(cls, name).offset, name
