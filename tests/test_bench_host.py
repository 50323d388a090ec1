"""Host logic of bench.py that needs no GPU: the source hash that ties the committed ncu
counters to the code of the kernel they were taken from, and the lookup of those counters."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_keeps_literals():
    src = 'int a = 1; // one\nconst char* s = "// not a comment /* either */";\n' \
          "char c = '/'; /* two\n lines */ int b;   \n"
    out = bench._code_only(src)
    assert "one" not in out and "two" not in out and "lines" not in out
    assert '"// not a comment /* either */"' in out and "'/'" in out
    assert out.count("\n") == src.count("\n")          # line structure kept
    assert not any(line.endswith(" ") for line in out.split("\n"))


def _tree(tmp_path, monkeypatch):
    csrc = tmp_path / "kimi_delta_attention_gate_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (tmp_path / "include" / "api.h").write_text("#define FLAG 1\n")
    (csrc / "common.cuh").write_text('#include "api.h"\nint helper;\n')
    (csrc / "k.cu").write_text('#include "common.cuh"\n#include <stdio.h>\n'
                               "__global__ void k(float* x) { x[0] = 1.f; }  // store\n")
    (csrc / "other.cu").write_text("__global__ void j() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return csrc


def test_translation_unit_follows_project_includes(tmp_path, monkeypatch):
    _tree(tmp_path, monkeypatch)
    names = sorted(os.path.basename(f) for f in bench.tu_files("k.cu"))
    assert names == ["api.h", "common.cuh", "k.cu"]     # <stdio.h> and other.cu are not in it


def test_unit_hash_ignores_comments_and_other_units(tmp_path, monkeypatch):
    csrc = _tree(tmp_path, monkeypatch)
    h0 = bench.kernel_source_hash("k.cu")
    body = '#include "common.cuh"\n#include <stdio.h>\n__global__ void k(float* x) { x[0] = %s; }%s\n'
    (csrc / "k.cu").write_text(body % ("1.f", "  // reworded"))
    assert bench.kernel_source_hash("k.cu") == h0
    (csrc / "other.cu").write_text("__global__ void j() { int changed; }\n")
    (csrc / "new_unit.cu").write_text("__global__ void n() {}\n")
    assert bench.kernel_source_hash("k.cu") == h0      # another unit changed or was added
    (tmp_path / "include" / "api.h").write_text("#define FLAG 2\n")
    assert bench.kernel_source_hash("k.cu") != h0      # an included header is part of the unit
    (tmp_path / "include" / "api.h").write_text("#define FLAG 1\n")
    (csrc / "k.cu").write_text(body % ("2.f", ""))
    assert bench.kernel_source_hash("k.cu") != h0


def test_profiled_traffic_is_used_only_for_the_matching_hash(tmp_path, monkeypatch):
    csrc = _tree(tmp_path, monkeypatch)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setitem(bench.KERNEL_TU, "stage", "k.cu")
    h = bench.kernel_source_hash("k.cu")
    summary = tmp_path / "profiles" / "stage_wl.txt"
    summary.write_text(f"kernel: k\nkernel_source_sha: {h} (translation unit k.cu)\n"
                       "dram_bytes_per_launch: 123456\n")
    assert bench.profiled_traffic("stage", "wl") == 123456.0
    (csrc / "common.cuh").write_text('#include "api.h"\nint helper2;\n')
    assert bench.profiled_traffic("stage", "wl") is None
    assert bench.profiled_traffic("unknown_stage", "wl") is None
