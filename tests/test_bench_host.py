"""Host logic of bench.py that needs no GPU: the kernel-source hash that ties the committed ncu
counters to the code they were taken from, and the lookup of those counters."""
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


def test_comment_edits_keep_the_hash_and_code_edits_change_it(tmp_path, monkeypatch):
    csrc = tmp_path / "kimi_delta_attention_gate_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("__global__ void k(float* x) { x[0] = 1.f; }  // store\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (csrc / "k.cu").write_text("__global__ void k(float* x) { x[0] = 1.f; }  // reworded\n")
    assert bench.kernel_source_hash() == h0
    (csrc / "k.cu").write_text("__global__ void k(float* x) { x[0] = 2.f; }  // store\n")
    assert bench.kernel_source_hash() != h0
    (csrc / "k.cu").write_text("__global__ void k(float* x) { x[0] = 1.f; }  // store\n")
    (csrc / "j.cuh").write_text("#pragma once\n")
    assert bench.kernel_source_hash() != h0              # a new file is part of the code


def test_profiled_traffic_is_used_only_for_the_matching_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "kimi_delta_attention_gate_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("int k;\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash()
    summary = tmp_path / "profiles" / "stage_wl.txt"
    summary.write_text(f"kernel: k\nkernel_source_sha: {h} (comments excluded)\n"
                       "dram_bytes_per_launch: 123456\n")
    assert bench.profiled_traffic("stage", "wl") == 123456.0
    (csrc / "k.cu").write_text("int k2;\n")
    assert bench.profiled_traffic("stage", "wl") is None
    assert bench.profiled_traffic("other", "wl") is None

