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


def test_backward_measurement_logic_with_the_gpu_calls_faked(monkeypatch):
    """measure_backward's bookkeeping on the CPU: the host-only entry points are the real
    ones, the launches, events and device status are stand-ins (every stage 'takes' a fixed
    time), so that the line it builds can be checked without a GPU."""
    torch = __import__("pytest").importorskip("torch")
    import numpy as np
    import kimi_delta_attention_gate_gb300 as kda
    from kimi_delta_attention_gate_gb300 import _binding as kb
    from kimi_delta_attention_gate_gb300 import build as kbuild
    from kimi_delta_attention_gate_gb300 import inputs as kin
    kbuild.build()

    clock = {"t": 0.0}
    per_stage_ms = {"zero_outputs": 0.5, "bwd_prep": 2.0, "bwd_states": 3.0, "bwd_dstate": 4.0,
                    "bwd_grads": 10.0, "bwd_gate": 1.0}

    class Event:
        def __init__(self, enable_timing=False):
            self.t = None

        def record(self, stream=None):
            self.t = clock["t"]

        def elapsed_time(self, other):
            return other.t - self.t

    class FakeKb:
        def __getattr__(self, name):
            return getattr(kb, name)

        def kda_bwd(self, p, sh):
            clock["t"] += sum(per_stage_ms.values())
            return kb.KDA_OK

        def kda_bwd_stage(self, p, sh, i):
            clock["t"] += per_stage_ms[kb.kda_bwd_stage_name(p, i)]
            return kb.KDA_OK

        def kda_get_device_status(self, sh):
            return 0

    class Stream:
        cuda_stream = 0

    monkeypatch.setattr(torch.cuda, "Event", Event)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a: None)
    wl = kin.Workload("tiny_bwd", B=1, T=130, H=2, HV=2, K=32, V=32, chunk_size=64, dtype="bf16",
                      gate=kin.GATE_SAFE, lower_bound=-5.0, seed=3)
    inp = kin.make_inputs(wl)

    def up(x, dtype):
        if x is None:
            return None
        if dtype == "bf16":
            return torch.from_numpy(kin.to_bf16_bits(x).view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(x, np.float32))

    t = dict(q=up(inp.q, "bf16"), k=up(inp.k, "bf16"), v=up(inp.v, "bf16"), g=up(inp.g, "bf16"),
             b=up(inp.beta, "bf16"), A_log=up(inp.A_log, "f32"), dt_bias=up(inp.dt_bias, "f32"),
             h0=None, cu=None, cu_cpu=None)
    out = bench.measure_backward(FakeKb(), kda, "cpu", Stream(), inp, t, {"lower_bound": -5.0}, 3)
    assert out["stages"] == {k: v for k, v in per_stage_ms.items()}
    assert abs(out["ms_per_step"] - sum(per_stage_ms.values())) < 1e-9
    assert out["value"] == inp.n_tokens / (out["ms_per_step"] / 1e3)
    roof = out["roofline"]
    assert roof["kernel"] == "bwd_grads" and roof["bound"] == "alu"
    nct = 3                                             # 130 tokens, chunk 64
    fl = bench.bwd_stage_flops("bwd_grads", 64, 32, 32, nct, 2)
    assert roof["flops_per_launch"] == fl
    assert abs(roof["achieved"] - fl / 10e-3 / 1e12) < 1e-12
    assert abs(roof["peak"] - 80.54784) < 1e-9 and 0 < roof["frac"] < 1
    assert out["gpu_launches_per_step"] == 5
    assert out["workspace_bytes"] > 0
