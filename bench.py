"""Benchmark of the GB300 chunk-parallel KDA forward pass.

One step = one full forward pass (every kernel of the path) over the
long-context workload B=1, T=65536, H=HV=32, K=V=128, chunk 64, bf16, safe gate
(lower_bound -5), on synthetic seeded inputs already resident in HBM.  Inputs
(2.7 GB per step) are larger than L2 (129 MB), so no L2 flush is needed between
steps.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun), every rank runs its own replica of the workload on its
own GPU (weak scaling, no collective on the data path); the timed region is
bracketed by barriers and the max over ranks is reported.  ``--impl reference``
times the CPU fp64 oracle on the host cores (rank 0 only), each step a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import re
import json
import os
import platform
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from kimi_delta_attention_gate_gb300 import inputs as kin  # noqa: E402

METRIC = "KDA chunk fwd tokens/s at T=64K,H=32,K=V=128 bf16; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def elem(dtype: str) -> int:
    return 2 if dtype == "bf16" else 4


def essential_bytes(inp: kin.Inputs) -> float:
    """Bytes the method must move: q, k, v, g, beta read once, o written once, plus
    the initial / final state and the gate parameters."""
    wl = inp.wl
    e = elem(wl.dtype)
    ntok = inp.n_tokens
    per_tok = e * (2 * wl.H * wl.K + wl.HV * (wl.V + wl.K + 1) + wl.HV * wl.V)
    state = inp.N * wl.HV * wl.K * wl.V * 4 * ((inp.h0 is not None) + 1)
    params = 4 * wl.HV * (1 + wl.K)
    return float(ntok * per_tok + state + params)


def dense_flops(inp: kin.Inputs) -> float:
    """2C(3K+2V) + 6KV flops per token per value head (chunk tiles counted dense)."""
    wl = inp.wl
    C, K, V = wl.chunk_size, wl.K, wl.V
    return float(inp.n_tokens * wl.HV * (2 * C * (3 * K + 2 * V) + 6 * K * V))


def own_bytes(name: str, inp: kin.Inputs) -> float:
    """Method bytes one launch of the named stage owns: the inputs it is the first to read
    and the outputs it writes, intermediates excluded (they sum to essential_bytes)."""
    wl = inp.wl
    e = elem(wl.dtype)
    ntok = inp.n_tokens
    state = inp.N * wl.HV * wl.K * wl.V * 4 * ((inp.h0 is not None) + 1)
    if name in ("tc_intra", "simt_intra"):
        return float(ntok * e * (2 * wl.H * wl.K + wl.HV * (wl.K + 1)) + 4 * wl.HV * (1 + wl.K))
    if name in ("tc_recur", "simt_recur"):
        return float(ntok * e * 2 * wl.HV * wl.V + state)
    if name == "chunk_table":
        return float(16 * (inp.N + 1))
    return essential_bytes(inp)


_C_TOKENS = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'', re.S)


def _code_only(text: str) -> str:
    """C / CUDA source with its comments removed (string and character literals kept) and
    trailing blanks dropped: what the compiler sees, so a comment edit keeps the hash."""
    text = _C_TOKENS.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else
                         ("\n" * m.group(0).count("\n") if m.group(0).startswith("/*") else ""), text)
    return "\n".join(line.rstrip() for line in text.split("\n"))


# Translation unit of each kernel the bench names: ncu counters depend on that unit's code only.
KERNEL_TU = {"tc_intra": "kda_tc.cu", "tc_recur": "kda_tc.cu", "recurrent_k128": "kda_recurrent.cu",
             "simt_intra": "kda_simt.cu", "simt_recur": "kda_simt.cu", "chunk_table": "kda_simt.cu"}
_INCLUDE = re.compile(r'^\s*#\s*include\s*"([^"]+)"', re.M)


def tu_files(root: str):
    """The project files one translation unit compiles: `root` (a file of csrc/) and every
    header it includes from csrc/ or include/, recursively."""
    csrc = os.path.join(ROOT, "kimi_delta_attention_gate_gb300", "csrc")
    dirs = (csrc, os.path.join(ROOT, "include"))
    seen, todo = [], [os.path.join(csrc, root)]
    while todo:
        f = todo.pop()
        if f in seen:
            continue
        seen.append(f)
        for inc in _INCLUDE.findall(open(f, encoding="utf-8").read()):
            for d in dirs:
                cand = os.path.join(d, inc)
                if os.path.exists(cand):
                    todo.append(cand)
                    break
    return sorted(seen)


def kernel_source_hash(tu: str = None) -> str:
    """Hash of the code (comments excluded) of one kernel's translation unit, or of every
    csrc/ file when `tu` is None: ncu counters committed under profiles/ are used only while
    it matches the hash recorded with them."""
    if tu is None:
        files = sorted(glob.glob(os.path.join(ROOT, "kimi_delta_attention_gate_gb300", "csrc", "*")))
    else:
        files = tu_files(tu)
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode() + b"\0")
        h.update(_code_only(open(f, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(stage: str, workload: str):
    """DRAM bytes per launch of `stage` from a committed ncu summary, if it was taken
    from the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"{stage}_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    tu = KERNEL_TU.get(stage)
    if tu is None or fields.get("kernel_source_sha", "").split(" ")[0] != kernel_source_hash(tu):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 <= r[0] <= t1] or \
            [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm, smax, power = [], [], []
        for _, parts in inside:
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                pass
            for i, n in enumerate(names):
                if parts[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "power_w_max": float(max(power)) if power else None,
                "samples": len(inside), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ---------------------------------------------------------------------------------------

def oracle_sample_time(inp: kin.Inputs, tokens: int, heads: int, nthreads: int):
    """Time the oracle on the first `tokens` tokens of every sequence-0 head in
    range(heads).  Returns seconds."""
    import oracle
    wl = inp.wl
    sl = slice(0, tokens)
    hs = slice(0, heads)
    q = inp.q[:1, sl, hs]
    k = inp.k[:1, sl, hs]
    v = inp.v[:1, sl, hs]
    g = inp.g[:1, sl, hs]
    b = inp.beta[:1, sl, hs]
    A_log = None if inp.A_log is None else inp.A_log[hs]
    dt = None if inp.dt_bias is None else inp.dt_bias.reshape(wl.HV, wl.K)[hs].reshape(-1)
    h0 = None if inp.h0 is None else inp.h0[:1, hs]
    lb = wl.lower_bound if wl.gate == kin.GATE_SAFE else None
    t = time.perf_counter()
    oracle.fwd(q, k, v, g, b, A_log=A_log, dt_bias=dt, gate_mode=wl.gate, lower_bound=lb,
               scale=inp.scale, initial_state=h0, nthreads=nthreads)
    return time.perf_counter() - t


def cpu_sample_plan(inp: kin.Inputs, target_s: float, nthreads: int):
    """Pick a bounded oracle sample (all heads of the first sequence, a prefix of its
    tokens) expected to take about target_s seconds; returns (tokens, heads)."""
    wl = inp.wl
    heads = wl.HV
    probe = min(wl.T, 256)
    dt = max(oracle_sample_time(inp, probe, heads, nthreads), 1e-4)
    tokens = int(min(wl.T, max(probe, probe * target_s / dt)))
    return tokens, heads


def run_reference(args, wl):
    """--impl reference: the oracle, as it stands, on the host cores."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    oracle.build()
    inp = kin.make_inputs(wl)
    nthreads = oracle.max_threads()
    # each step a bounded sample, sized so that the warm-up and timed steps together take
    # about two minutes of host time (at most 4 s a step)
    per_step = min(4.0, 120.0 / max(1, args.steps + args.warmup))
    tokens, heads = cpu_sample_plan(inp, per_step, nthreads)
    for _ in range(args.warmup):
        oracle_sample_time(inp, tokens, heads, nthreads)
    times = [oracle_sample_time(inp, tokens, heads, nthreads) for _ in range(args.steps)]
    tot = float(np.sum(times))
    equiv_tokens = tokens * heads / wl.HV          # tokens of the full-head workload
    value = equiv_tokens * args.steps / tot
    sample = (f"oracle (C fp64 token recurrence, OpenMP) on {heads} of {wl.HV} heads x first "
              f"{tokens} tokens of {wl.name} per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(inp, args),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads,
                             "kind": "oracle", "sample": sample,
                             "cpu": platform.processor() or platform.machine()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------
# replicas over ranks (one process per GPU; no exchange on the data path)
# ---------------------------------------------------------------------------------------

def replica_inputs(wl: kin.Workload, rank: int) -> kin.Inputs:
    """Rank `rank`'s own seeded copy of the workload (same shapes, different values)."""
    return kin.make_inputs(wl, seed=wl.seed + 1000 * rank)


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The slowest rank's figure (a time), identical on every rank."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's step time."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


def measure_decode(kb, kda, dev, steps, warmup, peak_gbs):
    """One decode step through kda_fused_recurrent_fwd (256 sequences x 1 token, 32 heads,
    K = V = 128, bf16): tokens/s and the HBM roofline of its state traffic (read h0 and
    write final_state, fp32, plus the token's q, k, v, g, beta, o)."""
    import torch
    inp = kin.make_inputs(kin.WORKLOADS["decode_bf16"])
    wl = inp.wl

    def up(x, dtype):
        if dtype == "bf16":
            return torch.from_numpy(kin.to_bf16_bits(x).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)

    q, k, v, g, b = (up(x, "bf16") for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    A_log, dt_bias, h0 = (up(x, "f32") for x in (inp.A_log, inp.dt_bias, inp.h0))
    o = torch.empty_like(v)
    fs = torch.empty_like(h0)
    p = kda.make_params(q, k, v, g, b, A_log=A_log, dt_bias=dt_bias, lower_bound=wl.lower_bound,
                        scale=inp.scale, initial_state=h0, final_state=fs, o=o)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    for _ in range(max(warmup, 3)):
        kb.raise_for(kb.kda_fused_recurrent_fwd(p, sh))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        kb.raise_for(kb.kda_fused_recurrent_fwd(p, sh))
    e1.record(stream)
    torch.cuda.synchronize()
    if kb.kda_get_device_status(sh) != 0:
        raise RuntimeError("device status flagged in the decode measurement")
    ms = e0.elapsed_time(e1) / steps
    ntok = wl.B * wl.T
    state = 2 * wl.B * wl.HV * wl.K * wl.V * 4
    per_tok = 2 * (2 * wl.H * wl.K + wl.HV * (2 * wl.V + wl.K + 1))   # q, k, v, g, beta, o
    nbytes = state + ntok * per_tok + 4 * wl.HV * (1 + wl.K)
    achieved = nbytes / (ms / 1e3) / 1e9
    return {"workload": "decode_bf16 (B=256 sequences x 1 token, H=HV=32, K=V=128)",
            "entry": "kda_fused_recurrent_fwd", "value": ntok / (ms / 1e3), "unit": "tokens/s",
            "ms_per_step": ms, "steps": steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak_gbs, "unit": "GB/s",
                         "frac": achieved / peak_gbs, "bytes_per_launch": float(nbytes)}}


# fp32 CUDA-core peak of one GB300: 152 SMs x 128 fp32 lanes x 2 flops (a fused multiply-add)
# per cycle at the maximum SM clock of 2070 MHz.
N_SM, FP32_LANES_PER_SM, MAX_SM_MHZ = 152, 128, 2070


def fp32_alu_peak_tflops(sm_mhz: float = MAX_SM_MHZ) -> float:
    return N_SM * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


def bwd_stage_flops(stage: str, C: int, K: int, V: int, nct: int, HV: int,
                    vprod: bool = False) -> float:
    """Algorithmic flops of one launch of a backward kernel over nct chunks x HV value heads
    (every chunk full; a fused multiply-add counts 2, an exponential 0): the dot products and
    triangular substitutions each kernel's stage computes.  With `vprod` the products over v
    (dAqk, dQg, dW, dKg, diag(S dS'^T)) run in their own stage, bwd_vprod, not in bwd_grads."""
    vp = V * C * (C + 1) + 6 * C * K * V + 2 * K * V
    per = {
        # Aqk and P over j <= i (2 FMA + 1 mul per channel); W, U forward substitution
        "bwd_prep": 5 * K * C * (C + 1) / 2 + 3 * (K + V) * C * (C - 1) / 2,
        # V_new = U - W S and S <- e^gamma S + Kg^T V_new
        "bwd_states": 4 * C * K * V,
        # dV_new = Kg dS' + Aqk^T dO (lower triangle); dS = Qg^T dO - W^T dV_new + ...
        "bwd_dstate": 2 * C * K * V + C * (C + 1) * V + 4 * C * K * V,
        # dAqk; dQg, dW, dKg; X, Y back substitution; A^T dA (strictly lower); the
        # e^(Gamma_i - Gamma_j) sums over rows and columns
        "bwd_grads": (vp + (K + V) * C * (C - 1)
                      + C * (C - 1) / 2 * (2 * V + 3 * K) + 5.5 * K * C * (C + 1)
                      - (vp if vprod else 0)),
        "bwd_vprod": vp,
    }.get(stage, 0.0)
    return float(per) * nct * HV


def measure_backward(kb, kda, dev, stream, inp, t, gate, steps):
    """The backward pass (kda_bwd) on the bench's workload with seeded incoming gradients:
    tokens/s, each kernel's time (the same passes stage by stage, an event after every
    kernel), and the fp32 CUDA-core roofline of the dominant kernel."""
    import torch
    wl = inp.wl
    rng = np.random.default_rng(wl.seed + 7)
    d_o = rng.standard_normal((wl.B, wl.T, wl.HV, wl.V), dtype=np.float32)
    if wl.dtype == "bf16":
        kin.round_to_bf16(d_o)
        d_o = torch.from_numpy(kin.to_bf16_bits(d_o).view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        d_o = torch.from_numpy(d_o).to(dev)
    st_shape = (inp.N, wl.HV, wl.K, wl.V)
    dht = torch.from_numpy(rng.standard_normal(st_shape, dtype=np.float32)).to(dev)
    f = kda.make_params(t["q"], t["k"], t["v"], t["g"], t["b"], A_log=t["A_log"],
                        dt_bias=t["dt_bias"], scale=inp.scale, initial_state=t["h0"],
                        cu_seqlens=t["cu"], cu_seqlens_cpu=t["cu_cpu"], chunk_size=wl.chunk_size,
                        **gate)
    f32 = dict(dtype=torch.float32, device=dev)
    outs = {"dq": torch.empty(t["q"].shape, **f32), "dk": torch.empty(t["k"].shape, **f32),
            "dv": torch.empty(t["v"].shape, **f32), "dg": torch.empty(t["g"].shape, **f32),
            "dbeta": torch.empty(t["b"].shape, **f32), "dh0": torch.empty(st_shape, **f32)}
    in_gate = wl.gate != kin.GATE_PREGATED
    if t["A_log"] is not None and in_gate:
        outs["dA_log"] = torch.empty((wl.HV,), **f32)
    if t["dt_bias"] is not None and in_gate:
        outs["ddt_bias"] = torch.empty(tuple(t["dt_bias"].shape), **f32)
    p = kb.kda_bwd_params()
    p.fwd = f
    p.d_o, p.d_final_state = d_o.data_ptr(), dht.data_ptr()
    for name, x in outs.items():
        setattr(p, name, x.data_ptr())
    kb.raise_for(kb.kda_bwd_check(p))
    ws = torch.empty(kb.kda_bwd_workspace_size(p), dtype=torch.uint8, device=dev)
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    sh = stream.cuda_stream
    nst = kb.kda_bwd_num_stages(p)
    names = [kb.kda_bwd_stage_name(p, i) for i in range(nst)]

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    whole = lambda: kb.raise_for(kb.kda_bwd(p, sh))
    first_ms = timed(whole, 1)                      # warm-up (and the size of a step)
    n = steps if first_ms < 2000 else 1
    ms = timed(whole, n)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(n)]
    s0 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s0.record(stream)
    for s_ in range(n):
        for i in range(nst):
            kb.raise_for(kb.kda_bwd_stage(p, sh, i))
            evs[s_][i].record(stream)
    torch.cuda.synchronize()
    stage_ms = np.zeros(nst)
    prev = s0
    for s_ in range(n):
        for i in range(nst):
            stage_ms[i] += prev.elapsed_time(evs[s_][i])
            prev = evs[s_][i]
    stage_ms /= n
    status = kb.kda_get_device_status(sh)
    if status != 0:
        raise RuntimeError(f"device status {status:#x} in the backward measurement")
    C = wl.chunk_size
    if inp.cu_seqlens is None:
        nct = wl.B * ((wl.T + C - 1) // C)
    else:
        nct = int(np.sum((np.diff(inp.cu_seqlens) + C - 1) // C))
    vprod = "bwd_vprod" in names
    flops = {nm: bwd_stage_flops(nm, wl.chunk_size, wl.K, wl.V, nct, wl.HV, vprod) for nm in names}
    kern = [i for i, nm in enumerate(names) if flops[nm] > 0]
    dom = max(kern, key=lambda i: stage_ms[i])
    peak = fp32_alu_peak_tflops()
    achieved = flops[names[dom]] / (stage_ms[dom] / 1e3) / 1e12
    total_flops = sum(flops.values())
    return {"workload": f"{wl.name} (the forward's workload), incoming gradients N(0, 1) seeded",
            "entry": "kda_bwd", "arithmetic": ("fp32 accumulation; CUDA cores, and tcgen05 with bf16 hi/lo operand "
                                               "splits in the state, state-gradient and v-product stages"),
            "value": inp.n_tokens / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "steps": n, "gpu_launches_per_step": int(kb.kda_bwd_num_launches(p)),
            "workspace_bytes": int(ws.numel()),
            "stages": {nm: float(x) for nm, x in zip(names, stage_ms)},
            "flops_per_step": total_flops,
            "tflops": total_flops / (ms / 1e3) / 1e12,
            "roofline": {"kernel": names[dom], "bound": "alu", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz",
                         "flops_per_launch": flops[names[dom]],
                         "ms_per_launch": float(stage_ms[dom]), "traffic": None}}


def config_of(inp: kin.Inputs, args):
    wl = inp.wl
    return {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "HV": wl.HV, "K": wl.K,
            "V": wl.V, "chunk_size": wl.chunk_size, "gate": {2: "safe", 1: "plain", 0: "pregated"}[wl.gate],
            "lower_bound": wl.lower_bound, "tokens_per_step": inp.n_tokens,
            "l2_flush": ("none: inputs per step (%.2f GB) exceed L2 (129 MB)" % (essential_bytes(inp) / 1e9)
                         if essential_bytes(inp) > 129e6 else
                         "none: inputs fit in L2, warm-cache figure"),
            "parallelism": f"replicas x{args.gpus}"}


# ---------------------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_bf16", choices=sorted(kin.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bwd-steps", type=int, default=3,
                    help="timed passes of the backward measurement (0: skip it)")
    ap.add_argument("--T", type=int, default=None,
                    help="override the workload's sequence length (small profiling captures)")
    args = ap.parse_args()
    wl = kin.WORKLOADS[args.workload]
    if args.T is not None:
        import dataclasses
        wl = dataclasses.replace(wl, T=args.T, name=f"{wl.name}_T{args.T}")

    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    import kimi_delta_attention_gate_gb300 as kda
    from kimi_delta_attention_gate_gb300 import _binding as kb
    from kimi_delta_attention_gate_gb300 import build as kbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if dist is not None:
            dist.barrier()

    if rank == 0:
        kbuild.build()
    barrier()
    kb.load()

    # Inputs: each rank its own replica (seed offset by rank), uploaded once.
    inp = replica_inputs(wl, rank)
    dev = torch.device("cuda", local_rank)

    def up(x, dtype):
        if x is None:
            return None
        if dtype == "bf16":
            return torch.from_numpy(kin.to_bf16_bits(x).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)

    q, k, v, g, b = (up(x, wl.dtype) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    A_log, dt_bias, h0 = (up(x, "f32") for x in (inp.A_log, inp.dt_bias, inp.h0))
    cu = cu_cpu = None
    if inp.cu_seqlens is not None:
        cu_cpu = torch.from_numpy(inp.cu_seqlens)
        cu = cu_cpu.to(dev)
    N = inp.N
    o = torch.zeros((wl.B, wl.T, wl.HV, wl.V), dtype=v.dtype, device=dev)
    fs = torch.empty((N, wl.HV, wl.K, wl.V), dtype=torch.float32, device=dev)
    gate = {} if wl.gate == kin.GATE_PLAIN else ({"use_gate_in_kernel": False}
                                                  if wl.gate == kin.GATE_PREGATED
                                                  else {"lower_bound": wl.lower_bound})
    p = kda.make_params(q, k, v, g, b, A_log=A_log, dt_bias=dt_bias, scale=inp.scale,
                        initial_state=h0, final_state=fs, o=o, cu_seqlens=cu, cu_seqlens_cpu=cu_cpu,
                        chunk_size=wl.chunk_size, **gate)
    kb.raise_for(kb.kda_fwd_check(p))
    ws = torch.empty(max(kb.kda_fwd_workspace_size(p), 1), dtype=torch.uint8, device=dev)
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    nst = kb.kda_fwd_num_stages(p)
    names = [kb.kda_fwd_stage_name(p, i) for i in range(nst)]
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    n_launch = kb.kda_fwd_num_launches(p)

    def step():  # one forward pass through the C ABI (the pipelined schedule, if any)
        kb.raise_for(kb.kda_fwd(p, sh))

    def stage_step(evs):  # the same pass stage by stage, an event after every kernel
        for i in range(nst):
            kb.raise_for(kb.kda_fwd_stage(p, sh, i))
            evs[i].record(stream)

    sampler = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else local_rank)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = kb.kda_get_device_status(sh)
    if status != 0:
        raise RuntimeError(f"device status {status:#x} after warm-up")

    # Timed region: K forward passes on the launching stream, CUDA events around them.
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start.record(stream)
    for s_ in range(args.steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.time()
    clocks = sampler.stop(t_wall0, t_wall1)
    total_ms = start.elapsed_time(stop)
    # Per-kernel durations (roofline of the dominant kernel): the same K passes stage by
    # stage, each kernel alone on the stream between two events.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(args.steps)]
    s0 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s0.record(stream)
    for s_ in range(args.steps):
        stage_step(evs[s_])
    torch.cuda.synchronize()
    stage_ms = np.zeros(nst)
    prev = s0
    for s_ in range(args.steps):
        for i in range(nst):
            stage_ms[i] += prev.elapsed_time(evs[s_][i])
            prev = evs[s_][i]
    stage_ms /= args.steps
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(inp.n_tokens, world, ms_per_step)
    status = kb.kda_get_device_status(sh)
    if status != 0:
        raise RuntimeError(f"device status {status:#x} after the timed region")

    # End to end through the public API on host buffers: kda_fwd_host copies every input in
    # from pinned host memory (the token rows segment by segment, overlapping the kernels) and
    # o / final_state back out.  For context the same pass as three serial phases (copy in,
    # kda_fwd, copy out) is timed too.
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 10))
    pin = lambda t: None if t is None else t.cpu().pin_memory()
    hq, hk, hv_, hg, hb = (pin(x) for x in (q, k, v, g, b))
    hA, hdt, hh0 = (pin(x) for x in (A_log, dt_bias, h0))
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hfs = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
    host_in = [x for x in (hq, hk, hv_, hg, hb, hA, hdt, hh0, cu_cpu) if x is not None]
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = ho.numel() * ho.element_size() + hfs.numel() * hfs.element_size()
    hp = kda.make_params(hq, hk, hv_, hg, hb, A_log=hA, dt_bias=hdt, scale=inp.scale,
                         initial_state=hh0, final_state=hfs, o=ho, cu_seqlens=cu_cpu,
                         cu_seqlens_cpu=cu_cpu, chunk_size=wl.chunk_size, **gate)
    hp.cu_seqlens = None
    arena = torch.empty(kb.kda_fwd_host_arena_size(hp), dtype=torch.uint8, device=dev)

    def e2e_step():
        kb.raise_for(kb.kda_fwd_host(hp, arena.data_ptr(), arena.numel(), sh))

    dq, dk, dv, dg, db = (torch.empty_like(x) for x in (q, k, v, g, b))

    def serial_step():
        for d, h in ((dq, hq), (dk, hk), (dv, hv_), (dg, hg), (db, hb)):
            d.copy_(h, non_blocking=True)
        oo, ff = kda.kda_fwd(dq, dk, dv, dg, db, A_log=A_log, dt_bias=dt_bias, scale=inp.scale,
                             initial_state=h0, cu_seqlens=cu, cu_seqlens_cpu=cu_cpu,
                             chunk_size=wl.chunk_size, workspace=ws, o=o, final_state=fs,
                             stream=stream, **gate)
        ho.copy_(oo, non_blocking=True)
        hfs.copy_(ff, non_blocking=True)

    def time_steps(fn, warm=1):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)

    serial_ms = time_steps(serial_step)
    # three windows of e2e_steps steps each, the median window reported (all three listed): the
    # host side of this path (pinned copies, the host thread issuing them) shares the machine,
    # and one stall in a single window would otherwise stand for the whole measurement
    e2e_windows = [time_steps(e2e_step, warm=3 if w == 0 else 1) for w in range(3)]
    e2e_ms = sorted(e2e_windows)[1]
    status = kb.kda_get_device_status(sh)
    if status != 0:
        raise RuntimeError(f"device status {status:#x} after the end-to-end passes")
    e2e_value = job_throughput(inp.n_tokens, world, e2e_ms)
    # The host link's own rates (one 512 MiB pinned copy each way): the step's bytes at these
    # rates, the two directions overlapping, are the floor of the end-to-end time.
    link_buf = torch.empty(1 << 29, dtype=torch.uint8).pin_memory()
    link_dev = torch.empty(1 << 29, dtype=torch.uint8, device=dev)
    link = {}
    for name, fn in (("h2d", lambda: link_dev.copy_(link_buf, non_blocking=True)),
                     ("d2h", lambda: link_buf.copy_(link_dev, non_blocking=True))):
        fn()
        torch.cuda.synchronize()
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(stream)
        for _ in range(3):
            fn()
        l1.record(stream)
        torch.cuda.synchronize()
        link[name] = 3 * link_buf.numel() / (l0.elapsed_time(l1) / 1e3) / 1e9
    del link_buf, link_dev
    link_floor_ms = 1e3 * max(h2d / (link["h2d"] * 1e9), d2h / (link["d2h"] * 1e9))

    # Roofline of the step by the method's byte model: q, k, v, g, beta read once, o written
    # once, plus the states and the gate parameters (intermediates are not counted), over the
    # device time of one step; the step is HBM-bound (arithmetic intensity below the ridge).
    peaks, peak_kind = load_peaks()
    peak = float(peaks["hbm_gbs"])
    ess = essential_bytes(inp)
    flops = dense_flops(inp)
    t_roof = max(ess / (peak * 1e9), flops / (float(peaks["bf16_tflops"]) * 1e12))
    stage_traffic = [profiled_traffic(n, wl.name) for n in names]
    roofline = {"kernel": "kda_fwd step (all kernels)", "bound": "hbm",
                "achieved": ess / (ms_per_step / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                "frac": ess / (ms_per_step / 1e3) / 1e9 / peak, "peak_source": peak_kind,
                "bytes_per_step": ess, "ms_per_step": ms_per_step,
                "traffic": (None if any(t is None for t in stage_traffic)
                            else float(sum(stage_traffic))),
                "dense_flops": flops, "tflops": flops / (ms_per_step / 1e3) / 1e12,
                "roofline_ms": 1e3 * t_roof, "frac_of_roofline_time": (1e3 * t_roof) / ms_per_step}
    # Each kernel against the method bytes it owns (the inputs it reads and outputs it
    # writes, intermediates excluded), timed alone stage by stage; "traffic" is its DRAM bytes
    # per launch from the committed ncu summary (null once its code changed), and
    # "traffic_over_own_bytes" the waste ratio.
    stages = {}
    for i, n in enumerate(names):
        own = own_bytes(n, inp)
        ach = own / (stage_ms[i] / 1e3) / 1e9
        stages[n] = {"ms": float(stage_ms[i]), "own_bytes": own, "achieved_gbs": ach,
                     "frac": ach / peak, "traffic": stage_traffic[i],
                     "traffic_over_own_bytes": (None if stage_traffic[i] is None or own <= 0
                                                else stage_traffic[i] / own)}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.dtype, "data": "synthetic (seeded PCG64, shapes and distributions of the workload)",
            "config": config_of(inp, args), "roofline": roofline, "stages": stages,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
                    "window_ms": e2e_windows, "steps_per_window": e2e_steps,
                    "entry": "kda_fwd_host", "serial_copy_run_copy_ms": serial_ms,
                    "link_h2d_gbs": link["h2d"], "link_d2h_gbs": link["d2h"],
                    "link_floor_ms": link_floor_ms},
            "gpu_launches": int(n_launch * args.steps), "clocks": clocks,
            "kernel_source_sha": kernel_source_hash()}

    if rank == 0 and world == 1:
        line["decode"] = measure_decode(kb, kda, dev, args.steps, args.warmup, peak)
    if rank == 0 and world == 1 and args.bwd_steps > 0:
        # Last on the GPU, and on its own: a failure here leaves the forward's figures as
        # they are.
        try:
            tens = dict(q=q, k=k, v=v, g=g, b=b, A_log=A_log, dt_bias=dt_bias, h0=h0, cu=cu,
                        cu_cpu=cu_cpu)
            line["backward"] = measure_backward(kb, kda, dev, stream, inp, tens, gate,
                                                args.bwd_steps)
        except Exception as exc:  # noqa: BLE001
            line["backward"] = {"error": f"{type(exc).__name__}: {exc}"[:400]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        nthreads = oracle.max_threads()
        tokens, heads = cpu_sample_plan(inp, args.cpu_seconds, nthreads)
        secs = oracle_sample_time(inp, tokens, heads, nthreads)
        line["cpu_baseline"] = {
            "value": tokens * heads / wl.HV / secs, "unit": "tokens/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"{heads} of {wl.HV} heads x first {tokens} tokens of {wl.name} "
                      f"({secs:.1f} s, C fp64 token recurrence, OpenMP)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
