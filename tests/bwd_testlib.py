"""Helpers of the backward tests: seeded upstream gradients, the oracle's gradients of the
same inputs, the host emulation of the backward stage bodies, and the comparison."""
from __future__ import annotations

import os
import shutil
import subprocess

import numpy as np

from kimi_delta_attention_gate_gb300 import inputs as kin

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EMU_SRC = os.path.join(ROOT, "tests", "emulation", "kda_bwd_emu.cpp")
GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias", "dh0")

# rel-L2 bounds of each gradient against the fp64 oracle.  The kernels compute in fp32 from
# inputs that are exact in fp32 (bf16 widens exactly), so only fp32 rounding separates them.
# Most gradients are short chains of dot products over K, V and the chunk (relative error a
# few 1e-7 measured on the emulation); 1e-4, the fp32 forward's bound, leaves a wide margin.
# The gate gradients pass through a cancellation that the method itself contains: dGamma is a
# row sum minus a column sum of the same e^(Gamma_i - Gamma_j) terms, then summed in reverse
# over the chunk, and dA_log / ddt_bias sum dg over the tokens.  With the safe gate near its
# bound this costs about two decimal digits (measured: dg 3e-5, dA_log 1e-4, ddt_bias 2.4e-4);
# those three get 1e-3.
REL_L2 = 1e-4
REL_L2_GATE = 1e-3
GATE_GRADS = ("dg", "dA_log", "ddt_bias")
# A gradient can be exactly zero in exact arithmetic while its terms are O(1) (the gate's
# gradient with no state to decay: one-token sequences without h0), where fp32 leaves
# rounding noise and a relative bound means nothing.  So the bound on |got - ref|_2 is
# REL_L2 |ref|_2 + ABS_PER_ELEM sqrt(n): 1e-7 per element is the fp32 rounding of the O(1)
# terms' sums (unit roundoff 6e-8), far below REL_L2 |ref| wherever the gradient is not zero.
ABS_PER_ELEM = 1e-7


def workload(name="bwd", B=2, T=150, H=1, HV=2, K=32, V=16, C=64, dtype="f32",
             gate=kin.GATE_SAFE, seed=7, **kw) -> kin.Workload:
    """A small workload for the backward tests (every gate mode with its usual inputs)."""
    lb = -5.0 if gate == kin.GATE_SAFE else None
    kw.setdefault("h0_std", 0.3)
    if gate == kin.GATE_PLAIN:
        kw.setdefault("a_log_mean", -1.0)
        kw.setdefault("a_log_std", 0.5)
    if gate == kin.GATE_PREGATED:
        kw.setdefault("has_a_log", False)
        kw.setdefault("has_dt_bias", False)
    return kin.Workload(name, B=B, T=T, H=H, HV=HV, K=K, V=V, chunk_size=C, dtype=dtype, gate=gate,
                        lower_bound=lb, seed=seed, **kw)


def random_case(seed: int):
    """A seeded random configuration (shapes, gate, dtype, varlen, options) and its inputs, for
    shape sweeps: returns (inputs, options for the backward)."""
    r = np.random.default_rng(seed)
    C = int(r.choice([32, 64]))
    H = int(r.integers(1, 3))
    G = int(r.choice([1, 1, 2, 3]))
    K = int(r.choice([8, 16, 24, 32, 48, 64]))
    V = int(r.choice([8, 16, 40, 64, 72]))
    gate = int(r.choice([kin.GATE_SAFE, kin.GATE_PLAIN, kin.GATE_PREGATED]))
    dtype = str(r.choice(["f32", "bf16"]))
    varlen = bool(r.random() < 0.4)
    B = 1 if varlen else int(r.integers(1, 4))
    T = int(r.integers(1, 3 * C + 5))
    kw = dict(h0_std=None if r.random() < 0.3 else 0.2)
    if varlen:
        kw.update(varlen_n=int(r.integers(1, 5)), varlen_max_len=max(1, T // 2))
        T = max(T, kw["varlen_n"] * kw["varlen_max_len"])
    if gate == kin.GATE_SAFE and r.random() < 0.3:
        kw["has_a_log"] = False
    wl = workload(f"rand{seed}", B=B, T=T, H=H, HV=H * G, K=K, V=V, C=C, dtype=dtype, gate=gate,
                  seed=seed, **kw)
    inp = kin.make_inputs(wl)
    if gate == kin.GATE_PREGATED:
        pregate(inp)
    opts = dict(allow_neg_eigval=bool(r.random() < 0.3), state_v_first=bool(r.random() < 0.3))
    if opts["state_v_first"] and inp.h0 is not None:
        inp.h0 = np.ascontiguousarray(np.swapaxes(inp.h0, -1, -2))
    return inp, opts


def pregate(inp: kin.Inputs) -> kin.Inputs:
    """A log decay in (-1, 0] for the pre-gated mode (g is used as it is)."""
    inp.g = -np.abs(inp.g) * np.float32(0.5)
    if inp.wl.dtype == "bf16":
        kin.round_to_bf16(inp.g)
    return inp


def upstream(inp: kin.Inputs, seed: int, state_v_first: bool = False):
    """Seeded gradients of o ([B,T,HV,V], in the input dtype's values) and of final_state
    ([N,HV,K,V] fp32, or [N,HV,V,K])."""
    wl = inp.wl
    rng = np.random.default_rng(seed)
    d_o = rng.standard_normal((wl.B, wl.T, wl.HV, wl.V), dtype=np.float32)
    if wl.dtype == "bf16":
        kin.round_to_bf16(d_o)
    dfs = rng.standard_normal((inp.N, wl.HV, wl.K, wl.V), dtype=np.float32)
    if state_v_first:
        dfs = np.ascontiguousarray(np.swapaxes(dfs, -1, -2))
    return d_o, dfs


def oracle_grads(inp: kin.Inputs, d_o, dfs, *, allow_neg_eigval=False, state_v_first=False,
                 chunk_form=False, heads=None) -> dict:
    """The oracle's gradients (fp64) for the inputs of ``inp`` (h0 and dfs in the layout that
    ``state_v_first`` names): the autograd form, or with ``chunk_form`` the chunked form.
    ``heads``: only these value heads (whole groups only when HV > H), the gradients of
    the other heads left out."""
    from oracle import backward as ob
    wl = inp.wl
    lb = wl.lower_bound if wl.gate == kin.GATE_SAFE else None
    fn = ob.chunk_bwd_np if chunk_form else ob.bwd
    extra = dict(chunk_size=wl.chunk_size) if chunk_form else {}
    f64 = lambda x: None if x is None else np.asarray(x, np.float64)
    q, k, v, g, b, A_log, dt, h0 = (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.A_log, inp.dt_bias,
                                    inp.h0)
    if heads is not None:
        heads = np.asarray(heads)
        assert wl.G == 1, "sample heads with HV == H only"
        q, k = q[:, :, heads], k[:, :, heads]
        v, g, b, d_o = v[:, :, heads], g[:, :, heads], b[:, :, heads], d_o[:, :, heads]
        A_log = None if A_log is None else A_log[heads]
        dt = None if dt is None else dt.reshape(wl.HV, wl.K)[heads].reshape(-1)
        h0 = None if h0 is None else h0[:, heads]
        dfs = None if dfs is None else dfs[:, heads]
    return fn(f64(q), f64(k), f64(v), f64(g), f64(b), f64(d_o), f64(dfs),
              A_log=f64(A_log), dt_bias=f64(dt), gate_mode=wl.gate, lower_bound=lb,
              scale=inp.scale, qk_l2norm=True, beta_sigmoid=True, allow_neg_eigval=allow_neg_eigval,
              initial_state=f64(h0), cu_seqlens=inp.cu_seqlens,
              transpose_state_layout=state_v_first, **extra)


def build_emulator(out_dir: str) -> str:
    """Compile the host emulation of the backward stage bodies with AddressSanitizer and
    UndefinedBehaviorSanitizer; returns the executable's path."""
    gxx = shutil.which("g++")
    if gxx is None:
        raise RuntimeError("g++ not found")
    exe = os.path.join(out_dir, "kda_bwd_emu")
    cmd = [gxx, "-std=c++17", "-O1", "-g", "-fsanitize=address,undefined", "-fno-omit-frame-pointer",
           "-fno-sanitize-recover=all", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(ROOT, "kimi_delta_attention_gate_gb300", "csrc"), EMU_SRC, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"emulator build failed:\n{r.stdout}\n{r.stderr}")
    return exe


def _raw(x: np.ndarray, dtype: str) -> bytes:
    if dtype == "bf16":
        return kin.to_bf16_bits(x).tobytes()
    return np.ascontiguousarray(x, np.float32).tobytes()


def run_emulator(exe: str, workdir: str, inp: kin.Inputs, d_o, dfs, *, seed=0,
                 allow_neg_eigval=False, state_v_first=False, want=GRADS) -> dict:
    """The backward stage bodies on the host: returns {gradient name: fp64 array} (the
    optional ones only when requested and defined) and the device status bits."""
    wl = inp.wl
    os.makedirs(workdir, exist_ok=True)
    has = dict(A_log=inp.A_log is not None, dt_bias=inp.dt_bias is not None, h0=inp.h0 is not None,
               cu_seqlens=inp.cu_seqlens is not None, d_final_state=dfs is not None)
    in_gate = wl.gate != kin.GATE_PREGATED
    spec = dict(B=wl.B, T=wl.T, H=wl.H, HV=wl.HV, K=wl.K, V=wl.V, chunk_size=wl.chunk_size,
                in_dtype=0 if wl.dtype == "bf16" else 1, gate_mode=wl.gate,
                lower_bound=wl.lower_bound if wl.gate == kin.GATE_SAFE else 0.0,
                scale=repr(float(np.float32(inp.scale))), qk_l2norm=1, beta_sigmoid=1,
                N=inp.N, allow_neg_eigval=int(allow_neg_eigval), state_v_first=int(state_v_first),
                seed=seed, **{f"has_{k}": int(v) for k, v in has.items()},
                want_dA_log=int("dA_log" in want and has["A_log"] and in_gate),
                want_ddt_bias=int("ddt_bias" in want and has["dt_bias"] and in_gate),
                want_dh0=int("dh0" in want))
    with open(os.path.join(workdir, "spec.txt"), "w") as f:
        for key, val in spec.items():
            f.write(f"{key} {val}\n")
    files = dict(q=_raw(inp.q, wl.dtype), k=_raw(inp.k, wl.dtype), v=_raw(inp.v, wl.dtype),
                 g=_raw(inp.g, wl.dtype), beta=_raw(inp.beta, wl.dtype), d_o=_raw(d_o, wl.dtype))
    if has["A_log"]:
        files["A_log"] = _raw(inp.A_log, "f32")
    if has["dt_bias"]:
        files["dt_bias"] = _raw(inp.dt_bias, "f32")
    if has["h0"]:
        files["h0"] = _raw(inp.h0, "f32")
    if has["cu_seqlens"]:
        files["cu_seqlens"] = np.ascontiguousarray(inp.cu_seqlens, np.int64).tobytes()
    if has["d_final_state"]:
        files["d_final_state"] = _raw(dfs, "f32")
    for name, data in files.items():
        with open(os.path.join(workdir, name + ".bin"), "wb") as f:
            f.write(data)
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=0:abort_on_error=0",
               UBSAN_OPTIONS="print_stacktrace=1")
    r = subprocess.run([exe, workdir], capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        raise AssertionError(f"emulator failed ({r.returncode}):\n{r.stdout}\n{r.stderr[-4000:]}")
    shapes = dict(dq=inp.q.shape, dk=inp.k.shape, dv=inp.v.shape, dg=inp.g.shape,
                  dbeta=inp.beta.shape, dA_log=(wl.HV,), ddt_bias=(wl.HV * wl.K,),
                  dh0=(inp.N, wl.HV, wl.V, wl.K) if state_v_first else (inp.N, wl.HV, wl.K, wl.V))
    out = {}
    for name in GRADS:
        path = os.path.join(workdir, f"out_{name}.bin")
        if os.path.exists(path):
            out[name] = np.fromfile(path, np.float32).reshape(shapes[name]).astype(np.float64)
    with open(os.path.join(workdir, "out_status.txt")) as f:
        out["status"] = int(f.read().split()[0])
    return out


def rel_l2(got, ref) -> float:
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


def assert_grads_close(got: dict, ref: dict, names=GRADS):
    """Every gradient in ``names`` that ``ref`` defines is present in ``got``, finite, and
    within its rel-L2 bound; returns the errors."""
    errs = {}
    for name in names:
        if ref.get(name) is None:
            continue
        assert name in got, f"{name} missing"
        g = got[name]
        assert g.shape == ref[name].shape, (name, g.shape, ref[name].shape)
        assert np.all(np.isfinite(g)), f"{name}: non-finite values"
        errs[name] = rel_l2(g, ref[name])
        tol = REL_L2_GATE if name in GATE_GRADS else REL_L2
        err = float(np.linalg.norm(g - ref[name]))
        bound = tol * float(np.linalg.norm(ref[name])) + ABS_PER_ELEM * np.sqrt(g.size)
        assert err <= bound, (f"{name}: |got - ref| {err:.3e} > {bound:.3e} "
                              f"(rel-L2 {errs[name]:.3e}, bound {tol:.0e} + {ABS_PER_ELEM:.0e}/elem)")
    return errs


def run_gpu_bwd(inp: kin.Inputs, d_o, dfs, *, allow_neg_eigval=False, state_v_first=False,
                heads=None) -> dict:
    """kda_bwd (the C ABI through the package's wrapper) on the GPU: {gradient: fp64 array};
    with ``heads`` (HV == H) only those value heads' gradients are copied back."""
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    from kda_testlib import f32_device, gate_kwargs, to_device
    wl = inp.wl
    q, k, v, g, b, do = (to_device(x, wl.dtype) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta, d_o))
    cu = None if inp.cu_seqlens is None else torch.from_numpy(inp.cu_seqlens).cuda()
    cu_cpu = None if inp.cu_seqlens is None else torch.from_numpy(inp.cu_seqlens)
    res = kda.kda_bwd(q, k, v, g, b, do, dht=f32_device(dfs), A_log=f32_device(inp.A_log),
                      dt_bias=f32_device(inp.dt_bias), scale=inp.scale,
                      initial_state=f32_device(inp.h0), cu_seqlens=cu, cu_seqlens_cpu=cu_cpu,
                      chunk_size=wl.chunk_size, allow_neg_eigval=allow_neg_eigval,
                      transpose_state_layout=state_v_first, **gate_kwargs(wl))
    torch.cuda.synchronize()
    status = kda.kda_get_device_status(0)
    assert status == 0, f"device status {status:#x}"
    out = {}
    for name, t in zip(GRADS, res):
        if t is None:
            continue
        if heads is not None:
            idx = torch.as_tensor(np.asarray(heads), device=t.device)
            if name == "ddt_bias":
                t = t.reshape(wl.HV, wl.K).index_select(0, idx).reshape(-1)
            elif name == "dA_log":
                t = t.index_select(0, idx)
            elif name == "dh0":
                t = t.index_select(1, idx)
            else:
                t = t.index_select(2, idx)
        out[name] = t.cpu().double().numpy()
    return out
