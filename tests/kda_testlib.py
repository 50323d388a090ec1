"""Helpers shared by the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI, run the oracle on the same bits, compare."""
from __future__ import annotations

import numpy as np

import oracle
from kimi_delta_attention_gate_gb300 import inputs as kin

# Tolerances on o and final_state against the fp64 oracle.
TOL = {
    "bf16": dict(rel_l2=5e-3, max_abs=3e-2),
    "f32": dict(rel_l2=1e-4, max_abs=None),
}


def to_device(x: np.ndarray, dtype: str, device="cuda"):
    import torch
    if dtype == "bf16":
        bits = kin.to_bf16_bits(x).view(np.int16)
        return torch.from_numpy(bits).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)


def f32_device(x, device="cuda"):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)


def gate_kwargs(wl: kin.Workload):
    if wl.gate == kin.GATE_PREGATED:
        return dict(use_gate_in_kernel=False)
    if wl.gate == kin.GATE_SAFE:
        return dict(use_gate_in_kernel=True, lower_bound=wl.lower_bound)
    return dict(use_gate_in_kernel=True)


def run_gpu(inp: kin.Inputs, chunk_size=None, stream=None, workspace=None, **opts):
    """The CUDA path on ``inp``; returns (o, final_state) as float64 numpy arrays.  ``opts``:
    allow_neg_eigval, transpose_state_layout (inp.h0 then already in that layout)."""
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    wl = inp.wl
    dev = "cuda"
    q, k, v, g, b = (to_device(x, wl.dtype, dev) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    cu = None if inp.cu_seqlens is None else torch.from_numpy(inp.cu_seqlens).to(dev)
    cu_cpu = None if inp.cu_seqlens is None else torch.from_numpy(inp.cu_seqlens)
    o, fs = kda.kda_fwd(q, k, v, g, b, A_log=f32_device(inp.A_log), dt_bias=f32_device(inp.dt_bias),
                        scale=inp.scale, initial_state=f32_device(inp.h0), output_final_state=True,
                        cu_seqlens=cu, cu_seqlens_cpu=cu_cpu,
                        chunk_size=chunk_size or wl.chunk_size, stream=stream, workspace=workspace,
                        **gate_kwargs(wl), **opts)
    torch.cuda.synchronize()
    status = kda.kda_get_device_status(0)
    assert status == 0, f"device status {status:#x}"
    return o.float().cpu().double().numpy(), fs.cpu().double().numpy()


def run_oracle(inp: kin.Inputs, heads=None, nthreads=0, **opts):
    """The oracle on ``inp`` (optionally only the value heads ``heads``); ``opts`` as run_gpu."""
    wl = inp.wl
    q, k, v, g, b = inp.q, inp.k, inp.v, inp.g, inp.beta
    A_log, dt, h0 = inp.A_log, inp.dt_bias, inp.h0
    if heads is not None:
        heads = np.asarray(heads)
        kh = np.unique(heads // wl.G)
        assert wl.G == 1 or len(kh) == len(heads), "sample whole GVA groups only with G == 1"
        q, k = q[:, :, heads // wl.G], k[:, :, heads // wl.G]
        v, g, b = v[:, :, heads], g[:, :, heads], b[:, :, heads]
        A_log = None if A_log is None else A_log[heads]
        dt = None if dt is None else dt.reshape(wl.HV, wl.K)[heads].reshape(-1)
        h0 = None if h0 is None else h0[:, heads]
    lb = wl.lower_bound if wl.gate == kin.GATE_SAFE else None
    return oracle.fwd(q, k, v, g, b, A_log=A_log, dt_bias=dt, gate_mode=wl.gate, lower_bound=lb,
                      scale=inp.scale, qk_l2norm=True, beta_sigmoid=True, initial_state=h0,
                      cu_seqlens=inp.cu_seqlens, nthreads=nthreads, **opts)


def errors(got: np.ndarray, ref: np.ndarray):
    diff = got - ref
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30))
    mx = float(np.max(np.abs(diff))) if diff.size else 0.0
    return rel, mx


def assert_close(got, ref, dtype: str, what: str):
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    rel, mx = errors(got, ref)
    tol = TOL[dtype]
    assert rel <= tol["rel_l2"], f"{what}: rel-L2 {rel:.3e} > {tol['rel_l2']:.0e} (max-abs {mx:.3e})"
    if tol["max_abs"] is not None:
        assert mx <= tol["max_abs"], f"{what}: max-abs {mx:.3e} > {tol['max_abs']:.0e}"
    return rel, mx


def run_gpu_stages(inp: kin.Inputs):
    """The CUDA path on ``inp`` through the per-stage entry point: every stage is one
    launch over the whole chunk range, in order, on the current stream."""
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    from kimi_delta_attention_gate_gb300 import _binding as kb
    wl = inp.wl
    q, k, v, g, b = (to_device(x, wl.dtype) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    cu = None if inp.cu_seqlens is None else torch.from_numpy(inp.cu_seqlens).cuda()
    cu_cpu = None if inp.cu_seqlens is None else torch.from_numpy(inp.cu_seqlens)
    # o starts as NaN: every row, padding included, must be written by the stages
    o = torch.full((wl.B, wl.T, wl.HV, wl.V), float("nan"), dtype=v.dtype, device="cuda")
    fs = torch.empty((inp.N, wl.HV, wl.K, wl.V), dtype=torch.float32, device="cuda")
    A_log, dt_bias, h0 = f32_device(inp.A_log), f32_device(inp.dt_bias), f32_device(inp.h0)
    p = kda.make_params(q, k, v, g, b, A_log=A_log, dt_bias=dt_bias, scale=inp.scale,
                        initial_state=h0, final_state=fs, o=o, cu_seqlens=cu,
                        cu_seqlens_cpu=cu_cpu, chunk_size=wl.chunk_size, **gate_kwargs(wl))
    ws = torch.empty(max(kb.kda_fwd_workspace_size(p), 1), dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    sh = torch.cuda.current_stream().cuda_stream
    for i in range(kb.kda_fwd_num_stages(p)):
        kb.raise_for(kb.kda_fwd_stage(p, sh, i))
    torch.cuda.synchronize()
    assert kb.kda_get_device_status(sh) == 0
    return o.float().cpu().double().numpy(), fs.cpu().double().numpy()


def to_pinned(x: np.ndarray, dtype: str):
    """``x`` as a page-locked host tensor in the path's input type."""
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(kin.to_bf16_bits(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, np.float32))
    return t.pin_memory()


def run_gpu_host(inp: kin.Inputs, sentinel=7.0, h_out_chunks=0, **opts):
    """The host-buffer entry point on ``inp``: every tensor in pinned host memory, the device
    arena pre-filled with NaN bits.  Host o starts at ``sentinel`` so that rows no sequence
    covers can be checked set to zero.  Returns (o, final_state[, h_out]) as float64 numpy
    arrays."""
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    wl = inp.wl
    q, k, v, g, b = (to_pinned(x, wl.dtype) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    pin32 = (lambda x: None if x is None else
             torch.from_numpy(np.ascontiguousarray(x, np.float32)).pin_memory())
    o = torch.full((wl.B, wl.T, wl.HV, wl.V), sentinel, dtype=v.dtype).pin_memory()
    st = (wl.V, wl.K) if opts.get("transpose_state_layout") else (wl.K, wl.V)
    fs = torch.zeros((inp.N, wl.HV) + st, dtype=torch.float32).pin_memory()
    hs = (torch.zeros((h_out_chunks, wl.HV) + st, dtype=torch.float32).pin_memory()
          if h_out_chunks else None)
    cu = None if inp.cu_seqlens is None else torch.from_numpy(inp.cu_seqlens)
    kw = dict(A_log=pin32(inp.A_log), dt_bias=pin32(inp.dt_bias), scale=inp.scale,
              initial_state=pin32(inp.h0), cu_seqlens=cu, chunk_size=wl.chunk_size,
              **gate_kwargs(wl), **opts)
    from kimi_delta_attention_gate_gb300 import _binding as kb
    p = kda.make_params(q, k, v, g, b, o=o, final_state=fs, h_out=hs, cu_seqlens_cpu=cu, **kw)
    need = kb.kda_fwd_host_arena_size(p)
    assert need > 0, kb.kda_last_error()
    arena = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    kda.kda_fwd_host(q, k, v, g, b, o=o, final_state=fs, h_out=hs, arena=arena, **kw)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status(0) == 0
    out = (o.float().double().numpy(), fs.double().numpy())
    return out + ((hs.double().numpy(),) if hs is not None else ())
