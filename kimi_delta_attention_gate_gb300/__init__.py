"""GB300 (sm_103a) chunk-parallel Kimi Delta Attention: forward pass and its backward.

``kda_fwd`` takes PyTorch CUDA tensors, allocates the outputs and the
workspace with PyTorch, fills the C parameter block and calls the C ABI
(``include/kda.h``).  Every step of the computation runs in the library's own
CUDA kernels; there is no CPU or PyTorch fallback.

The keyword arguments follow FLA's ``chunk_kda`` ("FLA-KDA engineering notes",
section 2.2; "Reading Notes: Implementation Notes for KDA in FLA", forward
entry): ``use_gate_in_kernel`` selects the in-kernel gate, and with it
``lower_bound`` given selects the safe gate
``lower_bound * sigmoid(exp(A_log) * (g + dt_bias))``, otherwise the plain gate
``-exp(A_log) * softplus(g + dt_bias)``.
"""
from __future__ import annotations

from typing import Optional

from . import _binding
from ._binding import (KDA_BF16, KDA_F32, KDA_GATE_PLAIN, KDA_GATE_PREGATED, KDA_GATE_SAFE,
                       KdaError, kda_abi_version, kda_bwd_params, kda_fwd_params,
                       kda_get_device_status, kda_last_error, kda_status_string)

__all__ = ["kda_fwd", "kda_bwd", "kda_fwd_host", "kda_fused_recurrent_fwd", "kda_fwd_workspace_size",
           "make_params", "KdaError", "kda_get_device_status", "kda_last_error", "kda_status_string", "kda_abi_version", "KDA_GATE_SAFE",
           "KDA_GATE_PLAIN", "KDA_GATE_PREGATED", "KDA_BF16", "KDA_F32"]


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _int64_seqlens(cu_seqlens, cu_seqlens_cpu):
    """int64 copies of the sequence offsets (FLA callers often hold them as int32) and a host
    copy when only the device tensor is given; the caller keeps the returned tensors alive
    while its launches are in flight (they are bound in the parameter block)."""
    import torch
    if cu_seqlens is not None:
        cu_seqlens = cu_seqlens.to(torch.int64).contiguous()
        if cu_seqlens_cpu is None:
            cu_seqlens_cpu = cu_seqlens.to("cpu")
    if cu_seqlens_cpu is not None:
        cu_seqlens_cpu = cu_seqlens_cpu.to(torch.int64).contiguous()
    return cu_seqlens, cu_seqlens_cpu


def _gate_mode(use_gate_in_kernel: bool, safe_gate: Optional[bool], lower_bound) -> int:
    if not use_gate_in_kernel:
        return KDA_GATE_PREGATED
    if safe_gate and lower_bound is None:
        raise ValueError("safe_gate=True needs lower_bound (-5 <= lower_bound < 0)")
    if safe_gate is False and lower_bound is not None:
        raise ValueError("lower_bound given with safe_gate=False")
    return KDA_GATE_SAFE if lower_bound is not None else KDA_GATE_PLAIN


def make_params(q, k, v, g, beta, *, A_log=None, dt_bias=None, lower_bound=None, scale=None,
                initial_state=None, final_state=None, o=None, cu_seqlens=None,
                cu_seqlens_cpu=None, chunk_size: int = 64, use_gate_in_kernel: bool = True,
                safe_gate: Optional[bool] = None, use_qk_l2norm_in_kernel: bool = True,
                use_beta_sigmoid_in_kernel: bool = True, allow_neg_eigval: bool = False,
                transpose_state_layout: bool = False, h_out=None, workspace=None) -> kda_fwd_params:
    """Fill a ``kda_fwd_params`` from tensors (no checks beyond shapes and dtypes; the C
    layer checks the rest).

    The struct holds raw addresses, so the returned object also keeps a reference to every
    tensor it points at (attribute ``_keep``): the memory stays valid for as long as the
    parameter block is alive, even when the caller passed temporaries.  ``cu_seqlens`` and
    ``cu_seqlens_cpu`` must be int64 (the C ABI reads 8-byte offsets); an int32 tensor is
    rejected rather than read as int64.

    ``allow_neg_eigval``: beta = 2 sigmoid(logit) in [0, 2).  ``transpose_state_layout``
    (the notes' ``state_v_first``): initial / final states are [N, HV, V, K]."""
    import torch
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or g.dim() != 4 or beta.dim() != 3:
        raise ValueError("expected q,k [B,T,H,K], v [B,T,HV,V], g [B,T,HV,K], beta [B,T,HV]")
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if tuple(g.shape) != (B, T, HV, K) or tuple(beta.shape) != (B, T, HV) or v.shape[:2] != q.shape[:2]:
        raise ValueError("g must be [B,T,HV,K] and beta [B,T,HV]")
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("q,k,v,g,beta must be bfloat16 or float32")
    for name, t in (("k", k), ("v", v), ("g", g), ("beta", beta)):
        if t.dtype != dt:
            raise ValueError(f"{name} must have q's dtype {dt}")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("A_log", A_log),
                    ("dt_bias", dt_bias), ("initial_state", initial_state)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    for name, t in (("A_log", A_log), ("dt_bias", dt_bias), ("initial_state", initial_state)):
        if t is not None and t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32")
    if A_log is not None and tuple(A_log.shape) != (HV,):
        raise ValueError("A_log must be [HV]")
    if dt_bias is not None and dt_bias.numel() != HV * K:
        raise ValueError("dt_bias must be [HV*K] (or [HV, K])")
    for name, t in (("cu_seqlens", cu_seqlens), ("cu_seqlens_cpu", cu_seqlens_cpu)):
        if t is not None and (t.dtype != torch.int64 or t.dim() != 1 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 1-D int64 tensor (got {t.dtype})")
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    st_shape = (N, HV, V, K) if transpose_state_layout else (N, HV, K, V)
    if initial_state is not None and tuple(initial_state.shape) != st_shape:
        raise ValueError(f"initial_state must be {list(st_shape)} float32")
    p = kda_fwd_params()
    p.B, p.T, p.H, p.HV, p.K, p.V = B, T, H, HV, K, V
    p.chunk_size = int(chunk_size)
    p.in_dtype = KDA_BF16 if dt == torch.bfloat16 else KDA_F32
    p.gate_mode = _gate_mode(use_gate_in_kernel, safe_gate, lower_bound)
    p.lower_bound = 0.0 if lower_bound is None else float(lower_bound)
    p.scale = float(K ** -0.5 if scale is None else scale)
    p.qk_l2norm = int(bool(use_qk_l2norm_in_kernel))
    p.beta_sigmoid = int(bool(use_beta_sigmoid_in_kernel))
    p.N = N
    p.allow_neg_eigval = int(bool(allow_neg_eigval))
    p.state_v_first = int(bool(transpose_state_layout))
    p.q, p.k, p.v, p.g, p.beta = _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta)
    p.A_log, p.dt_bias, p.h0 = _ptr(A_log), _ptr(dt_bias), _ptr(initial_state)
    p.cu_seqlens = _ptr(cu_seqlens)
    p.cu_seqlens_host = _ptr(cu_seqlens_cpu)
    p.o, p.final_state, p.h_out = _ptr(o), _ptr(final_state), _ptr(h_out)
    if workspace is not None:
        p.workspace, p.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    p._keep = tuple(t for t in (q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens,
                                cu_seqlens_cpu, o, final_state, h_out, workspace) if t is not None)
    return p


def kda_fwd_workspace_size(p: kda_fwd_params) -> int:
    return _binding.kda_fwd_workspace_size(p)


def kda_fwd(q, k, v, g, beta, *, A_log=None, dt_bias=None, lower_bound=None, scale=None,
            initial_state=None, output_final_state: bool = True, cu_seqlens=None,
            cu_seqlens_cpu=None, chunk_size: int = 64, use_gate_in_kernel: bool = True,
            safe_gate: Optional[bool] = None, use_qk_l2norm_in_kernel: bool = True,
            use_beta_sigmoid_in_kernel: bool = True, allow_neg_eigval: bool = False,
            transpose_state_layout: bool = False, return_intermediate_states: bool = False,
            workspace=None, o=None, final_state=None, stream=None):
    """Chunk-parallel KDA forward on the current CUDA device.  Returns (o, final_state).

    o has v's dtype and shape [B,T,HV,V]; final_state is fp32 [N,HV,K,V] ([N,HV,V,K] with
    ``transpose_state_layout``; None if ``output_final_state`` is False).  With
    ``return_intermediate_states`` a third result: the state before every chunk, fp32
    [nct, HV, K, V] (transposed like final_state), chunks of sequence n after those of
    sequences 0..n-1.  With ``cu_seqlens`` (int64 [N+1], B == 1),
    rows of o outside every sequence are zero.  Asynchronous on ``stream``
    (default: the current PyTorch stream).
    """
    import torch
    if not q.is_cuda:
        raise ValueError("kda_fwd runs on CUDA tensors only")
    cu_seqlens, cu_seqlens_cpu = _int64_seqlens(cu_seqlens, cu_seqlens_cpu)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:  # rows past the last sequence are zeroed by the library itself
        o = torch.empty((B, T, HV, V), dtype=v.dtype, device=v.device)
    if final_state is None and output_final_state:
        st_shape = (N, HV, V, K) if transpose_state_layout else (N, HV, K, V)
        final_state = torch.empty(st_shape, dtype=torch.float32, device=v.device)
    p = make_params(q, k, v, g, beta, A_log=A_log, dt_bias=dt_bias, lower_bound=lower_bound,
                    scale=scale, initial_state=initial_state, final_state=final_state, o=o,
                    cu_seqlens=cu_seqlens, cu_seqlens_cpu=cu_seqlens_cpu, chunk_size=chunk_size,
                    use_gate_in_kernel=use_gate_in_kernel, safe_gate=safe_gate,
                    use_qk_l2norm_in_kernel=use_qk_l2norm_in_kernel,
                    use_beta_sigmoid_in_kernel=use_beta_sigmoid_in_kernel,
                    allow_neg_eigval=allow_neg_eigval,
                    transpose_state_layout=transpose_state_layout)
    _binding.raise_for(_binding.kda_fwd_check(p))
    h_out = None
    if return_intermediate_states:
        nct = _binding.kda_fwd_num_chunks(p)
        hs_shape = (nct, HV, V, K) if transpose_state_layout else (nct, HV, K, V)
        h_out = torch.empty(hs_shape, dtype=torch.float32, device=v.device)
        p.h_out = _ptr(h_out)
    need = _binding.kda_fwd_workspace_size(p)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=v.device)
    p.workspace, p.workspace_bytes = _ptr(workspace), workspace.numel()
    if stream is None:
        stream = torch.cuda.current_stream(v.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _binding.raise_for(_binding.kda_fwd(p, handle))
    if return_intermediate_states:
        return o, final_state, h_out
    return o, final_state


def kda_fused_recurrent_fwd(q, k, v, g, beta, *, A_log=None, dt_bias=None, lower_bound=None,
                            scale=None, initial_state=None, output_final_state: bool = True,
                            cu_seqlens=None, cu_seqlens_cpu=None, use_gate_in_kernel: bool = True,
                            safe_gate: Optional[bool] = None, use_qk_l2norm_in_kernel: bool = True,
                            use_beta_sigmoid_in_kernel: bool = True, allow_neg_eigval: bool = False,
                            transpose_state_layout: bool = False, o=None, final_state=None,
                            stream=None):
    """The same forward pass as a token recurrence (decode / short prefill).  Returns
    (o, final_state) exactly as ``kda_fwd``; no workspace, no chunking."""
    import torch
    if not q.is_cuda:
        raise ValueError("kda_fused_recurrent_fwd runs on CUDA tensors only")
    cu_seqlens, cu_seqlens_cpu = _int64_seqlens(cu_seqlens, cu_seqlens_cpu)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:  # rows past the last sequence are zeroed by the library itself
        o = torch.empty((B, T, HV, V), dtype=v.dtype, device=v.device)
    if final_state is None and output_final_state:
        st_shape = (N, HV, V, K) if transpose_state_layout else (N, HV, K, V)
        final_state = torch.empty(st_shape, dtype=torch.float32, device=v.device)
    p = make_params(q, k, v, g, beta, A_log=A_log, dt_bias=dt_bias, lower_bound=lower_bound,
                    scale=scale, initial_state=initial_state, final_state=final_state, o=o,
                    cu_seqlens=cu_seqlens, cu_seqlens_cpu=cu_seqlens_cpu,
                    use_gate_in_kernel=use_gate_in_kernel, safe_gate=safe_gate,
                    use_qk_l2norm_in_kernel=use_qk_l2norm_in_kernel,
                    use_beta_sigmoid_in_kernel=use_beta_sigmoid_in_kernel,
                    allow_neg_eigval=allow_neg_eigval,
                    transpose_state_layout=transpose_state_layout)
    if stream is None:
        stream = torch.cuda.current_stream(v.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _binding.raise_for(_binding.kda_fused_recurrent_fwd(p, handle))
    return o, final_state


def kda_fwd_host(q, k, v, g, beta, *, o, final_state=None, A_log=None, dt_bias=None,
                 lower_bound=None, scale=None, initial_state=None, cu_seqlens=None,
                 chunk_size: int = 64, use_gate_in_kernel: bool = True,
                 safe_gate: Optional[bool] = None, use_qk_l2norm_in_kernel: bool = True,
                 use_beta_sigmoid_in_kernel: bool = True, allow_neg_eigval: bool = False,
                 transpose_state_layout: bool = False, h_out=None, arena=None, stream=None):
    """The forward pass on host (CPU) tensors; pinned memory makes the copies overlap the
    kernels.  ``o`` (and ``final_state`` / ``h_out`` if given) are host tensors the result is
    written to; ``cu_seqlens`` is a host int64 tensor.  ``arena`` (device uint8 tensor of at
    least ``kda_fwd_host_arena_size`` bytes) is allocated when not given.  Asynchronous on
    ``stream``: synchronise it before reading the outputs."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("o", o)):
        if t.is_cuda:
            raise ValueError(f"{name} must be a host tensor")
    cu_cpu = None if cu_seqlens is None else cu_seqlens.to(torch.int64).contiguous()
    p = make_params(q, k, v, g, beta, A_log=A_log, dt_bias=dt_bias, lower_bound=lower_bound,
                    scale=scale, initial_state=initial_state, final_state=final_state, o=o,
                    cu_seqlens=cu_cpu, cu_seqlens_cpu=cu_cpu, chunk_size=chunk_size,
                    use_gate_in_kernel=use_gate_in_kernel, safe_gate=safe_gate,
                    use_qk_l2norm_in_kernel=use_qk_l2norm_in_kernel,
                    use_beta_sigmoid_in_kernel=use_beta_sigmoid_in_kernel,
                    allow_neg_eigval=allow_neg_eigval,
                    transpose_state_layout=transpose_state_layout, h_out=h_out)
    p.cu_seqlens = None  # the host entry reads cu_seqlens_host only
    need = _binding.kda_fwd_host_arena_size(p)
    if need == 0:
        _binding.raise_for(_binding.kda_fwd_check(p))
    if arena is None:
        dev = torch.device("cuda", torch.cuda.current_device())
        arena = torch.empty(need, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(arena.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _binding.raise_for(_binding.kda_fwd_host(p, _ptr(arena), arena.numel(), handle))
    return o, final_state


def kda_bwd(q, k, v, g, beta, do, *, dht=None, A_log=None, dt_bias=None, lower_bound=None,
            scale=None, initial_state=None, cu_seqlens=None, cu_seqlens_cpu=None,
            chunk_size: int = 64, use_gate_in_kernel: bool = True, safe_gate: Optional[bool] = None,
            use_qk_l2norm_in_kernel: bool = True, use_beta_sigmoid_in_kernel: bool = True,
            allow_neg_eigval: bool = False, transpose_state_layout: bool = False,
            return_dh0: bool = True, workspace=None, stream=None):
    """Backward pass of ``kda_fwd`` (same inputs and keyword arguments) for the incoming
    gradients ``do`` (o's shape and dtype) and ``dht`` (final_state's shape, fp32; None = 0).

    Returns (dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dh0), fp32 tensors shaped like q, k, v,
    g, beta, A_log, dt_bias and the initial state; dA_log / ddt_bias are None when A_log /
    dt_bias are absent or the gate is not in-kernel, dh0 None unless ``return_dh0``.  dg is the
    gradient with respect to g as passed (the raw gate input).  Asynchronous on ``stream``."""
    import torch
    if not q.is_cuda:
        raise ValueError("kda_bwd runs on CUDA tensors only")
    cu_seqlens, cu_seqlens_cpu = _int64_seqlens(cu_seqlens, cu_seqlens_cpu)
    if tuple(do.shape) != tuple(v.shape) or do.dtype != v.dtype or not do.is_contiguous():
        raise ValueError("do must be contiguous with o's shape and dtype")
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    st_shape = (N, HV, V, K) if transpose_state_layout else (N, HV, K, V)
    if dht is not None and (tuple(dht.shape) != st_shape or dht.dtype != torch.float32
                            or not dht.is_contiguous()):
        raise ValueError(f"dht must be contiguous float32 {list(st_shape)}")
    f = make_params(q, k, v, g, beta, A_log=A_log, dt_bias=dt_bias, lower_bound=lower_bound,
                    scale=scale, initial_state=initial_state, cu_seqlens=cu_seqlens,
                    cu_seqlens_cpu=cu_seqlens_cpu, chunk_size=chunk_size,
                    use_gate_in_kernel=use_gate_in_kernel, safe_gate=safe_gate,
                    use_qk_l2norm_in_kernel=use_qk_l2norm_in_kernel,
                    use_beta_sigmoid_in_kernel=use_beta_sigmoid_in_kernel,
                    allow_neg_eigval=allow_neg_eigval,
                    transpose_state_layout=transpose_state_layout)
    dev = v.device
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dk = torch.empty(q.shape, **f32), torch.empty(k.shape, **f32)
    dv, dg, dbeta = torch.empty(v.shape, **f32), torch.empty(g.shape, **f32), torch.empty(beta.shape, **f32)
    in_gate = f.gate_mode != KDA_GATE_PREGATED
    dA_log = torch.empty((HV,), **f32) if (A_log is not None and in_gate) else None
    ddt_bias = torch.empty(tuple(dt_bias.shape), **f32) if (dt_bias is not None and in_gate) else None
    dh0 = torch.empty(st_shape, **f32) if return_dh0 else None
    p = kda_bwd_params()
    p.fwd = f
    p.d_o, p.d_final_state = _ptr(do), _ptr(dht)
    p.dq, p.dk, p.dv, p.dg, p.dbeta = _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta)
    p.dA_log, p.ddt_bias, p.dh0 = _ptr(dA_log), _ptr(ddt_bias), _ptr(dh0)
    _binding.raise_for(_binding.kda_bwd_check(p))
    need = _binding.kda_bwd_workspace_size(p)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    p.workspace, p.workspace_bytes = _ptr(workspace), workspace.numel()
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _binding.raise_for(_binding.kda_bwd(p, handle))
    return dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dh0
