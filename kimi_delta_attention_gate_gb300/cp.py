"""Context parallelism for the KDA forward pass: a batch of sequences sharded along time
over the ranks of a process group (each rank holds one contiguous range of tokens of every
sequence; shard lengths may differ between ranks).

The state recurrence ("Reading Notes: Implementation Notes for KDA in FLA", forward step 4)
is affine in the state, so a shard acts on the state entering it as S_out = P S_in + R per
(sequence, value head), with P (K x K) and R (K x V) depending only on the shard's tokens.
``cp_fwd`` on every rank:

1. forms its shard's maps with two forward passes over its own tokens (``state_map``):
   R is the final state from a zero initial state; P is the final state of the pass with
   v = 0 from the identity (with v = 0 the recurrence is linear in the state, so the state
   it reaches from I is the transition itself);
2. exchanges the maps over the group (one all-gather: K·K + K·V fp32 per sequence, value
   head and rank; NCCL for CUDA tensors, gloo for CPU ones);
3. chains the maps of the ranks before it from the batch's initial state, an exclusive
   prefix S_in(0) = h0, S_in(j+1) = P_j S_in(j) + R_j (``chain``; on the GPU each step is one
   ``kda_state_affine_apply`` launch);
4. runs the forward pass on its shard from S_in(rank).

The flag table of "FLA-KDA engineering notes" section 2.2 names this option (cp_context);
the pages give no mechanism, and this is the plain reading of the affine step.  Only the
exchange moves data between ranks.  ``fwd`` and ``apply`` default to this library's CUDA
entry points; they are parameters so that the exchange logic can be exercised on CPU ranks
with another implementation of the same two operations.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence

from . import _binding


def affine_apply(P, R, S_in, *, state_v_first: bool = False, stream=None):
    """S_out = P S_in + R per map on the GPU (``kda_state_affine_apply``).  P [..., K, K];
    R and S_in [..., K, V] ([..., V, K] with ``state_v_first``); S_in may be None (zero)."""
    import torch
    for name, t in (("P", P), ("R", R), ("S_in", S_in)):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    K = P.shape[-1]
    V = R.shape[-2] if state_v_first else R.shape[-1]
    nmaps = P.numel() // (K * K)
    if R.numel() != nmaps * K * V or (S_in is not None and S_in.shape != R.shape):
        raise ValueError("P, R and S_in describe different numbers of maps")
    out = torch.empty_like(R)
    if stream is None:
        stream = torch.cuda.current_stream(R.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _binding.raise_for(_binding.kda_state_affine_apply(
        P.data_ptr(), R.data_ptr(), None if S_in is None else S_in.data_ptr(), out.data_ptr(),
        nmaps, K, V, int(bool(state_v_first)), handle))
    return out


def state_map(q, k, v, g, beta, *, fwd: Optional[Callable] = None,
              transpose_state_layout: bool = False, **kw):
    """The affine map (P, R) of this shard per (sequence, value head).

    P: float32 [N, HV, K, K] (always acting on the left of a K x V state); R: float32
    [N, HV, K, V] ([N, HV, V, K] with ``transpose_state_layout``).  ``kw`` are the forward
    pass's keyword arguments (gate, scale, cu_seqlens, ...) except ``initial_state``."""
    import torch
    if fwd is None:
        from . import kda_fwd as fwd
    if "initial_state" in kw:
        raise ValueError("state_map takes no initial_state: the map does not depend on it")
    B, T, H, K = q.shape
    HV = v.shape[2]
    N = B if kw.get("cu_seqlens") is None else kw["cu_seqlens"].numel() - 1
    _, R = fwd(q, k, v, g, beta, initial_state=None, transpose_state_layout=transpose_state_layout,
               **kw)
    v0 = torch.zeros((B, T, HV, K), dtype=v.dtype, device=v.device)
    eye = torch.eye(K, dtype=torch.float32, device=v.device).expand(N, HV, K, K).contiguous()
    _, Pst = fwd(q, k, v0, g, beta, initial_state=eye,
                 transpose_state_layout=transpose_state_layout, **kw)
    # the pass stores its state transposed with transpose_state_layout; P keeps [K, K]
    P = Pst.transpose(-1, -2).contiguous() if transpose_state_layout else Pst
    return P, R


def chain(P_list: Sequence, R_list: Sequence, h0, *, apply: Optional[Callable] = None,
          state_v_first: bool = False) -> List:
    """Exclusive prefix of the maps: [S_in(0), S_in(1), ..., S_in(n)] with S_in(0) = h0
    (None = zero state) and S_in(j+1) = P_j S_in(j) + R_j.  S_in(j) is the state entering
    shard j; S_in(n) is the final state of the whole sequence."""
    if apply is None:
        def apply(P, R, S):
            return affine_apply(P, R, S, state_v_first=state_v_first)
    states = [h0]
    for P, R in zip(P_list, R_list):
        states.append(apply(P, R, states[-1]))
    return states


def cp_fwd(q, k, v, g, beta, *, group=None, initial_state=None, fwd: Optional[Callable] = None,
           apply: Optional[Callable] = None, transpose_state_layout: bool = False, **kw):
    """The forward pass of this rank's shard of a time-sharded batch.  Returns (o, S_out):
    o for this shard's tokens and the state after the shard (on the last rank, the final state
    of the whole sequences).  ``initial_state`` is the batch's initial state (the same tensor,
    or None, on every rank).  Collective: every rank of ``group`` must call it."""
    import torch
    import torch.distributed as dist
    if fwd is None:
        from . import kda_fwd as fwd
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    P, R = state_map(q, k, v, g, beta, fwd=fwd, transpose_state_layout=transpose_state_layout,
                     **kw)
    Ps = [torch.empty_like(P) for _ in range(world)]
    Rs = [torch.empty_like(R) for _ in range(world)]
    dist.all_gather(Ps, P, group=group)
    dist.all_gather(Rs, R, group=group)
    S_in = chain(Ps[:rank], Rs[:rank], initial_state, apply=apply,
                 state_v_first=transpose_state_layout)[-1]
    o, S_out = fwd(q, k, v, g, beta, initial_state=S_in,
                   transpose_state_layout=transpose_state_layout, **kw)
    return o, S_out
