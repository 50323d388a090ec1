"""fp64 reference gradients of the KDA forward pass (test infrastructure only).

The forward's backward pass ([reading] "Reading Notes: Implementation Notes for KDA in FLA",
backward-propagation section, entry chunk_kda_bwd) returns the gradients of o (and of the final
state) with respect to q, k, v, g, beta, A_log, dt_bias and the initial state.  The pages derive
them chunk by chunk (dAv, dh, WY, intra); whatever the blocking, the result is the derivative of
the forward map, which is unique.  This module therefore writes the forward once more as the plain
token recurrence ([reading] forward pass, the recurrence the chunk form reorganises; the same
steps as ``ref.recurrent_np``) in PyTorch fp64 on the CPU and lets autograd differentiate it.

It is only as correct as that restatement and autograd; the pins in tests/test_oracle_backward.py
tie it to things outside it: central finite differences of the C oracle's forward, closed-form
derivatives of one-token cases, and linearity in the incoming gradient.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from .ref import GATE_PLAIN, GATE_PREGATED, GATE_SAFE, L2_EPS


def _t(x):
    import torch
    return None if x is None else torch.tensor(np.asarray(x, np.float64), dtype=torch.float64)


def gate_t(g, mode, A_log=None, dt_bias=None, lower_bound=None):
    """The activated log-decay gate ([notes] section 2) for a torch fp64 g of shape [..., HV, K]."""
    import torch
    if mode == GATE_PREGATED:
        return g
    HV, K = g.shape[-2], g.shape[-1]
    x = g if dt_bias is None else g + dt_bias.reshape(HV, K)
    if mode == GATE_PLAIN:
        return -torch.exp(A_log).reshape(HV, 1) * torch.nn.functional.softplus(x)
    if mode == GATE_SAFE:
        a = 1.0 if A_log is None else torch.exp(A_log).reshape(HV, 1)
        return float(lower_bound) * torch.sigmoid(a * x)
    raise ValueError(f"unknown gate mode {mode}")


def recurrent_t(q, k, v, g, beta, *, A_log=None, dt_bias=None, gate_mode=GATE_SAFE,
                lower_bound=None, scale=None, qk_l2norm=True, beta_sigmoid=True,
                allow_neg_eigval=False, initial_state=None, l2_eps=L2_EPS):
    """The token recurrence on torch fp64 tensors (B sequences of T tokens, grouped value heads
    hv -> h = hv // (HV / H)); returns (o [B,T,HV,V], final_state [B,HV,K,V])."""
    import torch
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    G = HV // H
    if scale is None:
        scale = K ** -0.5
    if qk_l2norm:
        q = q / torch.sqrt((q * q).sum(-1, keepdim=True) + l2_eps)
        k = k / torch.sqrt((k * k).sum(-1, keepdim=True) + l2_eps)
    gp = gate_t(g, gate_mode, A_log, dt_bias, lower_bound)
    b = beta
    if beta_sigmoid:
        b = (2.0 if allow_neg_eigval else 1.0) * torch.sigmoid(beta)
    hmap = torch.arange(HV) // G
    outs, finals = [], []
    for n in range(B):
        S = torch.zeros(HV, K, V, dtype=torch.float64) if initial_state is None else initial_state[n]
        o_n = []
        for t in range(T):
            kt, qt = k[n, t, hmap], q[n, t, hmap]                  # [HV, K]
            S = S * torch.exp(gp[n, t])[:, :, None]                # Diag(alpha_t) S
            p = torch.einsum("hk,hkv->hv", kt, S)                  # S^T k
            u = b[n, t][:, None] * (v[n, t] - p)
            S = S + kt[:, :, None] * u[:, None, :]
            o_n.append(scale * torch.einsum("hk,hkv->hv", qt, S))
        outs.append(torch.stack(o_n) if o_n else torch.zeros(0, HV, V, dtype=torch.float64))
        finals.append(S)
    return torch.stack(outs), torch.stack(finals)


def bwd(q, k, v, g, beta, do, dfinal=None, *, A_log=None, dt_bias=None, gate_mode=GATE_SAFE,
        lower_bound=None, scale=None, qk_l2norm=True, beta_sigmoid=True, allow_neg_eigval=False,
        initial_state=None, l2_eps=L2_EPS) -> dict:
    """Gradients of <do, o> + <dfinal, final_state> with respect to every input, in fp64.

    Inputs as for ``ref.recurrent_np`` without varlen (B sequences of T tokens); do has o's
    shape [B,T,HV,V], dfinal the final state's [B,HV,K,V] (None: zero).  Returns a dict with
    o, final_state and dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dh0 (None for absent inputs),
    as float64 NumPy arrays."""
    import torch
    leaves = {"q": _t(q), "k": _t(k), "v": _t(v), "g": _t(g), "beta": _t(beta),
              "A_log": _t(A_log), "dt_bias": _t(dt_bias), "h0": _t(initial_state)}
    for x in leaves.values():
        if x is not None:
            x.requires_grad_(True)
    o, fs = recurrent_t(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                        A_log=leaves["A_log"], dt_bias=leaves["dt_bias"], gate_mode=gate_mode,
                        lower_bound=lower_bound, scale=scale, qk_l2norm=qk_l2norm,
                        beta_sigmoid=beta_sigmoid, allow_neg_eigval=allow_neg_eigval,
                        initial_state=leaves["h0"], l2_eps=l2_eps)
    loss = (o * _t(do)).sum()
    if dfinal is not None:
        loss = loss + (fs * _t(dfinal)).sum()
    present = [(name, x) for name, x in leaves.items() if x is not None]
    grads = torch.autograd.grad(loss, [x for _, x in present], allow_unused=True)
    out = {"o": o.detach().numpy(), "final_state": fs.detach().numpy()}
    for name in leaves:
        out["d" + name] = None
    for (name, x), gr in zip(present, grads):
        out["d" + name] = (torch.zeros_like(x) if gr is None else gr).detach().numpy()
    return out
