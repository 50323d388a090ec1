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

``chunk_bwd_np`` is the second form: the gradients derived by hand through the chunk form, stage
by stage as a chunked backward computes them (the intermediates a GPU backward can be checked
against one by one); it is pinned to ``bwd``.
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


def _split_varlen(cu_seqlens, arrays):
    """[1, total, ...] arrays -> per-sequence [1, len, ...] views (cu_seqlens, [notes] section
    2.2 varlen example)."""
    cu = np.asarray(cu_seqlens, np.int64)
    return [[None if a is None else a[:, cu[n]:cu[n + 1]] for a in arrays] for n in range(len(cu) - 1)]


def _varlen(fn, q, k, v, g, beta, do, dfinal, cu_seqlens, initial_state, transpose, kw) -> dict:
    """Run ``fn`` per sequence of a varlen batch and assemble the results: token gradients in
    the flattened layout (rows no sequence covers get 0), per-sequence states stacked, the
    shared A_log / dt_bias gradients summed."""
    tok = np.asarray(q).shape[1]
    outs = []
    for n, (qn, kn, vn, gn, bn, don) in enumerate(
            _split_varlen(cu_seqlens, [np.asarray(q), np.asarray(k), np.asarray(v), np.asarray(g),
                                       np.asarray(beta), np.asarray(do)])):
        h0n = None if initial_state is None else np.asarray(initial_state)[n:n + 1]
        dfn = None if dfinal is None else np.asarray(dfinal)[n:n + 1]
        outs.append(fn(qn, kn, vn, gn, bn, don, dfn, initial_state=h0n,
                       transpose_state_layout=transpose, **kw))
    cu = np.asarray(cu_seqlens, np.int64)
    res = {}
    for key, tokwise in (("o", True), ("dq", True), ("dk", True), ("dv", True), ("dg", True),
                         ("dbeta", True), ("final_state", False), ("dh0", False),
                         ("dA_log", None), ("ddt_bias", None)):
        parts = [r[key] for r in outs]
        if parts[0] is None:
            res[key] = None
        elif tokwise:
            full = np.zeros((1, tok) + parts[0].shape[2:])
            for n, part in enumerate(parts):
                full[:, cu[n]:cu[n + 1]] = part
            res[key] = full
        elif tokwise is False:
            res[key] = np.concatenate(parts, axis=0)
        else:
            res[key] = np.sum(parts, axis=0)
    return res


def bwd(q, k, v, g, beta, do, dfinal=None, *, A_log=None, dt_bias=None, gate_mode=GATE_SAFE,
        lower_bound=None, scale=None, qk_l2norm=True, beta_sigmoid=True, allow_neg_eigval=False,
        initial_state=None, cu_seqlens=None, transpose_state_layout=False, l2_eps=L2_EPS) -> dict:
    """Gradients of <do, o> + <dfinal, final_state> with respect to every input, in fp64.

    Inputs as for ``ref.recurrent_np``: B sequences of T tokens, or with ``cu_seqlens`` a
    varlen batch flattened to B = 1; do has o's shape [B,T,HV,V], dfinal the final state's
    [N,HV,K,V] (None: zero).  ``transpose_state_layout``: initial / final states (and their
    gradients) are [N,HV,V,K].  Returns a dict with o, final_state and dq, dk, dv, dg, dbeta,
    dA_log, ddt_bias, dh0 (None for absent inputs), as float64 NumPy arrays."""
    if cu_seqlens is not None:
        kw = dict(A_log=A_log, dt_bias=dt_bias, gate_mode=gate_mode, lower_bound=lower_bound,
                  scale=scale, qk_l2norm=qk_l2norm, beta_sigmoid=beta_sigmoid,
                  allow_neg_eigval=allow_neg_eigval, l2_eps=l2_eps)
        return _varlen(bwd, q, k, v, g, beta, do, dfinal, cu_seqlens, initial_state,
                       transpose_state_layout, kw)
    if transpose_state_layout:
        sw = lambda x: None if x is None else np.swapaxes(np.asarray(x), -1, -2)
        r = bwd(q, k, v, g, beta, do, sw(dfinal), A_log=A_log, dt_bias=dt_bias,
                gate_mode=gate_mode, lower_bound=lower_bound, scale=scale, qk_l2norm=qk_l2norm,
                beta_sigmoid=beta_sigmoid, allow_neg_eigval=allow_neg_eigval,
                initial_state=sw(initial_state), l2_eps=l2_eps)
        r["final_state"], r["dh0"] = sw(r["final_state"]), sw(r["dh0"])
        return r
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


# ----------------------------------------------------------------------------------------------
# The chunked backward, written out by hand
# ----------------------------------------------------------------------------------------------

def _l2norm_bwd(x, dxh, eps):
    """x_hat = x / sqrt(|x|^2 + eps) over the last axis: the gradient with respect to x."""
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
    return dxh / n - x * np.sum(x * dxh, axis=-1, keepdims=True) / n ** 3


def chunk_bwd_np(q, k, v, g, beta, do, dfinal=None, *, chunk_size=64, A_log=None, dt_bias=None,
                 gate_mode=GATE_SAFE, lower_bound=None, scale=None, qk_l2norm=True,
                 beta_sigmoid=True, allow_neg_eigval=False, initial_state=None, cu_seqlens=None,
                 transpose_state_layout=False, l2_eps=L2_EPS) -> dict:
    """The same gradients as ``bwd``, derived by hand through the chunk form ([reading] forward
    pass steps 1-5; its backward-propagation section runs the same derivative as recompute
    U, W, Qg and the states; dU and dAqk from O; the reverse cross-chunk recurrence of dS; the WY
    gradients; the intra-chunk terms; a reverse cumsum for the gate), NumPy fp64, dense.

    Per chunk, with S the state before it and dS' the gradient of the state after it:
      dV_new = Aqk^T dO + Kg dS'        dAqk = (dO V_new^T) . M       dQg = dO S^T
      dS = Qg^T dO - W^T dV_new + Diag(e^gamma_C) dS'
      dKg = V_new dS'^T                 d gamma_C += e^gamma_C . rowsum(S . dS')
      dU = dV_new, dW = -dV_new S^T, dA = dU (beta V)^T + dW (beta K~)^T
      d(beta V) = A^T dU, d(beta K~) = A^T dW, dAkk0 = -(A^T dA A^T) . M_-1
    then through Aqk_ij = sum_k Q_ik K_jk e^(Gamma_ik - Gamma_jk) (and the same for Akk0's
    K K term), K~ = e^Gamma . K, Qg = e^Gamma . Q, Kg = e^(gamma_C - Gamma) . K, and
    Gamma = cumsum(g') (a reverse cumsum).  Arguments and result as for ``bwd``."""
    if cu_seqlens is not None:
        kw = dict(chunk_size=chunk_size, A_log=A_log, dt_bias=dt_bias, gate_mode=gate_mode,
                  lower_bound=lower_bound, scale=scale, qk_l2norm=qk_l2norm,
                  beta_sigmoid=beta_sigmoid, allow_neg_eigval=allow_neg_eigval, l2_eps=l2_eps)
        return _varlen(chunk_bwd_np, q, k, v, g, beta, do, dfinal, cu_seqlens, initial_state,
                       transpose_state_layout, kw)
    if transpose_state_layout:
        sw = lambda x: None if x is None else np.swapaxes(np.asarray(x), -1, -2)
        r = chunk_bwd_np(q, k, v, g, beta, do, sw(dfinal), chunk_size=chunk_size, A_log=A_log,
                         dt_bias=dt_bias, gate_mode=gate_mode, lower_bound=lower_bound,
                         scale=scale, qk_l2norm=qk_l2norm, beta_sigmoid=beta_sigmoid,
                         allow_neg_eigval=allow_neg_eigval, initial_state=sw(initial_state),
                         l2_eps=l2_eps)
        r["final_state"], r["dh0"] = sw(r["final_state"]), sw(r["dh0"])
        return r
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64); beta = np.asarray(beta, np.float64)
    do = np.asarray(do, np.float64)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    G = HV // H
    if scale is None:
        scale = K ** -0.5
    from .ref import gate_np, sigmoid_np, softplus_np
    qh = q / np.sqrt(np.sum(q * q, -1, keepdims=True) + l2_eps) if qk_l2norm else q
    kh = k / np.sqrt(np.sum(k * k, -1, keepdims=True) + l2_eps) if qk_l2norm else k
    gp = gate_np(g, gate_mode, A_log, dt_bias, lower_bound)
    cb = 2.0 if (beta_sigmoid and allow_neg_eigval) else 1.0
    bb = cb * sigmoid_np(beta) if beta_sigmoid else beta
    dqh = np.zeros_like(qh); dkh = np.zeros_like(kh); dv = np.zeros_like(v)
    dgp = np.zeros_like(gp); dbb = np.zeros_like(bb)
    o = np.zeros((B, T, HV, V)); fs = np.zeros((B, HV, K, V)); dh0 = np.zeros((B, HV, K, V))
    C = int(chunk_size)
    for n in range(B):
        for hv in range(HV):
            h = hv // G
            S = np.zeros((K, V)) if initial_state is None else np.array(initial_state[n, hv], np.float64)
            chunks, states = [], []
            for cs in range(0, T, C):  # forward: the state before every chunk
                ce = min(cs + C, T)
                L = ce - cs
                Q = scale * qh[n, cs:ce, h]
                Kc = kh[n, cs:ce, h]
                Vc = v[n, cs:ce, hv]
                bc = bb[n, cs:ce, hv]
                Gam = np.cumsum(gp[n, cs:ce, hv], axis=0)
                gC = Gam[L - 1]
                lower = np.tril(np.ones((L, L), bool))
                strict = np.tril(np.ones((L, L), bool), -1)
                D = Gam[:, None, :] - Gam[None, :, :]
                E = np.where(lower[:, :, None], np.exp(np.where(lower[:, :, None], D, 0.0)), 0.0)
                Aqk = np.einsum("ik,jk,ijk->ij", Q, Kc, E)
                P = np.where(strict, np.einsum("ik,jk,ijk->ij", Kc, Kc, E), 0.0)
                A = np.linalg.inv(np.eye(L) + bc[:, None] * P)
                Kt = np.exp(Gam) * Kc
                BV, BK = bc[:, None] * Vc, bc[:, None] * Kt
                U, W = A @ BV, A @ BK
                Qg = np.exp(Gam) * Q
                Kg = np.exp(gC[None, :] - Gam) * Kc
                Vnew = U - W @ S
                o[n, cs:ce, hv] = Qg @ S + Aqk @ Vnew
                states.append(S)
                chunks.append((cs, ce, Q, Kc, Vc, bc, Gam, gC, lower, strict, E, Aqk, P, A, Kt,
                               BV, BK, Qg, Kg, Vnew))
                S = np.exp(gC)[:, None] * S + Kg.T @ Vnew
            fs[n, hv] = S
            dS = np.zeros((K, V)) if dfinal is None else np.array(dfinal[n, hv], np.float64)
            for (cs, ce, Q, Kc, Vc, bc, Gam, gC, lower, strict, E, Aqk, P, A, Kt, BV, BK, Qg, Kg,
                 Vnew), S in zip(reversed(chunks), reversed(states)):
                dO = do[n, cs:ce, hv]
                dVnew = Aqk.T @ dO + Kg @ dS
                dAqk = np.where(lower, dO @ Vnew.T, 0.0)
                dQg = dO @ S.T
                dKg = Vnew @ dS.T
                dgC = np.exp(gC) * np.sum(S * dS, axis=1)
                dS_prev = Qg.T @ dO - (A @ BK).T @ dVnew + np.exp(gC)[:, None] * dS
                dW = -dVnew @ S.T
                dA = dVnew @ BV.T + dW @ BK.T
                dBV, dBK = A.T @ dVnew, A.T @ dW
                dv[n, cs:ce, hv] += bc[:, None] * dBV
                db = np.sum(dBV * Vc, axis=1) + np.sum(dBK * Kt, axis=1)
                dKt = bc[:, None] * dBK
                dAkk0 = np.where(strict, -(A.T @ dA @ A.T), 0.0)
                db += np.sum(dAkk0 * P, axis=1)
                dP = bc[:, None] * dAkk0
                dbb[n, cs:ce, hv] += db
                # the e^(Gamma_i - Gamma_j) kernels: rows i, columns j
                tq = np.einsum("ij,ik,jk,ijk->ijk", dAqk, Q, Kc, E)
                tk = np.einsum("ij,ik,jk,ijk->ijk", dP, Kc, Kc, E)
                dQ = dQg * np.exp(Gam) + np.einsum("ij,jk,ijk->ik", dAqk, Kc, E)
                dK = (np.einsum("ij,ik,ijk->jk", dAqk, Q, E) + np.einsum("ij,jk,ijk->ik", dP, Kc, E)
                      + np.einsum("ij,ik,ijk->jk", dP, Kc, E)
                      + dKt * np.exp(Gam) + dKg * np.exp(gC[None, :] - Gam))
                dGam = (dQg * Qg + dKt * Kt - dKg * Kg
                        + tq.sum(1) - tq.sum(0) + tk.sum(1) - tk.sum(0))
                dgC = dgC + np.sum(dKg * Kg, axis=0)
                dGam[-1] += dgC
                dgp[n, cs:ce, hv] += np.cumsum(dGam[::-1], axis=0)[::-1]  # Gamma = cumsum(g')
                dqh[n, cs:ce, h] += scale * dQ
                dkh[n, cs:ce, h] += dK
                dS = dS_prev
            dh0[n, hv] = dS
    out = {"o": o, "final_state": fs}
    out["dq"] = _l2norm_bwd(q, dqh, l2_eps) if qk_l2norm else dqh
    out["dk"] = _l2norm_bwd(k, dkh, l2_eps) if qk_l2norm else dkh
    out["dv"] = dv
    if beta_sigmoid:
        sg = sigmoid_np(beta)
        out["dbeta"] = dbb * cb * sg * (1.0 - sg)
    else:
        out["dbeta"] = dbb
    # the gate activation ([notes] section 2)
    out["dA_log"] = out["ddt_bias"] = None
    if gate_mode == GATE_PREGATED:
        out["dg"] = dgp
    else:
        x = g + (0.0 if dt_bias is None else np.asarray(dt_bias, np.float64).reshape(HV, K))
        if gate_mode == GATE_PLAIN:
            a = np.exp(np.asarray(A_log, np.float64)).reshape(HV, 1)
            dx = dgp * (-a) * sigmoid_np(x)
            out["dA_log"] = np.sum(dgp * (-a) * softplus_np(x), axis=(0, 1, 3))
        else:
            a = 1.0 if A_log is None else np.exp(np.asarray(A_log, np.float64)).reshape(HV, 1)
            sg = sigmoid_np(a * x)
            ds = dgp * float(lower_bound) * sg * (1.0 - sg)
            dx = ds * a
            if A_log is not None:
                out["dA_log"] = np.sum(ds * a * x, axis=(0, 1, 3))
        out["dg"] = dx
        if dt_bias is not None:
            out["ddt_bias"] = np.sum(dx, axis=(0, 1)).reshape(np.shape(dt_bias))
    out["dh0"] = dh0 if initial_state is not None else None
    return out
