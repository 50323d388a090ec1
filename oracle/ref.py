"""fp64 reference implementations of the KDA forward pass (test infrastructure only).

Citations name the page and the section / equation:
  [notes]   "FLA-KDA engineering notes" -- flash-linear-attention KDA kernel
            engineering practice: gate modes, safe_gate numerics, chunk
            intra/inter paths (dpshk.com article).
  [reading] "Reading Notes: Implementation Notes for KDA in FLA"
            (mzeromiko.github.io), forward pass, steps 1-5.
  [flashkda] "FlashKDA gate-bias load path" (czchanglian.com article).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

GATE_PREGATED = 0
GATE_PLAIN = 1
GATE_SAFE = 2

# Epsilon inside the square root of the in-kernel L2 norm.  The pages name
# the norm (use_qk_l2norm_in_kernel, [notes] section 2.2) but not its epsilon.
L2_EPS = 1e-6

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP, IEEE fp64, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp,
                        "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            d = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.POINTER(ctypes.c_int64)
            ci, cd = ctypes.c_int, ctypes.c_double
            lib.kdao_fwd.restype = ci
            lib.kdao_fwd.argtypes = [ci, ci, ci, ci, ci, ci, d, d, d, d, d, d, d, ci, cd, cd,
                                     ci, ci, cd, d, i64, ci, d, d, ci, ci, d]
            lib.kdao_gate.restype = None
            lib.kdao_gate.argtypes = [ci, ctypes.c_int64, ci, ci, d, d, d, cd, d]
            lib.kdao_max_threads.restype = ci
            lib.kdao_max_threads.argtypes = []
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().kdao_max_threads())


def _dptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


# ----------------------------------------------------------------------------
# Elementwise pieces
# ----------------------------------------------------------------------------

def sigmoid_np(x):
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    e = np.exp(x[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def softplus_np(x):
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def gate_np(g, mode, A_log=None, dt_bias=None, lower_bound=None):
    """Activated log-decay gate g' for g of shape [..., HV, K].

    [notes] section 2 ("gate input contracts"):
      PLAIN (in-kernel, no safe gate):  g' = -exp(A_log) * softplus(g + dt_bias)
      SAFE  (in-kernel, safe gate):     g' = lower_bound * sigmoid(exp(A_log) * (g + dt_bias)),
                                        with A_log absent -> lower_bound * sigmoid(g + dt_bias)
      PREGATED (use_gate_in_kernel=False): g is already the log decay.
    dt_bias is optional ([HV*K], equivalently [HV, K]); A_log is [HV].
    """
    g = np.asarray(g, dtype=np.float64)
    if mode == GATE_PREGATED:
        return g.copy()
    HV, K = g.shape[-2], g.shape[-1]
    x = g + (0.0 if dt_bias is None else np.asarray(dt_bias, np.float64).reshape(HV, K))
    if mode == GATE_PLAIN:
        a = np.exp(np.asarray(A_log, np.float64)).reshape(HV, 1)
        return -a * softplus_np(x)
    if mode == GATE_SAFE:
        a = 1.0 if A_log is None else np.exp(np.asarray(A_log, np.float64)).reshape(HV, 1)
        return float(lower_bound) * sigmoid_np(a * x)
    raise ValueError(f"unknown gate mode {mode}")


def l2norm_np(x, eps=L2_EPS):
    """x / sqrt(sum(x^2) + eps) over the last axis ([notes] section 2.2, use_qk_l2norm_in_kernel)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def _prepare(q, k, g, beta, A_log, dt_bias, gate_mode, lower_bound, qk_l2norm, beta_sigmoid,
             l2_eps):
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    if qk_l2norm:
        q, k = l2norm_np(q, l2_eps), l2norm_np(k, l2_eps)
    gp = gate_np(g, gate_mode, A_log, dt_bias, lower_bound)
    b = np.asarray(beta, np.float64)
    if beta_sigmoid:
        b = sigmoid_np(b)
    return q, k, gp, b


def _segments(B, T, cu_seqlens):
    """(bos, eos) of every sequence in the flattened [B*T] token axis."""
    if cu_seqlens is None:
        return [(n * T, (n + 1) * T) for n in range(B)]
    cu = np.asarray(cu_seqlens, np.int64)
    return [(int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]


# ----------------------------------------------------------------------------
# The oracle proper (C, fp64)
# ----------------------------------------------------------------------------

def fwd(q, k, v, g, beta, *, A_log=None, dt_bias=None, gate_mode=GATE_SAFE, lower_bound=None,
        scale=None, qk_l2norm=True, beta_sigmoid=True, initial_state=None, cu_seqlens=None,
        allow_neg_eigval=False, transpose_state_layout=False, return_intermediate_states=False,
        chunk_size=64, l2_eps=L2_EPS, nthreads=0):
    """Token-recurrent KDA forward in fp64 (C).  Returns (o [B,T,HV,V], final_state [N,HV,K,V]).

    The recurrence S_t = Diag(a_t) S - b_t k_t (k_t^T Diag(a_t) S) + b_t k_t v_t^T,
    o_t = scale S_t^T q_t, with a_t = exp(g'_t).  With ``cu_seqlens`` the batch
    is flattened to B = 1 and sequence n spans tokens [cu[n], cu[n+1]) ([notes]
    section 2.2, varlen example); rows no sequence covers come back as 0.
    ``allow_neg_eigval`` ([notes] section 2.1): beta = 2 sigmoid(logit), which needs
    ``beta_sigmoid``.  ``transpose_state_layout`` ([notes] section 2.2, state_v_first):
    initial and final states are [N,HV,V,K], the transpose of the K x V state.
    ``return_intermediate_states`` ([notes] section 2.2): a third result, the state before
    every chunk of ``chunk_size`` tokens, [nct,HV,K,V] (chunks of sequence n after those of
    sequences 0..n-1; transposed like the other states).
    """
    lib = _load()
    q = _f64(q); k = _f64(k); v = _f64(v); g = _f64(g); beta = _f64(beta)
    if allow_neg_eigval:
        if not beta_sigmoid:
            raise ValueError("allow_neg_eigval needs beta_sigmoid")
        beta = 2.0 * sigmoid_np(beta)          # the C routine then takes beta as given
        beta_sigmoid = False
    if transpose_state_layout and initial_state is not None:
        initial_state = np.swapaxes(np.asarray(initial_state), -1, -2)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    N = B if cu is None else len(cu) - 1
    if scale is None:
        scale = K ** -0.5
    lb = 0.0 if lower_bound is None else float(lower_bound)
    A_log = _f64(A_log); dt_bias = _f64(dt_bias); h0 = _f64(initial_state)
    o = np.zeros((B, T, HV, V), dtype=np.float64)
    fs = np.zeros((N, HV, K, V), dtype=np.float64)
    hs = None
    if return_intermediate_states:
        lens = ([T] * B) if cu is None else np.diff(cu).tolist()
        nct = int(sum((ln + chunk_size - 1) // chunk_size for ln in lens))
        hs = np.zeros((nct, HV, K, V), dtype=np.float64)
    rc = lib.kdao_fwd(B, T, H, HV, K, V, _dptr(q), _dptr(k), _dptr(v), _dptr(g), _dptr(beta),
                      _dptr(A_log), _dptr(dt_bias), int(gate_mode), lb, float(scale),
                      int(bool(qk_l2norm)), int(bool(beta_sigmoid)), float(l2_eps), _dptr(h0),
                      None if cu is None else cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                      N, _dptr(o), _dptr(fs), int(nthreads), int(chunk_size), _dptr(hs))
    if rc != 0:
        raise ValueError("oracle: inconsistent arguments")
    if transpose_state_layout:
        fs = np.ascontiguousarray(np.swapaxes(fs, -1, -2))
        if hs is not None:
            hs = np.ascontiguousarray(np.swapaxes(hs, -1, -2))
    if return_intermediate_states:
        return o, fs, hs
    return o, fs


def gate_c(g, mode, A_log=None, dt_bias=None, lower_bound=None):
    """The C oracle's gate activation, for [ntok, HV, K] input."""
    lib = _load()
    g = _f64(g)
    ntok, HV, K = int(np.prod(g.shape[:-2])), g.shape[-2], g.shape[-1]
    out = np.empty_like(g)
    lib.kdao_gate(int(mode), ntok, HV, K, _dptr(g), _dptr(_f64(A_log)), _dptr(_f64(dt_bias)),
                  0.0 if lower_bound is None else float(lower_bound), _dptr(out))
    return out


# ----------------------------------------------------------------------------
# NumPy cross-checks
# ----------------------------------------------------------------------------

def recurrent_np(q, k, v, g, beta, *, A_log=None, dt_bias=None, gate_mode=GATE_SAFE,
                 lower_bound=None, scale=None, qk_l2norm=True, beta_sigmoid=True,
                 initial_state=None, cu_seqlens=None, l2_eps=L2_EPS):
    """The same token recurrence as ``fwd``, in NumPy fp64 (loops over tokens)."""
    B, T, H, K = np.shape(q)
    HV, V = np.shape(v)[2], np.shape(v)[3]
    G = HV // H
    if scale is None:
        scale = K ** -0.5
    qn, kn, gp, b = _prepare(q, k, g, beta, A_log, dt_bias, gate_mode, lower_bound, qk_l2norm,
                             beta_sigmoid, l2_eps)
    qn = qn.reshape(B * T, H, K)
    kn = kn.reshape(B * T, H, K)
    vv = np.asarray(v, np.float64).reshape(B * T, HV, V)
    gp = gp.reshape(B * T, HV, K)
    b = b.reshape(B * T, HV)
    segs = _segments(B, T, cu_seqlens)
    o = np.zeros((B * T, HV, V))
    fs = np.zeros((len(segs), HV, K, V))
    hmap = np.arange(HV) // G
    for n, (bos, eos) in enumerate(segs):
        S = np.zeros((HV, K, V)) if initial_state is None else \
            np.array(initial_state, np.float64)[n].copy()
        for t in range(bos, eos):
            kt = kn[t, hmap]                       # [HV, K]
            qt = qn[t, hmap]
            S = S * np.exp(gp[t])[:, :, None]      # Diag(alpha_t) S
            p = np.einsum("hk,hkv->hv", kt, S)     # S^T k
            u = b[t][:, None] * (vv[t] - p)
            S = S + kt[:, :, None] * u[:, None, :]
            o[t] = scale * np.einsum("hk,hkv->hv", qt, S)
        fs[n] = S
    return o.reshape(B, T, HV, V), fs


def chunk_np(q, k, v, g, beta, *, chunk_size=64, A_log=None, dt_bias=None, gate_mode=GATE_SAFE,
             lower_bound=None, scale=None, qk_l2norm=True, beta_sigmoid=True, initial_state=None,
             cu_seqlens=None, l2_eps=L2_EPS):
    """The chunk-parallel form, [reading] forward pass steps 1-5, fp64, dense.

    Per chunk [t] of C tokens (the last chunk of a sequence may be shorter):
      step 1  Gamma^r = sum_{i<=r in chunk} log alpha_i          (chunk-local cumsum)
      step 2  Aqk = (Q . e^Gamma)(K / e^Gamma)^T . M
              Akk0 = Diag(beta) ((K . e^Gamma)(K / e^Gamma)^T . M_-1),  A = (I + Akk0)^-1
      step 3  U = A (Diag(beta) V),  W = A (e^Gamma . Diag(beta) K)
              Qg = e^Gamma . Q,  Kg = e^(1 gamma_C^T - Gamma) . K
      step 4  V_new = U - W S,  S <- Diag(e^gamma_C) S + Kg^T V_new
      step 5  O = Qg S_prev + Aqk V_new
    M is lower triangular with the diagonal, M_-1 strictly lower.  ``scale``
    multiplies Q.  The products (Q . e^Gamma)(K / e^Gamma)^T are evaluated as
    sum_k q_ik k_jk e^(Gamma_ik - Gamma_jk) on the unmasked entries -- the same
    numbers, without forming e^-Gamma (which overflows for long gates).
    """
    B, T, H, K = np.shape(q)
    HV, V = np.shape(v)[2], np.shape(v)[3]
    G = HV // H
    if scale is None:
        scale = K ** -0.5
    qn, kn, gp, b = _prepare(q, k, g, beta, A_log, dt_bias, gate_mode, lower_bound, qk_l2norm,
                             beta_sigmoid, l2_eps)
    qn = qn.reshape(B * T, H, K)
    kn = kn.reshape(B * T, H, K)
    vv = np.asarray(v, np.float64).reshape(B * T, HV, V)
    gp = gp.reshape(B * T, HV, K)
    b = b.reshape(B * T, HV)
    segs = _segments(B, T, cu_seqlens)
    o = np.zeros((B * T, HV, V))
    fs = np.zeros((len(segs), HV, K, V))
    C = int(chunk_size)
    for n, (bos, eos) in enumerate(segs):
        for hv in range(HV):
            h = hv // G
            S = np.zeros((K, V)) if initial_state is None else \
                np.array(initial_state[n, hv], np.float64)
            for cs in range(bos, eos, C):
                ce = min(cs + C, eos)
                L = ce - cs
                Q = scale * qn[cs:ce, h]           # [L, K]
                Kc = kn[cs:ce, h]
                Vc = vv[cs:ce, hv]
                bc = b[cs:ce, hv]
                Gam = np.cumsum(gp[cs:ce, hv], axis=0)        # step 1
                gC = Gam[L - 1]
                lower = np.tril(np.ones((L, L), bool))         # M
                strict = np.tril(np.ones((L, L), bool), -1)    # M_-1
                D = Gam[:, None, :] - Gam[None, :, :]          # Gamma_i - Gamma_j
                E = np.where(lower[:, :, None], np.exp(np.where(lower[:, :, None], D, 0.0)), 0.0)
                Aqk = np.einsum("ik,jk,ijk->ij", Q, Kc, E)     # step 2
                Akk0 = bc[:, None] * np.where(strict, np.einsum("ik,jk,ijk->ij", Kc, Kc, E), 0.0)
                A = np.linalg.inv(np.eye(L) + Akk0)
                U = A @ (bc[:, None] * Vc)                     # step 3
                W = A @ (np.exp(Gam) * bc[:, None] * Kc)
                Qg = np.exp(Gam) * Q
                Kg = np.exp(gC[None, :] - Gam) * Kc
                Vnew = U - W @ S                               # step 4
                o[cs:ce, hv] = Qg @ S + Aqk @ Vnew             # step 5
                S = np.exp(gC)[:, None] * S + Kg.T @ Vnew
            fs[n, hv] = S
    return o.reshape(B, T, HV, V), fs


def transition_np(q, k, v, g, beta, *, A_log=None, dt_bias=None, gate_mode=GATE_SAFE,
                  lower_bound=None, scale=None, qk_l2norm=True, beta_sigmoid=True,
                  initial_state=None, l2_eps=L2_EPS):
    """Brute force for tiny inputs (no varlen): unrolled sum of explicit transitions.

    With M_t = (I - b_t k_t k_t^T) Diag(a_t) (a K x K matrix) the recurrence reads
    S_t = M_t S_{t-1} + b_t k_t v_t^T, hence
        S_t = (M_t ... M_1) S_0 + sum_{s<=t} (M_t ... M_{s+1}) b_s k_s v_s^T,
    evaluated here term by term with explicit matrix products (O(T^2) products),
    a different evaluation order from the token loop.
    """
    B, T, H, K = np.shape(q)
    HV, V = np.shape(v)[2], np.shape(v)[3]
    G = HV // H
    if scale is None:
        scale = K ** -0.5
    qn, kn, gp, b = _prepare(q, k, g, beta, A_log, dt_bias, gate_mode, lower_bound, qk_l2norm,
                             beta_sigmoid, l2_eps)
    vv = np.asarray(v, np.float64)
    o = np.zeros((B, T, HV, V))
    fs = np.zeros((B, HV, K, V))
    I = np.eye(K)
    for bb in range(B):
        for hv in range(HV):
            h = hv // G
            S0 = np.zeros((K, V)) if initial_state is None else \
                np.array(initial_state[bb, hv], np.float64)
            M = [(I - b[bb, t, hv] * np.outer(kn[bb, t, h], kn[bb, t, h])) @
                 np.diag(np.exp(gp[bb, t, hv])) for t in range(T)]
            for t in range(T):
                St = np.zeros((K, V))
                P = I.copy()                              # P = M_t ... M_{s+1}
                for s in range(t, -1, -1):
                    St = St + P @ (b[bb, s, hv] * np.outer(kn[bb, s, h], vv[bb, s, hv]))
                    P = P @ M[s]
                St = St + P @ S0                          # P = M_t ... M_0 here
                o[bb, t, hv] = scale * St.T @ qn[bb, t, h]
                if t == T - 1:
                    fs[bb, hv] = St
            if T == 0:
                fs[bb, hv] = S0
    return o, fs
