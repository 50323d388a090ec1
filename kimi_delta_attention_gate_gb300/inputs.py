"""Seeded synthetic inputs for the chunk-parallel KDA forward pass.

This module draws random tensors and nothing else: it holds none of the
method's arithmetic (no gate, no norm, no recurrence).  Both the CUDA path
(tests, bench, smoke check) and the CPU oracle are fed from it, so the two
see bit-identical inputs.

Generator: ``numpy.random.Generator(PCG64(seed))``.  Values are drawn in
float32; for bf16 workloads they are rounded to the nearest bf16 (ties to
even) and kept as float32 arrays whose values are exactly representable in
bf16.  ``to_bf16_bits`` gives the 16-bit patterns for upload.

Tensor layouts follow the FLA ``chunk_kda`` contract (FLA-KDA engineering
notes, section 2 "gate input contracts" and 2.1 "parameter checks"):
q, k ``[B,T,H,K]``; v ``[B,T,HV,V]``; g ``[B,T,HV,K]``; beta ``[B,T,HV]``;
A_log ``[HV]`` fp32; dt_bias ``[HV*K]`` fp32; h0 ``[N,HV,K,V]`` fp32.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

GATE_PREGATED = 0
GATE_PLAIN = 1
GATE_SAFE = 2


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, dtype and the distributions drawn."""

    name: str
    B: int
    T: int
    H: int
    HV: int
    K: int
    V: int
    chunk_size: int
    dtype: str                 # "f32" or "bf16": q,k,v,g,beta and o
    gate: int                  # GATE_SAFE / GATE_PLAIN / GATE_PREGATED
    lower_bound: Optional[float]
    a_log_mean: float = 0.0
    a_log_std: float = 1.0
    has_a_log: bool = True
    has_dt_bias: bool = True
    h0_std: Optional[float] = None     # None -> no initial state (zeros)
    varlen_n: int = 0                  # >0 -> B==1 buffer with this many sequences
    varlen_max_len: int = 0
    seed: int = 0

    @property
    def G(self) -> int:
        return self.HV // self.H


# The five workloads the method is measured and checked on.  Index i (1-based)
# uses seed 1000 + i.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", B=1, T=256, H=2, HV=2, K=64, V=64, chunk_size=64,
                          dtype="f32", gate=GATE_SAFE, lower_bound=-5.0, seed=1001),
    "equal_bf16": Workload("equal_bf16", B=4, T=2048, H=4, HV=4, K=128, V=128, chunk_size=64,
                           dtype="bf16", gate=GATE_SAFE, lower_bound=-5.0, h0_std=0.1, seed=1002),
    "gva_bf16": Workload("gva_bf16", B=2, T=4096, H=4, HV=8, K=128, V=128, chunk_size=64,
                         dtype="bf16", gate=GATE_PLAIN, lower_bound=None, a_log_mean=-1.0,
                         a_log_std=0.5, has_dt_bias=False, seed=1003),
    "varlen_bf16": Workload("varlen_bf16", B=1, T=32768, H=16, HV=16, K=128, V=128, chunk_size=64,
                            dtype="bf16", gate=GATE_SAFE, lower_bound=-5.0, h0_std=0.1,
                            varlen_n=8, varlen_max_len=8191, seed=1004),
    "long_bf16": Workload("long_bf16", B=1, T=65536, H=32, HV=32, K=128, V=128, chunk_size=64,
                          dtype="bf16", gate=GATE_SAFE, lower_bound=-5.0, seed=1005),
    # decode step of the token-recurrent entry point: 256 sequences of one token each
    "decode_bf16": Workload("decode_bf16", B=256, T=1, H=32, HV=32, K=128, V=128, chunk_size=64,
                            dtype="bf16", gate=GATE_SAFE, lower_bound=-5.0, h0_std=0.1,
                            seed=1006),
}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even), in place; returns x."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    u += bias
    u &= np.uint32(0xFFFF0000)
    return x


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-representable."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u >> np.uint32(16)).astype(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """float32 values of bf16 bit patterns."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def draw_varlen_lengths(rng: np.random.Generator, n: int, max_len: int, total: int) -> np.ndarray:
    """n lengths i.i.d. uniform on {1..max_len}, redrawn as a set until they fit in ``total``."""
    while True:
        lens = rng.integers(1, max_len + 1, size=n, dtype=np.int64)
        if int(lens.sum()) <= total:
            return lens


@dataclasses.dataclass
class Inputs:
    """A drawn workload.  Arrays are float32 (exact in ``dtype``), C-contiguous."""

    wl: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray            # logits; the kernel applies the sigmoid
    A_log: Optional[np.ndarray]
    dt_bias: Optional[np.ndarray]
    h0: Optional[np.ndarray]
    cu_seqlens: Optional[np.ndarray]   # int64 [N+1] or None
    scale: float

    @property
    def N(self) -> int:
        return self.wl.B if self.cu_seqlens is None else len(self.cu_seqlens) - 1

    @property
    def n_tokens(self) -> int:
        """Real tokens (padding excluded)."""
        if self.cu_seqlens is None:
            return self.wl.B * self.wl.T
        return int(self.cu_seqlens[-1])


def _normal(rng: np.random.Generator, shape, mean=0.0, std=1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return x


def make_inputs(wl: Workload, seed: Optional[int] = None, *, T: Optional[int] = None,
                B: Optional[int] = None) -> Inputs:
    """Draw the inputs of ``wl`` (optionally with a different seed, T or B).

    Draw order is fixed: [varlen lengths], q, k, v, g, beta, A_log, dt_bias, h0.
    """
    if T is not None or B is not None:
        wl = dataclasses.replace(wl, T=T if T is not None else wl.T, B=B if B is not None else wl.B)
    rng = np.random.Generator(np.random.PCG64(wl.seed if seed is None else seed))
    cu = None
    if wl.varlen_n > 0:
        assert wl.B == 1
        lens = draw_varlen_lengths(rng, wl.varlen_n, wl.varlen_max_len, wl.T)
        cu = np.zeros(wl.varlen_n + 1, dtype=np.int64)
        cu[1:] = np.cumsum(lens)
    B, T, H, HV, K, V = wl.B, wl.T, wl.H, wl.HV, wl.K, wl.V
    q = _normal(rng, (B, T, H, K))
    k = _normal(rng, (B, T, H, K))
    v = _normal(rng, (B, T, HV, V))
    g = _normal(rng, (B, T, HV, K))
    beta = _normal(rng, (B, T, HV))
    A_log = _normal(rng, (HV,), wl.a_log_mean, wl.a_log_std) if wl.has_a_log else None
    dt_bias = _normal(rng, (HV * K,)) if wl.has_dt_bias else None
    N = B if cu is None else len(cu) - 1
    h0 = _normal(rng, (N, HV, K, V), 0.0, wl.h0_std) if wl.h0_std is not None else None
    if wl.dtype == "bf16":
        for x in (q, k, v, g, beta):
            round_to_bf16(x)
    return Inputs(wl=wl, q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias, h0=h0,
                  cu_seqlens=cu, scale=float(K) ** -0.5)
