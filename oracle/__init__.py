"""CPU fp64 oracle for the chunk-parallel KDA forward pass.

TEST INFRASTRUCTURE ONLY.  The test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only users; the CUDA library neither
imports nor links anything here, and nothing here imports the CUDA library.

Contents
  * ``fwd``            -- the oracle proper: the C fp64 token recurrence
                          (``kda_oracle.c``), OpenMP over (sequence, value head).
  * ``gate_np``        -- gate activation, NumPy fp64.
  * ``recurrent_np``   -- the same token recurrence in NumPy (cross-check).
  * ``chunk_np``       -- the chunk-parallel form, steps 1-5 of the forward pass
                          in "KDA reading notes: Implementation Notes for KDA in
                          FLA", written out with a dense solve (cross-check).
  * ``transition_np``  -- brute force: explicit K x K transition matrices.
  * ``backward.bwd``   -- fp64 gradients of the forward (PyTorch autograd over the
                          token recurrence), the reference for a backward pass;
                          ``backward.chunk_bwd_np`` the same gradients derived by hand
                          through the chunk form.

Every function is pinned by ``tests/test_oracle_pins.py`` (``backward`` by
``tests/test_oracle_backward.py``) against things the pages and the mathematics
fix (closed forms, special cases, identities, finite differences of ``fwd``).
"""
from .ref import (GATE_PLAIN, GATE_PREGATED, GATE_SAFE, L2_EPS, build, chunk_np, fwd, gate_c, gate_np,
                  l2norm_np, lib_path, max_threads, recurrent_np, sigmoid_np, softplus_np,
                  transition_np)

__all__ = [
    "GATE_PLAIN", "GATE_PREGATED", "GATE_SAFE", "L2_EPS", "build", "chunk_np", "fwd", "gate_c", "gate_np",
    "l2norm_np", "lib_path", "max_threads", "recurrent_np", "sigmoid_np", "softplus_np",
    "transition_np",
]
