"""GPU parity of the backward pass (kda_bwd, include/kda_bwd.h) against the oracle's fp64
gradients (oracle/backward.py), on the cases the host emulation of the same stage bodies
covers, plus the head dimensions of the long-context workload.  Bounds: bwd_testlib."""
import numpy as np
import pytest

from kimi_delta_attention_gate_gb300 import inputs as kin

import bwd_testlib as bt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_gate_gb300 import build
    build.build()


def check(inp, up_seed=11, chunk_form=False, **opts):
    d_o, dfs = bt.upstream(inp, up_seed, state_v_first=opts.get("state_v_first", False))
    got = bt.run_gpu_bwd(inp, d_o, dfs, **opts)
    ref = bt.oracle_grads(inp, d_o, dfs, chunk_form=chunk_form, **opts)
    return bt.assert_grads_close(got, ref), got


@pytest.mark.parametrize("gate", [kin.GATE_SAFE, kin.GATE_PLAIN, kin.GATE_PREGATED])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gate_modes_and_dtypes(gate, dtype):
    inp = kin.make_inputs(bt.workload(gate=gate, dtype=dtype, seed=20 + gate))
    if gate == kin.GATE_PREGATED:
        bt.pregate(inp)
    check(inp)


@pytest.mark.parametrize("C,T", [(32, 97), (64, 1)])
def test_chunk_sizes_and_ragged_tails(C, T):
    check(kin.make_inputs(bt.workload(C=C, T=T, seed=30 + T)))


def test_grouped_heads_partial_value_tile():
    check(kin.make_inputs(bt.workload(B=1, H=2, HV=6, K=24, V=40, T=90, seed=41)))


def test_full_head_dimensions():
    """K = V = 128 (the long-context workload's heads), bf16, four chunks, two heads."""
    inp = kin.make_inputs(bt.workload(B=1, T=250, H=2, HV=2, K=128, V=128, dtype="bf16",
                                      seed=43, h0_std=0.1))
    check(inp, chunk_form=True)


def test_varlen_with_empty_sequences_and_padding():
    inp = kin.make_inputs(bt.workload(B=1, T=200, seed=44, varlen_n=5, varlen_max_len=60))
    inp.cu_seqlens[:] = np.array([0, 70, 70, 71, 135, 190], dtype=np.int64)
    errs, got = check(inp)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.all(got[name][:, 190:] == 0), name


def test_transposed_state_layout_and_negative_eigenvalues():
    inp = kin.make_inputs(bt.workload(seed=45))
    inp.h0 = np.ascontiguousarray(np.swapaxes(inp.h0, -1, -2))
    check(inp, state_v_first=True, allow_neg_eigval=True)


def test_safe_gate_at_its_bound():
    inp = kin.make_inputs(bt.workload(seed=47, T=128))
    inp.g[:] = np.float32(8.0)
    inp.A_log[:] = np.float32(0.0)
    check(inp)


def test_equal_heads_are_bit_reproducible():
    """With HV == H only dA_log and ddt_bias are summed by atomics."""
    inp = kin.make_inputs(bt.workload(H=2, HV=2, T=130, seed=49))
    d_o, dfs = bt.upstream(inp, 5)
    a = bt.run_gpu_bwd(inp, d_o, dfs)
    b = bt.run_gpu_bwd(inp, d_o, dfs)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert np.array_equal(a[name], b[name]), name
