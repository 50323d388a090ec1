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


def test_tensor_core_states_varlen_grouped_fp32():
    """K = V = 128 at chunk 64 (the shapes whose state stage runs on the tensor cores) with fp32
    inputs, two value heads on one q/k head, and a varlen batch: a sequence of three chunks, an
    empty one, a one-token one and a ragged one of 159 tokens, then padding rows."""
    inp = kin.make_inputs(bt.workload(B=1, T=300, H=1, HV=2, K=128, V=128, C=64, dtype="f32",
                                      seed=61, varlen_n=4, varlen_max_len=100, h0_std=0.1))
    inp.cu_seqlens[:] = np.array([0, 130, 130, 131, 290], dtype=np.int64)
    errs, got = check(inp, chunk_form=True)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.all(got[name][:, 290:] == 0), name


def test_tensor_core_states_and_gradients_varlen_grouped_bf16():
    """The same batch with bf16 inputs, where the state-gradient stage also runs on the tensor
    cores (dO loaded by TMA; the rows of the next sequence inside a ragged chunk zeroed)."""
    inp = kin.make_inputs(bt.workload(B=1, T=300, H=1, HV=2, K=128, V=128, C=64, dtype="bf16",
                                      seed=63, varlen_n=4, varlen_max_len=100, h0_std=0.1))
    inp.cu_seqlens[:] = np.array([0, 130, 130, 131, 290], dtype=np.int64)
    errs, got = check(inp, chunk_form=True)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.all(got[name][:, 290:] == 0), name


def test_tensor_core_states_transposed_layout_and_negative_eigenvalues():
    """The tensor-core state stage with [V, K] states and beta in (0, 2), two sequences."""
    inp = kin.make_inputs(bt.workload(B=2, T=140, H=1, HV=1, K=128, V=128, C=64, dtype="bf16",
                                      seed=62, h0_std=0.1))
    inp.h0 = np.ascontiguousarray(np.swapaxes(inp.h0, -1, -2))
    check(inp, state_v_first=True, allow_neg_eigval=True, chunk_form=True)


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


def test_long_workload_sampled_head():
    """The backward at the bench's full size (long_bf16: one sequence of 65,536 tokens, 32
    heads, K = V = 128) in one launch; head 13's gradients against the chunked oracle over
    the whole sequence (about half a minute of fp64 NumPy)."""
    inp = kin.make_inputs(kin.WORKLOADS["long_bf16"])
    d_o, dfs = bt.upstream(inp, 13)
    got = bt.run_gpu_bwd(inp, d_o, dfs, heads=[13])
    ref = bt.oracle_grads(inp, d_o, dfs, chunk_form=True, heads=[13])
    bt.assert_grads_close(got, ref)


def test_equal_heads_are_bit_reproducible():
    """With HV == H only dA_log and ddt_bias are summed by atomics."""
    inp = kin.make_inputs(bt.workload(H=2, HV=2, T=130, seed=49))
    d_o, dfs = bt.upstream(inp, 5)
    a = bt.run_gpu_bwd(inp, d_o, dfs)
    b = bt.run_gpu_bwd(inp, d_o, dfs)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert np.array_equal(a[name], b[name]), name


def test_stages_one_by_one_give_the_whole_pass():
    """kda_bwd_stage over every stage in order equals kda_bwd (the bench times it that way)."""
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    from kimi_delta_attention_gate_gb300 import _binding as kb
    from kda_testlib import f32_device, gate_kwargs, to_device
    inp = kin.make_inputs(bt.workload(H=2, HV=2, T=150, seed=52, varlen_n=3, varlen_max_len=60,
                                      B=1))
    wl = inp.wl
    d_o, dfs = bt.upstream(inp, 6)
    whole = bt.run_gpu_bwd(inp, d_o, dfs)
    q, k, v, g, b, do = (to_device(x, wl.dtype) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta, d_o))
    cu_cpu = torch.from_numpy(inp.cu_seqlens)
    # every device tensor the parameter blocks point at stays bound until the launches ran
    cu_dev = cu_cpu.cuda()
    A_log, dt_bias, h0 = f32_device(inp.A_log), f32_device(inp.dt_bias), f32_device(inp.h0)
    f = kda.make_params(q, k, v, g, b, A_log=A_log, dt_bias=dt_bias, scale=inp.scale,
                        initial_state=h0, cu_seqlens=cu_dev, cu_seqlens_cpu=cu_cpu,
                        chunk_size=wl.chunk_size, **gate_kwargs(wl))
    outs = {n: torch.full(s, float("nan"), dtype=torch.float32, device="cuda") for n, s in
            (("dq", q.shape), ("dk", k.shape), ("dv", v.shape), ("dg", g.shape),
             ("dbeta", b.shape), ("dA_log", (wl.HV,)), ("ddt_bias", (wl.HV * wl.K,)),
             ("dh0", tuple(inp.h0.shape)))}
    dht = f32_device(dfs)
    p = kb.kda_bwd_params()
    p.fwd = f
    p.d_o, p.d_final_state = do.data_ptr(), dht.data_ptr()
    for n, t in outs.items():
        setattr(p, n, t.data_ptr())
    ws = torch.empty(kb.kda_bwd_workspace_size(p), dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    sh = torch.cuda.current_stream().cuda_stream
    nst = kb.kda_bwd_num_stages(p)
    assert [kb.kda_bwd_stage_name(p, i) for i in range(nst)][:2] == ["zero_outputs", "chunk_table"]
    for i in range(nst):
        kb.raise_for(kb.kda_bwd_stage(p, sh, i))
    torch.cuda.synchronize()
    assert kda.kda_get_device_status(0) == 0
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert np.array_equal(outs[n].cpu().double().numpy(), whole[n]), n
    for n in ("dA_log", "ddt_bias"):
        assert bt.rel_l2(outs[n].cpu().double().numpy(), whole[n]) < 1e-6, n


@pytest.mark.parametrize("seed", range(100, 108))
def test_random_shapes(seed):
    """Seeded random configurations (the first half of the host emulation's sweep)."""
    inp, opts = bt.random_case(seed)
    check(inp, chunk_form=True, **opts)
