"""GPU tests of context parallelism (kimi_delta_attention_gate_gb300.cp): the affine-map
kernel against a NumPy product, and a sequence cut into shards whose maps are formed by the
CUDA forward pass, chained on the GPU and used as each shard's initial state, against the
oracle over the whole sequence (the shards run one after another in this process, as the
ranks of a group would run side by side)."""
import os

import numpy as np
import pytest

from kimi_delta_attention_gate_gb300 import inputs as kin

from kda_testlib import assert_close, f32_device, gate_kwargs, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_gate_gb300 import _binding as kb
    from kimi_delta_attention_gate_gb300 import build
    build.build()
    kb.load()


@pytest.mark.parametrize("K,V,v_first,with_s", [(128, 128, 0, 1), (64, 40, 1, 1), (256, 256, 0, 0),
                                                (5, 70, 0, 1), (96, 33, 1, 0)])
def test_affine_apply_matches_numpy(K, V, v_first, with_s):
    import torch
    from kimi_delta_attention_gate_gb300 import cp
    r = np.random.default_rng(K + V)
    n = 7
    P = (r.standard_normal((n, K, K)) / np.sqrt(K)).astype(np.float32)
    st = (n, V, K) if v_first else (n, K, V)
    R = r.standard_normal(st).astype(np.float32)
    S = r.standard_normal(st).astype(np.float32) if with_s else None
    out = cp.affine_apply(torch.from_numpy(P).cuda(), torch.from_numpy(R).cuda(),
                          None if S is None else torch.from_numpy(S).cuda(), state_v_first=bool(v_first))
    torch.cuda.synchronize()
    P64, R64 = P.astype(np.float64), R.astype(np.float64)
    if S is None:
        ref = R64
    elif v_first:
        ref = S.astype(np.float64) @ np.swapaxes(P64, -1, -2) + R64
    else:
        ref = P64 @ S.astype(np.float64) + R64
    got = out.cpu().double().numpy()
    assert np.max(np.abs(got - ref)) < 1e-4 * max(1.0, np.max(np.abs(ref)))


def test_affine_apply_rejects_bad_arguments():
    import torch
    from kimi_delta_attention_gate_gb300 import _binding as kb
    P = torch.zeros((2, 4, 4), device="cuda")
    R = torch.zeros((2, 4, 3), device="cuda")
    assert kb.kda_state_affine_apply(P.data_ptr(), R.data_ptr(), None, R.data_ptr(), 2, 4, 3, 0,
                                     0) == kb.KDA_ERR_INVALID_ARG
    assert kb.kda_state_affine_apply(P.data_ptr(), R.data_ptr(), None, P.data_ptr() + 1, 2, 4, 3, 0,
                                     0) == kb.KDA_ERR_INVALID_ARG
    assert kb.kda_state_affine_apply(P.data_ptr(), R.data_ptr(), None, R.data_ptr(), 2, 300, 3, 0,
                                     0) == kb.KDA_ERR_SHAPE
    assert kb.kda_state_affine_apply(0, 0, 0, 0, 0, 4, 3, 0, 0) == kb.KDA_OK


def _sharded(inp, bounds, **opts):
    """Every shard's map by the CUDA forward pass, chained on the GPU, then each shard run
    from the state entering it; returns (o over all shards, final state) as float64."""
    import torch
    from kimi_delta_attention_gate_gb300 import cp
    import kimi_delta_attention_gate_gb300 as kda
    wl = inp.wl
    dev = lambda x: to_device(np.ascontiguousarray(x), wl.dtype)
    kw = dict(A_log=f32_device(inp.A_log), dt_bias=f32_device(inp.dt_bias), scale=inp.scale,
              **gate_kwargs(wl), **opts)
    shards = [tuple(dev(x[:, t0:t1]) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
              for t0, t1 in zip(bounds[:-1], bounds[1:])]
    maps = [cp.state_map(*s, **kw) for s in shards]
    h0 = f32_device(inp.h0)
    states = cp.chain([m[0] for m in maps], [m[1] for m in maps], h0,
                      state_v_first=bool(opts.get("transpose_state_layout")))
    outs = [kda.kda_fwd(*s, initial_state=s_in, **kw) for s, s_in in zip(shards, states[:-1])]
    torch.cuda.synchronize()
    o = np.concatenate([x[0].float().cpu().double().numpy() for x in outs], axis=1)
    # the last shard's final state and the chain's last state are the same quantity
    fs_last = outs[-1][1].cpu().double().numpy()
    fs_chain = states[-1].cpu().double().numpy()
    return o, fs_last, fs_chain


def _wl(**kw):
    gate = kw.pop("gate", kin.GATE_SAFE)
    return kin.Workload(kw.pop("name", "cp"), chunk_size=64, gate=gate,
                        lower_bound=-5.0 if gate == kin.GATE_SAFE else None, h0_std=0.1,
                        has_dt_bias=True, has_a_log=True, a_log_mean=0.0, a_log_std=1.0, **kw)


@pytest.mark.parametrize("bounds", [(0, 4000, 9000, 16421), (0, 16421)])
def test_bf16_shards_equal_the_whole_sequence(bounds):
    """Three shards with boundaries inside chunks (tensor-core path; the longest shard takes
    the pipelined schedule) equal the oracle on the whole sequence."""
    inp = kin.make_inputs(_wl(B=2, T=16421, H=2, HV=2, K=128, V=128, dtype="bf16", seed=700))
    o, fs, fsc = _sharded(inp, bounds)
    ro, rfs = run_oracle(inp)
    assert_close(o, ro, "bf16", "o")
    assert_close(fs, rfs, "bf16", "final_state")
    assert_close(fsc, rfs, "bf16", "final_state (chained)")


def test_fp32_shards_grouped_heads_transposed_states():
    inp = kin.make_inputs(_wl(B=1, T=700, H=1, HV=3, K=64, V=48, dtype="f32", seed=701,
                              gate=kin.GATE_PLAIN))
    inp.h0 = np.ascontiguousarray(np.swapaxes(inp.h0, -1, -2))
    o, fs, fsc = _sharded(inp, (0, 130, 131, 700), transpose_state_layout=True,
                          allow_neg_eigval=True)
    ro, rfs = run_oracle(inp, transpose_state_layout=True, allow_neg_eigval=True)
    assert_close(o, ro, "f32", "o")
    assert_close(fs, rfs, "f32", "final_state")
    assert_close(fsc, rfs, "f32", "final_state (chained)")


def test_cp_fwd_on_a_one_rank_nccl_group():
    """cp_fwd itself (all-gather of CUDA tensors over NCCL) on a group of one rank."""
    import torch
    import torch.distributed as dist
    from kimi_delta_attention_gate_gb300 import cp
    inp = kin.make_inputs(_wl(B=1, T=300, H=2, HV=2, K=128, V=128, dtype="bf16", seed=702))
    wl = inp.wl
    port = 32000 + os.getpid() % 1000
    dist.init_process_group("nccl", rank=0, world_size=1, init_method=f"tcp://127.0.0.1:{port}")
    try:
        q, k, v, g, b = (to_device(x, wl.dtype) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
        o, fs = cp.cp_fwd(q, k, v, g, b, initial_state=f32_device(inp.h0),
                          A_log=f32_device(inp.A_log), dt_bias=f32_device(inp.dt_bias),
                          scale=inp.scale, **gate_kwargs(wl))
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    ro, rfs = run_oracle(inp)
    assert_close(o.float().cpu().double().numpy(), ro, "bf16", "o")
    assert_close(fs.cpu().double().numpy(), rfs, "bf16", "final_state")
