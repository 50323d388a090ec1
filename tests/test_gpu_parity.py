"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.  Tolerances on o and final_state: bf16 inputs rel-L2 <= 5e-3
and max-abs <= 3e-2; fp32 inputs rel-L2 <= 1e-4."""
import dataclasses

import numpy as np
import pytest

from kimi_delta_attention_gate_gb300 import inputs as kin

from kda_testlib import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_gate_gb300 import build
    build.build()


def small(name="s", *, B=1, T=100, H=2, HV=2, K=64, V=64, C=64, dtype="bf16",
          gate=kin.GATE_SAFE, lb=-5.0, h0=0.1, varlen=0, maxlen=0, seed=7, dt=True, alog=True):
    return kin.Workload(name, B=B, T=T, H=H, HV=HV, K=K, V=V, chunk_size=C, dtype=dtype, gate=gate,
                        lower_bound=lb if gate == kin.GATE_SAFE else None, h0_std=h0,
                        varlen_n=varlen, varlen_max_len=maxlen, seed=seed, has_dt_bias=dt,
                        has_a_log=alog, a_log_mean=-1.0 if gate == kin.GATE_PLAIN else 0.0,
                        a_log_std=0.5 if gate == kin.GATE_PLAIN else 1.0)


def check_case(wl, chunk_size=None, heads=None):
    inp = kin.make_inputs(wl)
    o, fs = run_gpu(inp, chunk_size=chunk_size)
    ro, rfs = run_oracle(inp, heads=heads)
    if heads is not None:
        o, fs = o[:, :, heads], fs[:, heads]
    assert_close(o, ro, wl.dtype, "o")
    assert_close(fs, rfs, wl.dtype, "final_state")


# ---- the five workloads --------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny_fp32", "equal_bf16", "gva_bf16", "varlen_bf16"])
def test_workload_full(name):
    check_case(kin.WORKLOADS[name])


def test_long_bf16_sampled_heads():
    """T=65536, H=32: the full launch, compared on sampled value heads."""
    check_case(kin.WORKLOADS["long_bf16"], heads=[0, 13, 31])


@pytest.mark.parametrize("name", ["tiny_fp32", "equal_bf16"])
def test_workload_chunk32(name):
    check_case(kin.WORKLOADS[name], chunk_size=32)


# ---- edge cases -----------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 130])
@pytest.mark.parametrize("C", [32, 64])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_lengths(T, C, dtype):
    check_case(small(T=T, C=C, dtype=dtype, seed=T * 3 + C))


@pytest.mark.parametrize("gate", [kin.GATE_SAFE, kin.GATE_PLAIN, kin.GATE_PREGATED])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gate_modes(gate, dtype):
    wl = small(T=150, gate=gate, dtype=dtype, seed=40 + gate)
    if gate == kin.GATE_PREGATED:
        inp = kin.make_inputs(wl)
        inp.g[:] = -np.abs(inp.g) * 0.5            # a non-positive log decay
        o, fs = run_gpu(inp)
        ro, rfs = run_oracle(inp)
        assert_close(o, ro, dtype, "o")
        assert_close(fs, rfs, dtype, "final_state")
    else:
        check_case(wl)


def test_safe_gate_without_alog_and_dt_bias():
    check_case(small(T=90, alog=False, dt=False, seed=51))


@pytest.mark.parametrize("K,V", [(48, 40), (256, 256), (128, 32), (32, 200)])
def test_head_dims(K, V):
    check_case(small(T=80, K=K, V=V, seed=K + V))


def test_gva_groups():
    check_case(small(T=130, H=2, HV=6, seed=61))


def test_varlen_with_empty_and_single_token_sequences():
    wl = small(T=400, varlen=6, maxlen=120, seed=71)
    inp = kin.make_inputs(wl)
    inp.cu_seqlens[:] = np.array([0, 1, 1, 65, 66, 130, 300], dtype=np.int64)
    o, fs = run_gpu(inp)
    ro, rfs = run_oracle(inp)
    assert_close(o, ro, "bf16", "o")
    assert_close(fs, rfs, "bf16", "final_state")
    assert np.all(o[:, 300:] == 0)


def test_empty_sequence_axis():
    """T = 0: nothing to compute; final_state equals the initial state."""
    wl = small(T=0, seed=81)
    inp = kin.make_inputs(wl)
    o, fs = run_gpu(inp)
    assert o.shape == (1, 0, 2, 64)
    assert np.array_equal(fs, inp.h0.astype(np.float64))


def test_resume_chaining_matches_one_call():
    wl = small(T=200, dtype="f32", seed=91)
    inp = kin.make_inputs(wl)
    o, fs = run_gpu(inp)
    a = dataclasses.replace(inp, q=inp.q[:, :77].copy(), k=inp.k[:, :77].copy(),
                            v=inp.v[:, :77].copy(), g=inp.g[:, :77].copy(),
                            beta=inp.beta[:, :77].copy(), wl=dataclasses.replace(wl, T=77))
    oa, fa = run_gpu(a)
    b = dataclasses.replace(inp, q=inp.q[:, 77:].copy(), k=inp.k[:, 77:].copy(),
                            v=inp.v[:, 77:].copy(), g=inp.g[:, 77:].copy(),
                            beta=inp.beta[:, 77:].copy(), h0=fa.astype(np.float32),
                            wl=dataclasses.replace(wl, T=123))
    ob, fb = run_gpu(b)
    assert_close(np.concatenate([oa, ob], axis=1), o, "f32", "o")
    assert_close(fb, fs, "f32", "final_state")


def test_repeat_calls_are_deterministic():
    inp = kin.make_inputs(small(T=100, seed=101))
    o1, f1 = run_gpu(inp)
    o2, f2 = run_gpu(inp)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)


# ---- bf16 tensor-core path (K = V = 128, chunk 64) ---------------------------------------

def tc(**kw):
    kw.setdefault("K", 128)
    kw.setdefault("V", 128)
    return small(**kw)


@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 130, 300])
def test_tc_ragged_lengths(T):
    check_case(tc(T=T, seed=200 + T))


@pytest.mark.parametrize("gate", [kin.GATE_SAFE, kin.GATE_PLAIN, kin.GATE_PREGATED])
def test_tc_gate_modes(gate):
    wl = tc(T=200, B=2, gate=gate, seed=300 + gate)
    inp = kin.make_inputs(wl)
    if gate == kin.GATE_PREGATED:
        inp.g[:] = kin.round_to_bf16(-np.abs(inp.g) * 0.5)
    o, fs = run_gpu(inp)
    ro, rfs = run_oracle(inp)
    assert_close(o, ro, "bf16", "o")
    assert_close(fs, rfs, "bf16", "final_state")


def test_tc_plain_gate_exact_diagonal_guard():
    """A plain gate with exp(A_log) ~ 20 decays a 16-token block far beyond 2^120: the
    diagonal blocks must come from the exact element-wise evaluation."""
    wl = tc(T=160, gate=kin.GATE_PLAIN, seed=311)
    inp = kin.make_inputs(wl)
    inp.A_log[:] = 3.0
    o, fs = run_gpu(inp)
    ro, rfs = run_oracle(inp)
    assert_close(o, ro, "bf16", "o")
    assert_close(fs, rfs, "bf16", "final_state")


def test_tc_safe_gate_at_lower_bound():
    """Safe gate saturated at lower_bound = -5: 16 tokens decay by 2^-115 (the largest
    in-block factor the block references must hold)."""
    wl = tc(T=192, seed=321)
    inp = kin.make_inputs(wl)
    inp.g[:] = kin.round_to_bf16(np.abs(inp.g) + 4.0)
    o, fs = run_gpu(inp)
    ro, rfs = run_oracle(inp)
    assert_close(o, ro, "bf16", "o")
    assert_close(fs, rfs, "bf16", "final_state")


def test_tc_gva_and_no_alog():
    check_case(tc(T=130, H=2, HV=4, seed=331))
    check_case(tc(T=90, alog=False, dt=False, seed=332))


def test_tc_varlen_with_empty_and_single_token_sequences():
    wl = tc(T=400, varlen=6, maxlen=120, seed=341)
    inp = kin.make_inputs(wl)
    inp.cu_seqlens[:] = np.array([0, 1, 1, 65, 66, 130, 300], dtype=np.int64)
    o, fs = run_gpu(inp)
    ro, rfs = run_oracle(inp)
    assert_close(o, ro, "bf16", "o")
    assert_close(fs, rfs, "bf16", "final_state")
    assert np.all(o[:, 300:] == 0)


def test_tc_path_is_selected():
    import kimi_delta_attention_gate_gb300 as kda
    from kimi_delta_attention_gate_gb300 import _binding as kb
    import torch
    q = torch.zeros((1, 64, 2, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((1, 64, 2, 128), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((1, 64, 2), dtype=torch.bfloat16, device="cuda")
    p = kda.make_params(q, q, v, v, b, lower_bound=-5.0, o=v)
    names = [kb.kda_fwd_stage_name(p, i) for i in range(kb.kda_fwd_num_stages(p))]
    assert names == ["tc_intra", "tc_recur"]


# ---- pipelined schedule: segments of the chunk range on two streams ---------------------------

def check_pipelined(inp):
    from kda_testlib import run_gpu_stages
    o, fs = run_gpu(inp)
    ro, rfs = run_oracle(inp)
    assert_close(o, ro, "bf16", "o")
    assert_close(fs, rfs, "bf16", "final_state")
    # the carried fp32 state makes the segmented schedule bit-identical to one launch per stage
    so, sfs = run_gpu_stages(inp)
    assert np.array_equal(o, so) and np.array_equal(fs, sfs)


@pytest.mark.parametrize("gate", [kin.GATE_SAFE, kin.GATE_PLAIN])
def test_tc_pipelined_one_long_sequence(gate):
    """257 chunks of one sequence: two segments, the state carried between them."""
    check_pipelined(kin.make_inputs(tc(T=64 * 256 + 37, gate=gate, seed=400 + gate)))


def test_tc_pipelined_six_segments():
    """640 chunks: six segments."""
    check_pipelined(kin.make_inputs(tc(T=64 * 640, H=1, HV=1, seed=402)))


def test_tc_pipelined_batch_boundary_inside_a_sequence():
    """B=3 x 91 chunks: the segment boundary (chunk 136) falls inside the second sequence."""
    check_pipelined(kin.make_inputs(tc(B=3, T=64 * 90 + 10, seed=405)))


def test_tc_pipelined_varlen_with_empty_sequences():
    """Varlen with an empty sequence in the middle and one at the end; the boundary (chunk
    133) falls inside the third sequence."""
    wl = tc(T=17037, varlen=5, maxlen=9100, seed=410)
    inp = kin.make_inputs(wl)
    inp.cu_seqlens[:] = np.array([0, 8000, 8000, 17000, 17037, 17037], dtype=np.int64)
    check_pipelined(inp)



# ---- allow_neg_eigval and the transposed ([V, K]) state layout ---------------------------------

@pytest.mark.parametrize("dtype,K", [("bf16", 128), ("f32", 64)])
def test_allow_neg_eigval(dtype, K):
    """beta = 2 sigmoid(logit) in [0, 2) on both paths (bf16 tensor-core, fp32 CUDA-core)."""
    inp = kin.make_inputs(small(T=150, K=K, V=K, dtype=dtype, seed=500 + K))
    o, fs = run_gpu(inp, allow_neg_eigval=True)
    ro, rfs = run_oracle(inp, allow_neg_eigval=True)
    assert_close(o, ro, dtype, "o")
    assert_close(fs, rfs, dtype, "final_state")


@pytest.mark.parametrize("dtype,K,T", [("bf16", 128, 150), ("f32", 64, 150),
                                       ("bf16", 128, 64 * 256 + 37)])
def test_transposed_state_layout(dtype, K, T):
    """Initial and final states as [N, HV, V, K]; the last case runs the pipelined schedule,
    whose carried state between segments stays internal."""
    wl = small(T=T, K=K, V=K, dtype=dtype, seed=510 + K + T)
    inp = kin.make_inputs(wl)
    inp.h0 = np.ascontiguousarray(np.swapaxes(inp.h0, -1, -2))
    o, fs = run_gpu(inp, transpose_state_layout=True)
    ro, rfs = run_oracle(inp, transpose_state_layout=True)
    assert fs.shape == (1, wl.HV, wl.V, wl.K)
    assert_close(o, ro, dtype, "o")
    assert_close(fs, rfs, dtype, "final_state")



# ---- per-chunk states (return_intermediate_states) -------------------------------------------

@pytest.mark.parametrize("dtype,K,T,transposed", [("bf16", 128, 300, False), ("f32", 64, 200, False),
                                                  ("bf16", 128, 64 * 256 + 37, False),
                                                  ("bf16", 128, 150, True)])
def test_intermediate_states(dtype, K, T, transposed):
    """The state before every chunk, on both paths; the third case runs the pipelined schedule
    (segments in the middle of the sequence), the last the transposed layout."""
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    from kda_testlib import f32_device, gate_kwargs, to_device
    wl = small(T=T, K=K, V=K, dtype=dtype, seed=520 + K + T)
    inp = kin.make_inputs(wl)
    if transposed:
        inp.h0 = np.ascontiguousarray(np.swapaxes(inp.h0, -1, -2))
    q, k, v, g, b = (to_device(x, dtype) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    o, fs, hs = kda.kda_fwd(q, k, v, g, b, A_log=f32_device(inp.A_log),
                            dt_bias=f32_device(inp.dt_bias), scale=inp.scale,
                            initial_state=f32_device(inp.h0), return_intermediate_states=True,
                            transpose_state_layout=transposed, **gate_kwargs(wl))
    torch.cuda.synchronize()
    ro, rfs, rhs = run_oracle(inp, return_intermediate_states=True, chunk_size=64,
                              transpose_state_layout=transposed)
    assert hs.shape == rhs.shape == ((T + 63) // 64, wl.HV) + rfs.shape[2:]
    assert_close(hs.cpu().double().numpy(), rhs, dtype, "intermediate states")
    assert_close(o.float().cpu().double().numpy(), ro, dtype, "o")


# ---- CUDA graph capture -------------------------------------------------------------------------

def test_pipelined_schedule_replays_from_a_cuda_graph():
    """The pipelined schedule (internal streams joined back by events) captures into a CUDA
    graph; replays with new inputs copied into the captured buffers give bit for bit what direct
    calls give."""
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    from kda_testlib import f32_device, gate_kwargs, to_device
    wl = tc(T=64 * 256 + 37, seed=700)
    inps = [kin.make_inputs(wl), kin.make_inputs(tc(T=64 * 256 + 37, seed=701))]
    dev = [tuple(to_device(x, "bf16") for x in (i.q, i.k, i.v, i.g, i.beta)) for i in inps]
    q, k, v, g, b = (x.clone() for x in dev[0])
    A, dt, h0 = f32_device(inps[0].A_log), f32_device(inps[0].dt_bias), f32_device(inps[0].h0)
    o = torch.empty_like(v)
    fs = torch.empty(h0.shape, dtype=torch.float32, device="cuda")
    p = kda.make_params(q, k, v, g, b, A_log=A, dt_bias=dt, scale=inps[0].scale, initial_state=h0,
                        final_state=fs, o=o, **gate_kwargs(wl))
    ws = torch.empty(kda.kda_fwd_workspace_size(p), dtype=torch.uint8, device="cuda")
    call = dict(A_log=A, dt_bias=dt, scale=inps[0].scale, initial_state=h0, workspace=ws, o=o,
                final_state=fs, **gate_kwargs(wl))
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        kda.kda_fwd(q, k, v, g, b, **call)  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        kda.kda_fwd(q, k, v, g, b, **call)
    for src in dev:
        for dst, x in zip((q, k, v, g, b), src):
            dst.copy_(x)
        graph.replay()
        torch.cuda.synchronize()
        go, gfs = o.clone(), fs.clone()
        ro, rfs = kda.kda_fwd(*src, **{**call, "o": None, "final_state": None})
        torch.cuda.synchronize()
        assert torch.equal(go, ro) and torch.equal(gfs, rfs)
    assert kda.kda_get_device_status(0) == 0
