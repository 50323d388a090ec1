"""kda_fwd_noalloc: the allocation-free entry point, against kda_fwd.

Some callers cannot allocate device memory (no cudaMalloc, no allocator handle
to give the library a workspace).  kda_fwd_noalloc serves them from a static
device array inside the library.  This test calls it through the C ABI twice in
a row, on different inputs, and checks each result against kda_fwd (which runs
with a caller-provided workspace) within the tolerance the parity tests use.
It sits in a file of its own, collected after the other forward tests."""
import numpy as np
import pytest

from kimi_delta_attention_gate_gb300 import inputs as kin

from kda_testlib import TOL, errors, f32_device, to_device

pytestmark = pytest.mark.gpu


def _inputs(seed):
    wl = kin.Workload("noalloc", B=2, T=150, H=2, HV=4, K=128, V=128, chunk_size=64,
                      dtype="bf16", gate=kin.GATE_SAFE, lower_bound=-5.0, h0_std=0.1, seed=seed)
    return kin.make_inputs(wl)


def _tensors(inp):
    wl = inp.wl
    q, k, v, g, b = (to_device(x, wl.dtype) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    return q, k, v, g, b, f32_device(inp.A_log), f32_device(inp.dt_bias), f32_device(inp.h0)


def test_noalloc_matches_kda_fwd_on_two_calls_in_a_row():
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    from kimi_delta_attention_gate_gb300 import _binding as kb
    from kimi_delta_attention_gate_gb300 import build
    build.build()
    kb.load()
    stream = torch.cuda.current_stream()
    for seed in (11, 12):
        inp = _inputs(seed)
        q, k, v, g, b, A_log, dt_bias, h0 = _tensors(inp)
        common = dict(A_log=A_log, dt_bias=dt_bias, lower_bound=-5.0, scale=inp.scale,
                      initial_state=h0)
        o_ref, fs_ref = kda.kda_fwd(q, k, v, g, b, **common)
        o = torch.empty_like(o_ref)
        fs = torch.empty_like(fs_ref)
        p = kda.make_params(q, k, v, g, b, o=o, final_state=fs, **common)
        assert kb.kda_fwd_workspace_size(p) <= kb.NOALLOC_SCRATCH_BYTES
        rc = kb.kda_fwd_noalloc(p, stream.cuda_stream)
        assert rc == kb.KDA_OK, kb.kda_last_error()
        torch.cuda.synchronize()
        assert kb.kda_get_device_status(stream.cuda_stream) == 0
        tol = TOL["bf16"]
        for got, ref, what in ((o, o_ref, "o"), (fs, fs_ref, "final_state")):
            gn = got.float().cpu().double().numpy()
            rn = ref.float().cpu().double().numpy()
            assert np.all(np.isfinite(gn))
            rel, mx = errors(gn, rn)
            assert rel <= tol["rel_l2"] and mx <= tol["max_abs"], (seed, what, rel, mx)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    from kimi_delta_attention_gate_gb300 import _binding as kb
    T = 8192   # 2 x 4 heads x 128 chunks of fp32 intermediates: well beyond 32 MiB
    q = torch.zeros((2, T, 2, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((2, T, 4, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((2, T, 4, 128), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((2, T, 4), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(v)
    p = kda.make_params(q, q, v, g, b, lower_bound=-5.0, o=o)
    assert kb.kda_fwd_workspace_size(p) > kb.NOALLOC_SCRATCH_BYTES
    rc = kb.kda_fwd_noalloc(p, torch.cuda.current_stream().cuda_stream)
    assert rc == kb.KDA_ERR_WORKSPACE
    msg = kb.kda_last_error()
    assert "static scratch" in msg and str(kb.NOALLOC_SCRATCH_BYTES) in msg
