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


@pytest.fixture(scope="module", autouse=True)
def _built():
    """Build and load the library, so that the file also runs alone in a fresh process."""
    from kimi_delta_attention_gate_gb300 import _binding as kb
    from kimi_delta_attention_gate_gb300 import build
    build.build()
    kb.load()


def _inputs(seed, B=2, T=150, HV=4, varlen=None):
    wl = kin.Workload("noalloc", B=B, T=T, H=min(2, HV), HV=HV, K=128, V=128, chunk_size=64,
                      dtype="bf16", gate=kin.GATE_SAFE, lower_bound=-5.0, h0_std=0.1, seed=seed,
                      **({} if varlen is None else dict(varlen_n=varlen[0], varlen_max_len=varlen[1])))
    return kin.make_inputs(wl)


def _tensors(inp):
    wl = inp.wl
    q, k, v, g, b = (to_device(x, wl.dtype) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    return q, k, v, g, b, f32_device(inp.A_log), f32_device(inp.dt_bias), f32_device(inp.h0)


def _compare(inp, stream):
    """One kda_fwd_noalloc call against kda_fwd on the same inputs: the same kernels on the
    same bits, so the results must agree bit for bit (and both within the bf16 tolerance of
    each other, which bit-identity implies).  o starts as NaN so that every row, padding
    included, must be written."""
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    from kimi_delta_attention_gate_gb300 import _binding as kb
    q, k, v, g, b, A_log, dt_bias, h0 = _tensors(inp)
    cu = cu_cpu = None
    if inp.cu_seqlens is not None:
        cu_cpu = torch.from_numpy(inp.cu_seqlens)
        cu = cu_cpu.cuda()
    common = dict(A_log=A_log, dt_bias=dt_bias, lower_bound=-5.0, scale=inp.scale,
                  initial_state=h0, cu_seqlens=cu, cu_seqlens_cpu=cu_cpu)
    o_ref, fs_ref = kda.kda_fwd(q, k, v, g, b, **common)
    o = torch.full_like(o_ref, float("nan"))
    fs = torch.full_like(fs_ref, float("nan"))
    p = kda.make_params(q, k, v, g, b, o=o, final_state=fs, **common)
    need = kb.kda_fwd_workspace_size(p)
    assert 0 < need <= kb.NOALLOC_SCRATCH_BYTES
    rc = kb.kda_fwd_noalloc(p, stream.cuda_stream)
    assert rc == kb.KDA_OK, kb.kda_last_error()
    torch.cuda.synchronize()
    assert kb.kda_get_device_status(stream.cuda_stream) == 0
    tol = TOL["bf16"]
    for got, ref, what in ((o, o_ref, "o"), (fs, fs_ref, "final_state")):
        gn = got.float().cpu().double().numpy()
        rn = ref.float().cpu().double().numpy()
        assert np.all(np.isfinite(gn)), what
        rel, mx = errors(gn, rn)
        assert rel <= tol["rel_l2"] and mx <= tol["max_abs"], (what, rel, mx)
        assert np.array_equal(gn, rn), f"{what}: kda_fwd_noalloc differs from kda_fwd"
    return need


def test_noalloc_matches_kda_fwd_on_two_calls_in_a_row():
    """Two calls in a row on different inputs, each bit-identical to kda_fwd."""
    import torch
    stream = torch.cuda.current_stream()
    for seed in (11, 12):
        _compare(_inputs(seed), stream)


def test_noalloc_smaller_call_after_a_larger_one():
    """A large call (long sequence, close to the scratch size) leaves its intermediates in the
    shared array; the smaller calls after it (one varlen, one batched) must not pick any of
    them up: each is still bit-identical to kda_fwd."""
    import torch
    stream = torch.cuda.current_stream()
    big = _compare(_inputs(21, B=1, T=64 * 300 + 17, HV=1), stream)   # 301 chunks, ~20 MB
    small = _compare(_inputs(22, B=1, T=700, HV=4, varlen=(5, 300)), stream)
    assert small < big
    _compare(_inputs(23, B=3, T=100, HV=2), stream)


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
