"""GPU parity of the token-recurrent entry point (kda_fused_recurrent_fwd, decode and short
prefill) against the fp64 oracle, which is the same token recurrence.  Tolerances as for
kda_fwd: bf16 inputs rel-L2 <= 5e-3 and max-abs <= 3e-2, fp32 inputs rel-L2 <= 1e-4."""
import numpy as np
import pytest

from kimi_delta_attention_gate_gb300 import inputs as kin

from kda_testlib import assert_close, f32_device, gate_kwargs, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_gate_gb300 import build
    build.build()


def wl_of(*, B=2, T=7, H=2, HV=2, K=64, V=64, dtype="bf16", gate=kin.GATE_SAFE, h0=0.1,
          varlen=0, maxlen=0, seed=1):
    return kin.Workload("rec", B=B, T=T, H=H, HV=HV, K=K, V=V, chunk_size=64, dtype=dtype,
                        gate=gate, lower_bound=-5.0 if gate == kin.GATE_SAFE else None,
                        h0_std=h0, varlen_n=varlen, varlen_max_len=maxlen, seed=seed,
                        a_log_mean=-1.0 if gate == kin.GATE_PLAIN else 0.0,
                        a_log_std=0.5 if gate == kin.GATE_PLAIN else 1.0)


def run_rec(inp, **opts):
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    wl = inp.wl
    q, k, v, g, b = (to_device(x, wl.dtype) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    cu = None if inp.cu_seqlens is None else torch.from_numpy(inp.cu_seqlens).cuda()
    o, fs = kda.kda_fused_recurrent_fwd(q, k, v, g, b, A_log=f32_device(inp.A_log),
                                        dt_bias=f32_device(inp.dt_bias), scale=inp.scale,
                                        initial_state=f32_device(inp.h0), cu_seqlens=cu,
                                        **gate_kwargs(wl), **opts)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status(0) == 0
    return o.float().cpu().double().numpy(), fs.cpu().double().numpy()


def check(inp, **opts):
    o, fs = run_rec(inp, **opts)
    ro, rfs = run_oracle(inp, **opts)
    assert_close(o, ro, inp.wl.dtype, "o")
    assert_close(fs, rfs, inp.wl.dtype, "final_state")


def test_decode_one_token_many_sequences():
    """Decode: 64 sequences of one token each, K = V = 128, a nonzero incoming state."""
    check(kin.make_inputs(wl_of(B=64, T=1, H=4, HV=4, K=128, V=128, seed=601)))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("gate", [kin.GATE_SAFE, kin.GATE_PLAIN, kin.GATE_PREGATED])
def test_short_prefill_gate_modes(dtype, gate):
    inp = kin.make_inputs(wl_of(T=37, dtype=dtype, gate=gate, seed=610 + gate))
    if gate == kin.GATE_PREGATED:
        inp.g[:] = kin.round_to_bf16(-np.abs(inp.g) * 0.5) if dtype == "bf16" else -np.abs(inp.g) * 0.5
    check(inp)


@pytest.mark.parametrize("K,V", [(48, 40), (256, 256), (128, 32)])
def test_head_dims_and_gva(K, V):
    check(kin.make_inputs(wl_of(T=9, H=2, HV=6, K=K, V=V, seed=620 + K + V)))


def test_varlen_with_empty_sequence_neg_eigval_and_transposed_state():
    wl = wl_of(B=1, T=40, varlen=4, maxlen=20, seed=630)
    inp = kin.make_inputs(wl)
    inp.cu_seqlens[:] = np.array([0, 7, 7, 22, 31], dtype=np.int64)
    inp.h0 = np.ascontiguousarray(np.swapaxes(inp.h0, -1, -2))
    check(inp, allow_neg_eigval=True, transpose_state_layout=True)


def test_agrees_with_the_chunk_path():
    """The two entry points compute the same thing (both within tolerance of the oracle and
    of each other) on a multi-chunk bf16 case with K = V = 128."""
    from kda_testlib import run_gpu
    inp = kin.make_inputs(wl_of(B=1, T=200, K=128, V=128, seed=640))
    o1, f1 = run_rec(inp)
    o2, f2 = run_gpu(inp)
    assert_close(o1, o2, "bf16", "o (recurrent vs chunk)")
    assert_close(f1, f2, "bf16", "final_state (recurrent vs chunk)")


def test_rejects_per_chunk_states():
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    from kimi_delta_attention_gate_gb300 import _binding as kb
    q = torch.zeros((1, 4, 1, 64), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((1, 4, 1, 64), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((1, 4, 1), dtype=torch.bfloat16, device="cuda")
    h = torch.zeros((1, 1, 64, 64), dtype=torch.float32, device="cuda")
    p = kda.make_params(q, q, v, v, b, lower_bound=-5.0, o=v, h_out=h)
    assert kb.kda_fused_recurrent_fwd(p, 0) == kb.KDA_ERR_INVALID_ARG
