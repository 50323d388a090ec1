"""GPU tests of the host-buffer entry point kda_fwd_host: on pinned host tensors it must give
bit for bit what kda_fwd gives on device tensors (same kernels, same schedule), whatever the
device arena held before, and set host rows of o outside every sequence to zero."""
import numpy as np
import pytest

from kimi_delta_attention_gate_gb300 import inputs as kin

from kda_testlib import assert_close, run_gpu, run_gpu_host, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_gate_gb300 import build
    build.build()


def wl_(**kw):
    kw.setdefault("K", 128)
    kw.setdefault("V", 128)
    gate = kw.pop("gate", kin.GATE_SAFE)
    return kin.Workload(kw.pop("name", "host"), chunk_size=64, gate=gate,
                        lower_bound=-5.0 if gate == kin.GATE_SAFE else None, h0_std=0.1,
                        has_dt_bias=True, has_a_log=True, a_log_mean=0.0, a_log_std=1.0, **kw)


def same_as_device(inp, **opts):
    o, fs = run_gpu_host(inp, **opts)[:2]
    ro, rfs = run_gpu(inp, **opts)
    covered = inp.wl.T if inp.cu_seqlens is None else int(inp.cu_seqlens[-1])
    assert np.array_equal(o, ro), "o differs from kda_fwd"
    assert np.array_equal(fs, rfs), "final_state differs from kda_fwd"
    assert np.all(o[:, covered:] == 0.0), "rows outside every sequence are not zero"
    return o, fs


def test_host_entry_pipelined_long_sequence():
    """257 chunks: two segments, the second segment's rows copied in during the first."""
    inp = kin.make_inputs(wl_(B=1, T=64 * 256 + 37, H=2, HV=2, dtype="bf16", seed=600))
    o, fs = same_as_device(inp)
    ro, rfs = run_oracle(inp, heads=[1])
    assert_close(o[:, :, [1]], ro, "bf16", "o")
    assert_close(fs[:, [1]], rfs, "bf16", "final_state")


def test_host_entry_pipelined_batch_six_segments():
    """B=3 sequences over six segments (boundaries inside sequences)."""
    same_as_device(kin.make_inputs(wl_(B=3, T=64 * 200 + 10, H=1, HV=1, dtype="bf16", seed=601)))


def test_host_entry_pipelined_varlen_with_tail_rows():
    """Varlen with empty sequences; 63 rows past the last sequence come back as zeros."""
    inp = kin.make_inputs(wl_(B=1, T=17100, H=2, HV=2, dtype="bf16", varlen_n=5,
                              varlen_max_len=9100, seed=602))
    inp.cu_seqlens[:] = np.array([0, 8000, 8000, 17000, 17037, 17037], dtype=np.int64)
    same_as_device(inp)


@pytest.mark.parametrize("dtype,K", [("bf16", 128), ("f32", 64)])
def test_host_entry_single_schedule_varlen(dtype, K):
    """Short input (one launch per stage, copies around them) on both kernel paths."""
    inp = kin.make_inputs(wl_(B=1, T=300, H=2, HV=4, K=K, V=K, dtype=dtype, varlen_n=6,
                              varlen_max_len=120, seed=603 + K))
    inp.cu_seqlens[:] = np.array([0, 1, 1, 65, 66, 130, 250], dtype=np.int64)
    same_as_device(inp)


def test_host_entry_transposed_states_and_neg_eigval():
    inp = kin.make_inputs(wl_(B=1, T=64 * 256 + 5, H=1, HV=1, dtype="bf16", seed=604))
    inp.h0 = np.ascontiguousarray(np.swapaxes(inp.h0, -1, -2))
    same_as_device(inp, transpose_state_layout=True, allow_neg_eigval=True)


def test_host_entry_intermediate_states():
    """Per-chunk states through the host entry equal kda_fwd's (pipelined schedule)."""
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    from kda_testlib import f32_device, gate_kwargs, to_device
    T = 64 * 256 + 37
    inp = kin.make_inputs(wl_(B=1, T=T, H=1, HV=1, dtype="bf16", seed=605))
    nct = (T + 63) // 64
    o, fs, hs = run_gpu_host(inp, h_out_chunks=nct)
    q, k, v, g, b = (to_device(x, "bf16") for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    do, dfs, dhs = kda.kda_fwd(q, k, v, g, b, A_log=f32_device(inp.A_log),
                               dt_bias=f32_device(inp.dt_bias), scale=inp.scale,
                               initial_state=f32_device(inp.h0), return_intermediate_states=True,
                               **gate_kwargs(inp.wl))
    torch.cuda.synchronize()
    assert np.array_equal(hs, dhs.cpu().double().numpy())
    assert np.array_equal(fs, dfs.cpu().double().numpy())
    assert np.array_equal(o, do.float().cpu().double().numpy())
