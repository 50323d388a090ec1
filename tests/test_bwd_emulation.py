"""The backward kernels' stage bodies (csrc/kda_bwd.cuh), compiled for the host with
AddressSanitizer and UndefinedBehaviorSanitizer and run with the GPU's block size, every
phase's threads in a shuffled order, against the oracle's fp64 gradients (oracle/backward.py,
pinned to finite differences of the C oracle's forward).  No GPU: these check the index
arithmetic, the barriers, the work split and the arithmetic of the GPU code before it runs on
one; the GPU parity tests run the same bodies as kernels."""
import numpy as np
import pytest

pytest.importorskip("torch")

from kimi_delta_attention_gate_gb300 import inputs as kin

import bwd_testlib as bt


@pytest.fixture(scope="module")
def emu(tmp_path_factory):
    return bt.build_emulator(str(tmp_path_factory.mktemp("bwd_emu")))


wl_ = bt.workload
pregate = bt.pregate


def check(emu, tmp_path, inp, *, seed=0, chunk_form=False, up_seed=11, **opts):
    d_o, dfs = bt.upstream(inp, up_seed, state_v_first=opts.get("state_v_first", False))
    got = bt.run_emulator(emu, str(tmp_path / f"run{seed}"), inp, d_o, dfs, seed=seed, **opts)
    assert got["status"] == 0
    ref = bt.oracle_grads(inp, d_o, dfs, chunk_form=chunk_form, **opts)
    return bt.assert_grads_close(got, ref), got


@pytest.mark.parametrize("gate", [kin.GATE_SAFE, kin.GATE_PLAIN, kin.GATE_PREGATED])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gate_modes_and_dtypes(emu, tmp_path, gate, dtype):
    inp = kin.make_inputs(wl_(gate=gate, dtype=dtype, seed=20 + gate))
    if gate == kin.GATE_PREGATED:
        pregate(inp)
    check(emu, tmp_path, inp)


@pytest.mark.parametrize("C,T", [(32, 97), (64, 64), (64, 1), (32, 31)])
def test_chunk_sizes_and_ragged_tails(emu, tmp_path, C, T):
    check(emu, tmp_path, kin.make_inputs(wl_(C=C, T=T, seed=30 + T)))


def test_equal_heads_and_wider_groups(emu, tmp_path):
    check(emu, tmp_path, kin.make_inputs(wl_(H=2, HV=2, seed=40)))
    check(emu, tmp_path, kin.make_inputs(wl_(B=1, H=2, HV=6, T=90, seed=41)))


def test_partial_and_several_value_tiles(emu, tmp_path):
    """V = 40: one full and one partial 32-column tile; K != V."""
    check(emu, tmp_path, kin.make_inputs(wl_(K=24, V=40, seed=42)))


def test_full_head_dimensions(emu, tmp_path):
    """K = V = 128, the dimensions of the long-context workload, over two chunks."""
    inp = kin.make_inputs(wl_(B=1, T=100, H=1, HV=1, K=128, V=128, dtype="bf16", seed=43,
                              h0_std=0.1))
    check(emu, tmp_path, inp, chunk_form=True)


def test_largest_head_dimensions(emu, tmp_path):
    """K = 256 (the largest the checks allow) and V = 200 (six full V tiles and a partial one),
    chunk 32, over three chunks."""
    inp = kin.make_inputs(wl_(B=1, T=70, H=1, HV=1, K=256, V=200, C=32, seed=53, h0_std=0.05))
    check(emu, tmp_path, inp, chunk_form=True)


def test_varlen_with_empty_sequences_and_padding(emu, tmp_path):
    inp = kin.make_inputs(wl_(B=1, T=200, seed=44, varlen_n=5, varlen_max_len=60))
    inp.cu_seqlens[:] = np.array([0, 70, 70, 71, 135, 190], dtype=np.int64)  # 10 padding rows
    errs, got = check(emu, tmp_path, inp)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.all(got[name][:, 190:] == 0), name


def test_transposed_state_layout_and_negative_eigenvalues(emu, tmp_path):
    inp = kin.make_inputs(wl_(seed=45))
    inp.h0 = np.ascontiguousarray(np.swapaxes(inp.h0, -1, -2))
    check(emu, tmp_path, inp, state_v_first=True, allow_neg_eigval=True)


def test_without_optional_inputs(emu, tmp_path):
    """No initial state (dh0 is the gradient at zero), no dt_bias, a safe gate without
    A_log."""
    inp = kin.make_inputs(wl_(seed=46, h0_std=None, has_dt_bias=False, has_a_log=False))
    check(emu, tmp_path, inp)


def test_safe_gate_at_its_bound(emu, tmp_path):
    """g' near lower_bound = -5 on every element: Gamma reaches about -320 within a chunk,
    e^Gamma underflows in fp32 and the e^(Gamma_i - Gamma_j) terms span the whole range.
    (x = g + dt_bias around 8, where the fp64 oracle's sigmoid derivative s (1 - s) is still
    exact to about 1e-12.)"""
    inp = kin.make_inputs(wl_(seed=47, T=128))
    inp.g[:] = np.float32(8.0)
    inp.A_log[:] = np.float32(0.0)
    check(emu, tmp_path, inp)


def test_no_tokens(emu, tmp_path):
    """T = 0: the state gradient passes straight through (dh0 = d_final_state)."""
    inp = kin.make_inputs(wl_(T=0, seed=48))
    d_o, dfs = bt.upstream(inp, 3)
    got = bt.run_emulator(emu, str(tmp_path / "t0"), inp, d_o, dfs)
    assert got["status"] == 0
    assert np.array_equal(got["dh0"], dfs.astype(np.float64))
    assert np.all(got["dA_log"] == 0) and np.all(got["ddt_bias"] == 0)


def test_thread_order_does_not_change_the_result(emu, tmp_path):
    """With HV == H nothing is summed by atomics except dA_log and ddt_bias: two runs with
    different thread orders inside every phase give the same bits (a phase that read what
    another thread writes in the same phase would not)."""
    inp = kin.make_inputs(wl_(H=2, HV=2, T=130, seed=49))
    d_o, dfs = bt.upstream(inp, 5)
    a = bt.run_emulator(emu, str(tmp_path / "a"), inp, d_o, dfs, seed=1)
    b = bt.run_emulator(emu, str(tmp_path / "b"), inp, d_o, dfs, seed=2)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert np.array_equal(a[name], b[name]), name
    for name in ("dA_log", "ddt_bias"):
        assert bt.rel_l2(a[name], b[name]) < 1e-6, name


def test_a_planted_error_in_the_oracle_is_caught(emu, tmp_path, monkeypatch):
    """The comparison has teeth: the oracle with the gate's dt_bias gradient halved (a
    plausible slip) no longer matches the kernels, nor with dv off by one part in 1e3."""
    from oracle import backward as ob
    real = ob.bwd

    def planted(*args, **kw):
        r = real(*args, **kw)
        r["ddt_bias"] = r["ddt_bias"] * 0.5
        return r

    monkeypatch.setattr(ob, "bwd", planted)
    with pytest.raises(AssertionError, match="ddt_bias"):
        check(emu, tmp_path, kin.make_inputs(wl_(seed=50)))

    def planted_dv(*args, **kw):
        r = real(*args, **kw)
        r["dv"] = r["dv"] * (1 + 1e-3)
        return r

    monkeypatch.setattr(ob, "bwd", planted_dv)
    with pytest.raises(AssertionError, match="dv"):
        check(emu, tmp_path, kin.make_inputs(wl_(seed=51)))


def test_no_decay(emu, tmp_path):
    """Pre-gated log decay 0 (alpha = 1): Gamma = 0, every exponential is 1."""
    inp = kin.make_inputs(wl_(gate=kin.GATE_PREGATED, seed=54))
    inp.g[:] = 0.0
    check(emu, tmp_path, inp)


def test_beta_near_zero(emu, tmp_path):
    """beta logits of -30: beta ~ 1e-13, the state is barely written."""
    inp = kin.make_inputs(wl_(seed=55))
    inp.beta[:] = np.float32(-30.0)
    check(emu, tmp_path, inp)


def test_zero_query_and_key_rows(emu, tmp_path):
    """All-zero q and k rows: the L2 norm sits at its epsilon (|x| = 0 < sqrt(1e-6))."""
    inp = kin.make_inputs(wl_(seed=56))
    inp.q[:, 5] = 0.0
    inp.k[:, 70] = 0.0
    check(emu, tmp_path, inp)


def test_zero_incoming_gradients_give_zero(emu, tmp_path):
    inp = kin.make_inputs(wl_(seed=57))
    d_o, dfs = bt.upstream(inp, 1)
    d_o[:] = 0.0
    dfs[:] = 0.0
    got = bt.run_emulator(emu, str(tmp_path / "z"), inp, d_o, dfs)
    for name in bt.GRADS:
        assert np.all(got[name] == 0), name


def test_single_token_sequences(emu, tmp_path):
    """B = 3 sequences of one token (one one-row chunk each)."""
    check(emu, tmp_path, kin.make_inputs(wl_(B=3, T=1, seed=58)))


@pytest.mark.parametrize("seed", range(100, 116))
def test_random_shapes(emu, tmp_path, seed):
    """Seeded random configurations: batch, length (ragged tails), grouped heads, K, V
    (partial value tiles), chunk size, gate mode, dtype, varlen, optional inputs, options."""
    inp, opts = bt.random_case(seed)
    check(emu, tmp_path, inp, chunk_form=True, **opts)


@pytest.mark.parametrize("C", [32, 64])
def test_steep_decay_takes_the_exact_exponent_path(emu, tmp_path, C):
    """A pre-gated log decay of -9 to -15 per element: within a 16-row block Gamma drops by
    more than 60 nat on one side of the middle row, so the gradient kernel evaluates every
    e^(Gamma_i - Gamma_j) directly instead of through block references; a milder chunk in the
    same batch (the first sequence) keeps the blocked path.  Both against the oracle."""
    inp = kin.make_inputs(wl_(B=2, T=100, C=C, gate=kin.GATE_PREGATED, seed=60 + C))
    r = np.random.default_rng(61 + C)
    inp.g[1] = -r.uniform(9.0, 15.0, size=inp.g[1].shape).astype(np.float32)
    inp.g[0] = -np.abs(inp.g[0]) * np.float32(0.5)
    check(emu, tmp_path, inp)
