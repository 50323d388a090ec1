"""Pins for the oracle's reference gradients (oracle/backward.py), all on the CPU.

None compares the autograd restatement with itself: its forward is checked against the C
oracle, its gradients against central finite differences of the C oracle's forward (independent
code), against closed-form derivatives of one-token cases, and against linearity in the incoming
gradient."""
import numpy as np
import pytest

pytest.importorskip("torch")

import oracle
from oracle import GATE_PLAIN, GATE_PREGATED, GATE_SAFE
from oracle import backward as ob


def case(seed, B=2, T=5, H=1, HV=2, K=4, V=3, gate=GATE_SAFE):
    r = np.random.default_rng(seed)
    d = dict(q=r.standard_normal((B, T, H, K)), k=r.standard_normal((B, T, H, K)),
             v=r.standard_normal((B, T, HV, V)), g=r.standard_normal((B, T, HV, K)),
             beta=r.standard_normal((B, T, HV)), initial_state=0.3 * r.standard_normal((B, HV, K, V)),
             dt_bias=0.5 * r.standard_normal(HV * K))
    if gate == GATE_PREGATED:
        d["g"] = -np.abs(d["g"]) * 0.5
        d.pop("dt_bias")
        opts = dict(gate_mode=GATE_PREGATED)
    elif gate == GATE_PLAIN:
        d["A_log"] = r.uniform(-1.0, 0.5, HV)
        opts = dict(gate_mode=GATE_PLAIN)
    else:
        d["A_log"] = r.uniform(-0.5, 0.5, HV)
        opts = dict(gate_mode=GATE_SAFE, lower_bound=-5.0)
    do = r.standard_normal((B, T, HV, V))
    dfinal = r.standard_normal((B, HV, K, V))
    return d, opts, do, dfinal


def c_loss(d, opts, do, dfinal, **extra):
    o, fs = oracle.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], A_log=d.get("A_log"),
                       dt_bias=d.get("dt_bias"), initial_state=d.get("initial_state"),
                       **opts, **extra)
    return float(np.sum(o * do) + np.sum(fs * dfinal))


def grads(d, opts, do, dfinal, **extra):
    return ob.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], do, dfinal, A_log=d.get("A_log"),
                  dt_bias=d.get("dt_bias"), initial_state=d.get("initial_state"), **opts, **extra)


NAMES = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "A_log": "dA_log",
         "dt_bias": "ddt_bias", "initial_state": "dh0"}


def test_forward_matches_the_c_oracle():
    d, opts, do, dfinal = case(1)
    r = grads(d, opts, do, dfinal)
    o, fs = oracle.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], A_log=d["A_log"],
                       dt_bias=d["dt_bias"], initial_state=d["initial_state"], **opts)
    assert np.allclose(r["o"], o, rtol=0, atol=1e-12)
    assert np.allclose(r["final_state"], fs, rtol=0, atol=1e-12)


@pytest.mark.parametrize("gate", [GATE_SAFE, GATE_PLAIN, GATE_PREGATED])
@pytest.mark.parametrize("neg", [False, True])
def test_directional_derivatives_match_finite_differences_of_the_c_oracle(gate, neg):
    """<grad, delta> against (L(x + eps delta) - L(x - eps delta)) / (2 eps), L evaluated by
    the C oracle, for a random direction in every input."""
    extra = dict(allow_neg_eigval=True) if neg else {}
    d, opts, do, dfinal = case(10 + gate + 3 * neg, gate=gate)
    r = grads(d, opts, do, dfinal, **extra)
    rng = np.random.default_rng(99)
    eps = 1e-6
    for name, key in NAMES.items():
        if name not in d:
            assert r[key] is None
            continue
        delta = rng.standard_normal(np.shape(d[name]))
        plus = dict(d); plus[name] = d[name] + eps * delta
        minus = dict(d); minus[name] = d[name] - eps * delta
        fd = (c_loss(plus, opts, do, dfinal, **extra) - c_loss(minus, opts, do, dfinal, **extra)) / (2 * eps)
        an = float(np.sum(r[key] * delta))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_one_token_closed_forms():
    """One token, K = V = 1, no norms, beta taken as given, pre-gated decay g:
    o = s q (a S0 + b k (v - k a S0)), a = e^g."""
    q, k, v, g, b, S0, s = 0.7, -1.3, 0.4, -0.35, 0.6, 0.9, 0.8
    a = np.exp(g)
    r = ob.bwd(np.full((1, 1, 1, 1), q), np.full((1, 1, 1, 1), k), np.full((1, 1, 1, 1), v),
               np.full((1, 1, 1, 1), g), np.full((1, 1, 1), b), np.ones((1, 1, 1, 1)), None,
               gate_mode=GATE_PREGATED, scale=s, qk_l2norm=False, beta_sigmoid=False,
               initial_state=np.full((1, 1, 1, 1), S0))
    expect = {"dv": s * q * b * k,
              "dq": s * (a * S0 + b * k * (v - k * a * S0)),
              "dbeta": s * q * k * (v - k * a * S0),
              "dk": s * q * b * (v - 2 * k * a * S0),
              "dg": s * q * a * S0 * (1 - b * k * k),
              "dh0": s * q * a * (1 - b * k * k)}
    for key, val in expect.items():
        assert np.isclose(float(r[key].ravel()[0]), val, rtol=1e-13, atol=1e-15), key


def test_gradients_are_linear_in_the_incoming_gradient():
    d, opts, do1, df1 = case(21)
    _, _, do2, df2 = case(22)
    r1, r2 = grads(d, opts, do1, df1), grads(d, opts, do2, df2)
    r12 = grads(d, opts, do1 + 2.0 * do2, df1 + 2.0 * df2)
    for key in NAMES.values():
        assert np.allclose(r12[key], r1[key] + 2.0 * r2[key], rtol=1e-12, atol=1e-12), key


def test_final_state_gradient_alone_leaves_q_untouched():
    """The final state does not depend on q: with do = 0 the gradient of q is exactly zero."""
    d, opts, do, dfinal = case(31)
    r = grads(d, opts, np.zeros_like(do), dfinal)
    assert np.all(r["dq"] == 0)
    assert np.any(r["dk"] != 0)


@pytest.mark.parametrize("gate", [GATE_SAFE, GATE_PLAIN, GATE_PREGATED])
@pytest.mark.parametrize("C,T", [(4, 13), (5, 5), (16, 11)])
def test_chunked_backward_matches_autograd(gate, C, T):
    """The hand-derived chunked backward (chunks of C tokens, a ragged last chunk) against the
    autograd reference, which is itself pinned to finite differences of the C oracle."""
    d, opts, do, dfinal = case(40 + gate + C, T=T, gate=gate)
    ref = grads(d, opts, do, dfinal)
    got = ob.chunk_bwd_np(d["q"], d["k"], d["v"], d["g"], d["beta"], do, dfinal, chunk_size=C,
                          A_log=d.get("A_log"), dt_bias=d.get("dt_bias"),
                          initial_state=d.get("initial_state"), **opts)
    for key in ["o", "final_state"] + list(NAMES.values()):
        if ref[key] is None:
            assert got[key] is None, key
            continue
        assert np.allclose(got[key], ref[key], rtol=1e-9, atol=1e-10), key


def test_chunked_backward_options():
    """No norms, beta taken as given; and beta = 2 sigmoid(logit)."""
    d, opts, do, dfinal = case(51, T=9)
    for extra in (dict(qk_l2norm=False, beta_sigmoid=False), dict(allow_neg_eigval=True)):
        ref = grads(d, opts, do, dfinal, **extra)
        got = ob.chunk_bwd_np(d["q"], d["k"], d["v"], d["g"], d["beta"], do, dfinal, chunk_size=4,
                              A_log=d["A_log"], dt_bias=d["dt_bias"],
                              initial_state=d["initial_state"], **opts, **extra)
        for key in NAMES.values():
            assert np.allclose(got[key], ref[key], rtol=1e-9, atol=1e-10), (extra, key)


def test_varlen_gradients_pin_to_the_c_oracle_and_match_the_chunked_form():
    """A varlen batch (an empty sequence included): finite differences of the C oracle's varlen
    forward pin the autograd form, and the chunked form agrees with it."""
    r = np.random.default_rng(61)
    tot, H, HV, K, V = 14, 1, 2, 4, 3
    cu = np.array([0, 5, 5, 11, 14], np.int64)
    N = len(cu) - 1
    d = dict(q=r.standard_normal((1, tot, H, K)), k=r.standard_normal((1, tot, H, K)),
             v=r.standard_normal((1, tot, HV, V)), g=r.standard_normal((1, tot, HV, K)),
             beta=r.standard_normal((1, tot, HV)), initial_state=0.3 * r.standard_normal((N, HV, K, V)),
             dt_bias=0.5 * r.standard_normal(HV * K), A_log=r.uniform(-0.5, 0.5, HV))
    opts = dict(gate_mode=GATE_SAFE, lower_bound=-5.0)
    do, dfinal = r.standard_normal((1, tot, HV, V)), r.standard_normal((N, HV, K, V))
    ref = grads(d, opts, do, dfinal, cu_seqlens=cu)
    got = ob.chunk_bwd_np(d["q"], d["k"], d["v"], d["g"], d["beta"], do, dfinal, chunk_size=4,
                          A_log=d["A_log"], dt_bias=d["dt_bias"], initial_state=d["initial_state"],
                          cu_seqlens=cu, **opts)
    for key in NAMES.values():
        assert np.allclose(got[key], ref[key], rtol=1e-9, atol=1e-10), key
    rng = np.random.default_rng(62)
    eps = 1e-6
    for name, key in NAMES.items():
        delta = rng.standard_normal(np.shape(d[name]))
        plus = dict(d); plus[name] = d[name] + eps * delta
        minus = dict(d); minus[name] = d[name] - eps * delta
        fd = (c_loss(plus, opts, do, dfinal, cu_seqlens=cu)
              - c_loss(minus, opts, do, dfinal, cu_seqlens=cu)) / (2 * eps)
        an = float(np.sum(ref[key] * delta))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_transposed_state_layout_is_the_transpose():
    d, opts, do, dfinal = case(71, T=6)
    ref = grads(d, opts, do, dfinal)
    sw = lambda x: np.ascontiguousarray(np.swapaxes(x, -1, -2))
    dt = dict(d); dt["initial_state"] = sw(d["initial_state"])
    for fn in (lambda **kw: grads(dt, opts, do, sw(dfinal), **kw),
               lambda **kw: ob.chunk_bwd_np(dt["q"], dt["k"], dt["v"], dt["g"], dt["beta"], do,
                                            sw(dfinal), chunk_size=4, A_log=dt["A_log"],
                                            dt_bias=dt["dt_bias"], initial_state=dt["initial_state"],
                                            **opts, **kw)):
        got = fn(transpose_state_layout=True)
        assert np.allclose(got["dh0"], sw(ref["dh0"]), rtol=1e-9, atol=1e-10)
        assert np.allclose(got["final_state"], sw(ref["final_state"]), rtol=1e-9, atol=1e-10)
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            assert np.allclose(got[key], ref[key], rtol=1e-9, atol=1e-10), key
