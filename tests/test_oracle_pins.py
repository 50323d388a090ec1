"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

None of these compare the oracle with itself.  Each pin is either a number the
pages print (tests/golden/page_constants.json), a closed form, a special case
that reduces to something checkable by hand, a structural identity of the
method (chunk form == token recurrence, resume, varlen, GVA), or brute force
with explicit transition matrices.  All run on the CPU.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import GATE_PLAIN, GATE_PREGATED, GATE_SAFE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def make_case(seed, B=1, T=20, H=1, HV=1, K=8, V=6, gate=GATE_SAFE, h0=True, dt=True, alog=True):
    r = np.random.default_rng(seed)
    d = dict(
        q=r.standard_normal((B, T, H, K)), k=r.standard_normal((B, T, H, K)),
        v=r.standard_normal((B, T, HV, V)), g=r.standard_normal((B, T, HV, K)),
        beta=r.standard_normal((B, T, HV)),
    )
    kw = dict(gate_mode=gate,
              A_log=(r.standard_normal(HV) if alog else None),
              dt_bias=(r.standard_normal(HV * K) if dt else None),
              lower_bound=(-5.0 if gate == GATE_SAFE else None),
              initial_state=(0.3 * r.standard_normal((B, HV, K, V)) if h0 else None))
    if gate == GATE_PREGATED:
        d["g"] = -np.abs(d["g"])        # a log decay: non-positive
    return d, kw


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# --------------------------------------------------------------------------------------
# Gate: printed constants and closed forms
# --------------------------------------------------------------------------------------

def test_golden_page_constants_and_gate_saturation():
    c = json.load(open(GOLDEN))
    lb = c["recommended_lower_bound"]["value"]
    # Saturated safe gate (sigmoid -> 1) gives the lower bound; the printed per-step
    # decay exp(-5) ~ 0.0067 follows.
    big = np.full((1, 1, 1), 60.0)
    gsat = oracle.gate_np(big, GATE_SAFE, A_log=np.zeros(1), lower_bound=lb)[0, 0, 0]
    assert abs(gsat - lb) < 1e-20
    printed = c["per_step_decay_at_recommended_lower_bound"]
    assert round(math.exp(gsat), 4) == pytest.approx(printed["value"], abs=0.5e-4)
    # Worst sub-chunk decay: BC tokens at the bound.
    bc = c["subchunk_size"]["value"]
    gc = oracle.gate_c(np.full((bc, 1, 1), 60.0), GATE_SAFE, np.zeros(1), None, lb)
    assert float(np.sum(gc)) == pytest.approx(c["worst_subchunk_log_decay"]["value"], abs=1e-9)
    # Midpoint leaves half a sub-chunk: 8 tokens x 5 = 40 nat = 40/ln2 in log2 units < 85.
    half = (bc // 2) * (-lb) / math.log(2.0)
    assert half == pytest.approx(40.0 / math.log(2.0))
    assert half < c["midpoint_half_span_log2"]["ceiling"]
    # gate_scale = lb * 1.4427 is lb * log2(e) to the printed digits.
    assert round(math.log2(math.e), 4) == c["gate_scale_log2e"]["value"]


@pytest.mark.parametrize("impl", ["np", "c"])
def test_gate_special_values(impl):
    gate = (lambda g, m, a, d, lb: oracle.gate_np(g, m, a, d, lb)) if impl == "np" else \
        (lambda g, m, a, d, lb: oracle.gate_c(g, m, a, d, lb))
    HV, K = 3, 4
    A_log = np.array([0.0, 0.7, -1.3])
    dt = rnd(1, HV * K)
    # x = g + dt_bias = 0 everywhere
    g0 = -dt.reshape(1, HV, K)
    s = gate(g0, GATE_SAFE, A_log, dt, -5.0)
    assert np.all(s == -2.5)                               # lb * sigmoid(0) = lb / 2 exactly
    p = gate(g0, GATE_PLAIN, A_log, dt, None)
    assert np.allclose(p, -np.exp(A_log)[None, :, None] * math.log(2.0), rtol=1e-15, atol=0)
    # softplus(ln(e - 1)) = 1  ->  plain gate = -exp(A_log)
    x1 = np.full((1, HV, K), math.log(math.e - 1.0))
    p1 = gate(x1, GATE_PLAIN, A_log, None, None)
    assert np.allclose(p1, -np.exp(A_log)[None, :, None], rtol=1e-14, atol=0)
    # A_log absent in safe mode: lb * sigmoid(g + dt); sigmoid(ln 3) = 3/4
    x3 = np.full((1, HV, K), math.log(3.0))
    s3 = gate(x3, GATE_SAFE, None, None, -4.0)
    assert np.allclose(s3, -3.0, rtol=1e-15, atol=0)
    # exp(A_log) multiplies the argument: A_log = ln 2 doubles it
    s4 = gate(np.full((1, 1, 1), math.log(3.0) / 2), GATE_SAFE, np.array([math.log(2.0)]), None, -4.0)
    assert s4[0, 0, 0] == pytest.approx(-3.0, rel=1e-14)
    # pre-gated passes g through
    gp = rnd(2, 2, HV, K)
    assert np.array_equal(gate(gp, GATE_PREGATED, None, None, None), gp)


def test_gate_safe_range():
    g = 4.0 * rnd(3, 4000, 2, 8)
    A_log = rnd(4, 2)
    dt = rnd(5, 16)
    for lb in (-5.0, -1.0, -0.01):
        out = oracle.gate_np(g, GATE_SAFE, A_log, dt, lb)
        assert np.all(out >= lb) and np.all(out < 0.0)
    outc = oracle.gate_c(g, GATE_SAFE, A_log, dt, -5.0)
    assert np.all(outc >= -5.0) and np.all(outc < 0.0)
    assert np.all(oracle.gate_np(g, GATE_PLAIN, A_log, dt) < 0.0)


def test_gate_c_matches_np_all_modes():
    g = 3.0 * rnd(6, 50, 3, 5)
    A_log, dt = rnd(7, 3), rnd(8, 15)
    for mode, lb in ((GATE_SAFE, -5.0), (GATE_PLAIN, None), (GATE_PREGATED, None)):
        for a in (A_log, None) if mode == GATE_SAFE else (A_log,):
            for d in (dt, None):
                x = oracle.gate_np(g, mode, a, d, lb)
                y = oracle.gate_c(g, mode, a, d, lb)
                assert np.allclose(x, y, rtol=1e-14, atol=1e-300)


# --------------------------------------------------------------------------------------
# Recurrence: brute force, closed forms, special cases
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("gate", [GATE_SAFE, GATE_PLAIN, GATE_PREGATED])
@pytest.mark.parametrize("seed", [0, 1])
def test_brute_force_transition_products(gate, seed):
    d, kw = make_case(seed, B=2, T=7, H=1, HV=2, K=4, V=3, gate=gate)
    o, fs = oracle.fwd(**d, **kw)
    ob, fb = oracle.transition_np(**d, **kw)
    assert np.max(np.abs(o - ob)) < 1e-12
    assert np.max(np.abs(fs - fb)) < 1e-12


def test_scalar_geometric_closed_form():
    """K = V = 1, k = q = 1, constant alpha and beta, v = 1:
    S_t = c S_{t-1} + beta with c = alpha (1 - beta), so
    S_t = c^t S_0 + beta (1 - c^t) / (1 - c), and o_t = scale * S_t."""
    T, alpha, beta, S0, scale = 37, 0.83, 0.41, 0.7, 1.9
    ones = np.ones((1, T, 1, 1))
    g = np.full((1, T, 1, 1), math.log(alpha))
    b = np.full((1, T, 1), beta)
    o, fs = oracle.fwd(ones, ones, ones, g, b, gate_mode=GATE_PREGATED, scale=scale,
                       qk_l2norm=False, beta_sigmoid=False,
                       initial_state=np.full((1, 1, 1, 1), S0))
    c = alpha * (1 - beta)
    t = np.arange(1, T + 1)
    expect = c ** t * S0 + beta * (1 - c ** t) / (1 - c)
    assert np.allclose(o[0, :, 0, 0], scale * expect, rtol=1e-13, atol=0)
    assert fs[0, 0, 0, 0] == pytest.approx(expect[-1], rel=1e-13)


def test_scalar_signed_keys():
    """K = V = 1 with k = +-1: S_t = alpha_t (1 - beta_t) S_{t-1} + beta_t k_t v_t."""
    r = np.random.default_rng(11)
    T = 25
    kk = np.where(r.random((1, T, 1, 1)) < 0.5, -1.0, 1.0)
    v = r.standard_normal((1, T, 1, 1))
    q = r.standard_normal((1, T, 1, 1))
    g = -r.random((1, T, 1, 1))
    b = r.random((1, T, 1))
    o, fs = oracle.fwd(q, kk, v, g, b, gate_mode=GATE_PREGATED, scale=1.0, qk_l2norm=False,
                       beta_sigmoid=False)
    S = 0.0
    for t in range(T):
        S = math.exp(g[0, t, 0, 0]) * (1 - b[0, t, 0]) * S + b[0, t, 0] * kk[0, t, 0, 0] * v[0, t, 0, 0]
        assert o[0, t, 0, 0] == pytest.approx(S * q[0, t, 0, 0], rel=1e-13, abs=1e-15)


def test_identity_alpha1_beta0():
    """alpha = 1 (pre-gated g = 0), beta = 0: the state never changes, o_t = scale h0^T q_t."""
    d, kw = make_case(21, B=2, T=30, H=2, HV=2, K=8, V=5, gate=GATE_PREGATED)
    d["g"][:] = 0.0
    d["beta"][:] = 0.0
    kw["gate_mode"] = GATE_PREGATED
    o, fs = oracle.fwd(**d, **kw, beta_sigmoid=False, qk_l2norm=False, scale=0.5)
    h0 = kw["initial_state"]
    assert np.array_equal(fs, h0)
    expect = 0.5 * np.einsum("btgk,bgkv->btgv", d["q"], h0)
    assert np.allclose(o, expect, rtol=1e-14, atol=1e-15)


def test_exact_overwrite_orthonormal_keys():
    """alpha = 1, beta = 1, one-hot keys: writing v at key e_j replaces row j of S
    exactly, so querying e_j returns scale * v (delta rule overwrite)."""
    K, V, T = 4, 3, 8
    r = np.random.default_rng(5)
    keys = np.array([0, 1, 2, 3, 2, 0, 3, 1])
    k = np.zeros((1, T, 1, K)); k[0, np.arange(T), 0, keys] = 1.0
    v = r.standard_normal((1, T, 1, V))
    h0 = r.standard_normal((1, 1, K, V))
    o, fs = oracle.fwd(k, k, v, np.zeros((1, T, 1, K)), np.ones((1, T, 1)),
                       gate_mode=GATE_PREGATED, scale=2.0, qk_l2norm=False, beta_sigmoid=False,
                       initial_state=h0)
    assert np.allclose(o[0, :, 0], 2.0 * v[0, :, 0], rtol=0, atol=1e-15)
    last = {int(j): t for t, j in enumerate(keys)}
    for j in range(K):
        assert np.allclose(fs[0, 0, j], v[0, last[j], 0], rtol=0, atol=1e-15)


def test_superposition_in_v_and_h0():
    d, kw = make_case(31, B=1, T=40, H=1, HV=1, K=6, V=4)
    o1, f1 = oracle.fwd(**d, **kw)
    d2 = dict(d); d2["v"] = rnd(32, *d["v"].shape)
    kw2 = dict(kw); kw2["initial_state"] = rnd(33, *kw["initial_state"].shape)
    o2, f2 = oracle.fwd(**d2, **kw2)
    d3 = dict(d); d3["v"] = 2.0 * d["v"] - 3.0 * d2["v"]
    kw3 = dict(kw); kw3["initial_state"] = 2.0 * kw["initial_state"] - 3.0 * kw2["initial_state"]
    o3, f3 = oracle.fwd(**d3, **kw3)
    assert np.allclose(o3, 2 * o1 - 3 * o2, rtol=1e-12, atol=1e-13)
    assert np.allclose(f3, 2 * f1 - 3 * f2, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("split", [1, 17, 63, 64, 65, 99])
def test_resume_chaining(split):
    """initial_state / final_state resume: two calls chained equal one call."""
    d, kw = make_case(41, B=1, T=130, H=1, HV=2, K=8, V=5)
    o, fs = oracle.fwd(**d, **kw)
    cut = lambda a, s: a[:, s]
    da = {n: cut(a, slice(0, split)) for n, a in d.items()}
    db = {n: cut(a, slice(split, None)) for n, a in d.items()}
    oa, fa = oracle.fwd(**da, **kw)
    kwb = dict(kw); kwb["initial_state"] = fa
    ob, fb = oracle.fwd(**db, **kwb)
    assert np.allclose(np.concatenate([oa, ob], axis=1), o, rtol=1e-12, atol=1e-13)
    assert np.allclose(fb, fs, rtol=1e-12, atol=1e-13)


def test_varlen_equals_separate_calls():
    r = np.random.default_rng(51)
    lens = [1, 5, 64, 33, 0, 97]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    Tpad = int(cu[-1]) + 7
    H, HV, K, V = 1, 2, 8, 5
    d = dict(q=r.standard_normal((1, Tpad, H, K)), k=r.standard_normal((1, Tpad, H, K)),
             v=r.standard_normal((1, Tpad, HV, V)), g=r.standard_normal((1, Tpad, HV, K)),
             beta=r.standard_normal((1, Tpad, HV)))
    h0 = r.standard_normal((len(lens), HV, K, V))
    kw = dict(A_log=r.standard_normal(HV), dt_bias=r.standard_normal(HV * K),
              gate_mode=GATE_SAFE, lower_bound=-3.0)
    o, fs = oracle.fwd(**d, **kw, initial_state=h0, cu_seqlens=cu)
    for n in range(len(lens)):
        s = slice(int(cu[n]), int(cu[n + 1]))
        dn = {name: a[:, s] for name, a in d.items()}
        on, fn = oracle.fwd(**dn, **kw, initial_state=h0[n:n + 1])
        assert np.allclose(o[:, s], on, rtol=1e-13, atol=1e-14)
        assert np.allclose(fs[n], fn[0], rtol=1e-13, atol=1e-14)
    assert np.all(o[:, int(cu[-1]):] == 0.0)
    # numpy recurrence and chunk form agree on the varlen layout as well
    o2, f2 = oracle.recurrent_np(**d, **kw, initial_state=h0, cu_seqlens=cu)
    o3, f3 = oracle.chunk_np(**d, **kw, initial_state=h0, cu_seqlens=cu, chunk_size=16)
    assert rel(o2, o) < 1e-12 and rel(f2, fs) < 1e-12
    assert rel(o3, o) < 1e-10 and rel(f3, fs) < 1e-10


def test_gva_equals_repeated_heads():
    """HV = G*H: value head hv reads q/k head hv // G, i.e. q, k repeat-interleaved by G."""
    d, kw = make_case(61, B=2, T=24, H=2, HV=6, K=8, V=4)
    o, fs = oracle.fwd(**d, **kw)
    dr = dict(d)
    dr["q"] = np.repeat(d["q"], 3, axis=2)
    dr["k"] = np.repeat(d["k"], 3, axis=2)
    orr, fr = oracle.fwd(**dr, **kw)
    assert np.allclose(o, orr, rtol=1e-14, atol=1e-15)
    assert np.allclose(fs, fr, rtol=1e-14, atol=1e-15)
    # ... and not the modulo mapping hv % H
    dm = dict(d)
    dm["q"] = np.tile(d["q"], (1, 1, 3, 1))
    dm["k"] = np.tile(d["k"], (1, 1, 3, 1))
    om, _ = oracle.fwd(**dm, **kw)
    assert rel(om, o) > 1e-3


# --------------------------------------------------------------------------------------
# Chunk form of the reading notes == token recurrence
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("gate", [GATE_SAFE, GATE_PLAIN, GATE_PREGATED])
@pytest.mark.parametrize("C", [32, 64, 5])
def test_chunk_form_equals_recurrence(gate, C):
    d, kw = make_case(71 + C, B=2, T=150, H=2, HV=4, K=16, V=8, gate=gate)
    o, fs = oracle.fwd(**d, **kw)
    oc, fc = oracle.chunk_np(**d, **kw, chunk_size=C)
    assert rel(oc, o) < 1e-10
    assert rel(fc, fs) < 1e-10


def test_chunk32_equals_chunk64_long_safe_gate():
    """At lower_bound = -5 the chunk cumsum reaches about -320 nat; the chunk form
    must still match (it never forms e^-Gamma on its own)."""
    d, kw = make_case(81, B=1, T=200, H=1, HV=1, K=32, V=16)
    d["g"] = 3.0 + np.abs(d["g"])          # push the safe gate towards its bound
    o32, f32 = oracle.chunk_np(**d, **kw, chunk_size=32)
    o64, f64 = oracle.chunk_np(**d, **kw, chunk_size=64)
    o, fs = oracle.fwd(**d, **kw)
    assert rel(o32, o64) < 1e-10 and rel(f32, f64) < 1e-10
    assert rel(o64, o) < 1e-10 and rel(f64, fs) < 1e-10


def test_numpy_recurrence_matches_c():
    d, kw = make_case(91, B=3, T=50, H=2, HV=4, K=16, V=8, gate=GATE_PLAIN)
    o, fs = oracle.fwd(**d, **kw)
    o2, f2 = oracle.recurrent_np(**d, **kw)
    assert rel(o2, o) < 1e-13 and rel(f2, fs) < 1e-13


def test_l2norm_eps_below_tolerance():
    """The norm's epsilon (pages silent) moves o by far less than the bf16 tolerance."""
    d, kw = make_case(101, B=1, T=64, H=1, HV=1, K=128, V=32)
    o0, f0 = oracle.fwd(**d, **kw, l2_eps=0.0)
    o1, f1 = oracle.fwd(**d, **kw, l2_eps=1e-6)
    assert rel(o1, o0) < 1e-6 and rel(f1, f0) < 1e-6


# --------------------------------------------------------------------------------------
# In-kernel L2 norm of q and k (use_qk_l2norm_in_kernel, "FLA-KDA engineering notes" 2.2)
# --------------------------------------------------------------------------------------

def _row_scaled(d, seed, lo=0.01, hi=100.0):
    """q and k with every (batch, token, head) row multiplied by its own positive constant."""
    r = np.random.default_rng(seed)
    out = dict(d)
    for name in ("q", "k"):
        c = np.exp(r.uniform(np.log(lo), np.log(hi), d[name].shape[:3]))[..., None]
        out[name] = d[name] * c
    return out


@pytest.mark.parametrize("gate", [GATE_SAFE, GATE_PLAIN])
def test_l2norm_output_is_invariant_to_row_scaling(gate):
    """x / ||x|| over K does not see a positive factor on a row: o and final_state are the
    same when every q and k row (each token and head its own factor, 1e-2 .. 1e2) is
    scaled.  Exact with epsilon 0; with the default epsilon to within its own size."""
    d, kw = make_case(141, B=2, T=30, H=2, HV=4, K=8, V=5, gate=gate)
    ds = _row_scaled(d, 142)
    o0, f0 = oracle.fwd(**d, **kw, l2_eps=0.0)
    o1, f1 = oracle.fwd(**ds, **kw, l2_eps=0.0)
    assert rel(o1, o0) < 1e-12 and rel(f1, f0) < 1e-12
    ds = _row_scaled(d, 143, lo=1.0, hi=10.0)
    o2, f2 = oracle.fwd(**ds, **kw)
    assert rel(o2, o0) < 1e-6 and rel(f2, f0) < 1e-6


def test_l2norm_three_four_five():
    """With K = 2 the key (3, 4) normalises to (0.6, 0.8) and the query (0, -2) to (0, -1):
    the normalising call equals the call given those unit vectors with the norm switched off."""
    r = np.random.default_rng(144)
    T = 3
    q = np.array([[0.0, -2.0], [5.0, 12.0], [-8.0, 6.0]]).reshape(1, T, 1, 2)
    k = np.array([[3.0, 4.0], [-0.3, 0.4], [1.0, 0.0]]).reshape(1, T, 1, 2)
    qu = np.array([[0.0, -1.0], [5 / 13, 12 / 13], [-0.8, 0.6]]).reshape(1, T, 1, 2)
    ku = np.array([[0.6, 0.8], [-0.6, 0.8], [1.0, 0.0]]).reshape(1, T, 1, 2)
    v = r.standard_normal((1, T, 1, 3))
    g = r.standard_normal((1, T, 1, 2))
    beta = r.standard_normal((1, T, 1))
    kw = dict(gate_mode=GATE_SAFE, A_log=np.zeros(1), lower_bound=-3.0,
              initial_state=r.standard_normal((1, 1, 2, 3)), scale=0.7)
    o_n, f_n = oracle.fwd(q, k, v, g, beta, qk_l2norm=True, l2_eps=0.0, **kw)
    o_u, f_u = oracle.fwd(qu, ku, v, g, beta, qk_l2norm=False, **kw)
    assert np.max(np.abs(o_n - o_u)) < 1e-12 and np.max(np.abs(f_n - f_u)) < 1e-12
    # the default epsilon (1e-6 inside the square root) moves a row of squared norm s by a
    # relative 1e-6 / (2 s) at most: 2e-6 for the shortest row here (s = 0.25)
    o_e, f_e = oracle.fwd(q, k, v, g, beta, qk_l2norm=True, **kw)
    assert rel(o_e, o_u) < 5e-6 and rel(f_e, f_u) < 5e-6


@pytest.mark.parametrize("mistake", ["no_sqrt", "norm_over_tokens", "norm_over_heads"])
def test_l2norm_pins_catch_a_planted_mistake(mistake):
    """The two pins above reject plausible wrong norms.  The mistake is planted on the CPU:
    q and k are normalised by the wrong formula here and passed with the norm switched off,
    which is what an oracle with that mistake would compute."""
    def wrong(x):
        if mistake == "no_sqrt":
            return x / np.sum(x * x, axis=-1, keepdims=True)
        axis = 1 if mistake == "norm_over_tokens" else 2
        return x / np.sqrt(np.sum(x * x, axis=axis, keepdims=True))
    d, kw = make_case(145, B=1, T=12, H=2, HV=2, K=4, V=3)
    ds = _row_scaled(d, 146)
    def mutant(dd):
        ee = dict(dd, q=wrong(dd["q"]), k=wrong(dd["k"]))
        return oracle.fwd(**ee, **kw, qk_l2norm=False)
    o0, _ = mutant(d)
    o1, _ = mutant(ds)
    assert rel(o1, o0) > 1e-3      # the invariance pin fails for the mutant
    q = np.array([0.0, -2.0, 3.0, 4.0]).reshape(1, 1, 2, 2)
    unit = np.array([0.0, -1.0, 0.6, 0.8]).reshape(1, 1, 2, 2)
    if mistake != "norm_over_heads":   # a per-row check does not see the head axis
        with np.errstate(invalid="ignore", divide="ignore"):
            assert not np.allclose(wrong(q), unit, atol=1e-3)


def test_empty_sequence_keeps_state():
    d, kw = make_case(111, B=1, T=0, H=1, HV=1, K=4, V=3)
    o, fs = oracle.fwd(**d, **kw)
    assert o.shape == (1, 0, 1, 3)
    assert np.array_equal(fs, kw["initial_state"])


# ---- allow_neg_eigval and the transposed state layout ------------------------------------

def test_neg_eigval_beta_near_two_is_a_householder_reflection():
    """With beta = 2 sigmoid(b) -> 2 (b = 40), no decay (pre-gated g = 0), v = 0 and a unit
    key, each token applies I - 2 k k^T to the state: a reflection.  One token negates the
    state's component along k; the same token twice restores the initial state."""
    rng = np.random.default_rng(17)
    K = V = 8
    kvec = rng.standard_normal(K)
    kvec /= np.sqrt(np.sum(kvec ** 2))                # a unit key (no in-kernel norm below)
    k = np.tile(kvec, (1, 2, 1, 1))                   # [1, 2, 1, K]: the same key twice
    q = rng.standard_normal((1, 2, 1, K))
    v = np.zeros((1, 2, 1, V))
    g = np.zeros((1, 2, 1, K))
    beta = np.full((1, 2, 1), 40.0)
    h0 = rng.standard_normal((1, 1, K, V))
    kw = dict(gate_mode=GATE_PREGATED, qk_l2norm=False, beta_sigmoid=True, allow_neg_eigval=True,
              initial_state=h0)
    _, fs2 = oracle.fwd(q, k, v, g, beta, **kw)
    assert np.allclose(fs2, h0, rtol=0, atol=1e-12)
    _, fs1 = oracle.fwd(q[:, :1], k[:, :1], v[:, :1], g[:, :1], beta[:, :1], **kw)
    assert np.allclose(kvec @ fs1[0, 0], -(kvec @ h0[0, 0]), rtol=0, atol=1e-12)
    # the part of the state orthogonal to k is untouched
    perp = h0[0, 0] - np.outer(kvec, kvec @ h0[0, 0])
    assert np.allclose(fs1[0, 0] - np.outer(kvec, kvec @ fs1[0, 0]), perp, rtol=0, atol=1e-12)


def test_neg_eigval_needs_beta_sigmoid():
    with pytest.raises(ValueError):
        oracle.fwd(np.zeros((1, 1, 1, 4)), np.zeros((1, 1, 1, 4)), np.zeros((1, 1, 1, 4)),
                   np.zeros((1, 1, 1, 4)), np.zeros((1, 1, 1)), gate_mode=GATE_PREGATED,
                   beta_sigmoid=False, allow_neg_eigval=True)


def test_transposed_state_layout_is_the_transpose():
    """state_v_first stores the K x V state as V x K, both ways."""
    rng = np.random.default_rng(23)
    B, T, H, K, V = 1, 9, 1, 6, 5
    d = dict(q=rng.standard_normal((B, T, H, K)), k=rng.standard_normal((B, T, H, K)),
             v=rng.standard_normal((B, T, H, V)), g=-np.abs(rng.standard_normal((B, T, H, K))),
             beta=rng.standard_normal((B, T, H)))
    h0 = rng.standard_normal((1, 1, K, V))
    o, fs = oracle.fwd(**d, gate_mode=GATE_PREGATED, initial_state=h0)
    oT, fsT = oracle.fwd(**d, gate_mode=GATE_PREGATED, initial_state=np.swapaxes(h0, -1, -2),
                         transpose_state_layout=True)
    assert fsT.shape == (1, 1, V, K)
    assert np.array_equal(oT, o) and np.array_equal(fsT, np.swapaxes(fs, -1, -2))



def test_intermediate_states_are_the_prefix_final_states():
    """return_intermediate_states: entry c of sequence n is the state after the first c
    chunks of that sequence, i.e. the final state of the same recurrence run on that prefix;
    chunks of later sequences follow those of earlier ones; an empty sequence has none."""
    rng = np.random.default_rng(29)
    H, K, V, C = 1, 6, 5, 4
    cu = np.array([0, 10, 10, 17], dtype=np.int64)   # lengths 10, 0, 7 -> 3 + 0 + 2 chunks
    T = int(cu[-1])
    d = dict(q=rng.standard_normal((1, T, H, K)), k=rng.standard_normal((1, T, H, K)),
             v=rng.standard_normal((1, T, H, V)), g=-np.abs(rng.standard_normal((1, T, H, K))),
             beta=rng.standard_normal((1, T, H)))
    h0 = rng.standard_normal((3, H, K, V))
    kw = dict(gate_mode=GATE_PREGATED, initial_state=h0)
    o, fs, hs = oracle.fwd(**d, **kw, cu_seqlens=cu, return_intermediate_states=True, chunk_size=C)
    assert hs.shape == (5, H, K, V)
    order = [(0, 0), (0, 1), (0, 2), (2, 0), (2, 1)]  # (sequence, chunk) of each entry
    for idx, (n, c) in enumerate(order):
        bos = int(cu[n])
        if c == 0:
            assert np.array_equal(hs[idx], h0[n])
            continue
        pre = {key: val[:, bos:bos + c * C] for key, val in d.items()}
        _, fpre = oracle.fwd(**pre, gate_mode=GATE_PREGATED, initial_state=h0[n:n + 1])
        assert np.allclose(hs[idx], fpre[0], rtol=1e-13, atol=1e-13)
