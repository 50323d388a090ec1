"""Context parallelism (sequence sharding, kimi_delta_attention_gate_gb300.cp) on CPU ranks.

Two (and three) gloo ranks each hold a contiguous, unequal range of the tokens of every
sequence.  Each forms its shard's affine state maps, the ranks exchange them, each chains
the maps before its own and runs its shard from the state that enters it.  The forward pass
and the map application are given as the oracle's token recurrence and a NumPy product, so
the exchange logic of the product code runs without a GPU; the result must equal one oracle
call over the whole sequences (o of every shard, and the final state on the last rank)."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(seed, B=2, T=41, H=2, HV=4, K=6, V=5):
    r = np.random.default_rng(seed)
    return dict(q=r.standard_normal((B, T, H, K)), k=r.standard_normal((B, T, H, K)),
                v=r.standard_normal((B, T, HV, V)), g=r.standard_normal((B, T, HV, K)),
                beta=r.standard_normal((B, T, HV)), A_log=r.standard_normal(HV),
                dt_bias=r.standard_normal(HV * K), h0=0.3 * r.standard_normal((B, HV, K, V)))


def _oracle_ops(opts):
    """fwd / apply callables with the signatures cp.py expects, computed by the oracle."""
    import torch
    import oracle

    def fwd(q, k, v, g, beta, *, initial_state=None, transpose_state_layout=False, A_log=None,
            dt_bias=None, lower_bound=None, scale=None, allow_neg_eigval=False):
        h0 = None if initial_state is None else initial_state.double().numpy()
        o, fs = oracle.fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                           g.double().numpy(), beta.double().numpy(), A_log=A_log.numpy(),
                           dt_bias=dt_bias.numpy(), gate_mode=oracle.GATE_SAFE,
                           lower_bound=lower_bound, scale=scale, initial_state=h0,
                           allow_neg_eigval=allow_neg_eigval,
                           transpose_state_layout=transpose_state_layout)
        return torch.from_numpy(o), torch.from_numpy(np.ascontiguousarray(fs))

    def apply(P, R, S):
        if S is None:
            return R.clone()
        if opts.get("transpose_state_layout"):
            return S @ P.transpose(-1, -2) + R       # stored transposed: S^T P^T + R^T
        return P @ S + R

    return fwd, apply


def _rank_main(rank, world, port, bounds, opts, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    from kimi_delta_attention_gate_gb300 import cp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = _inputs(7)
        t0, t1 = bounds[rank], bounds[rank + 1]
        sh = {n: torch.from_numpy(np.ascontiguousarray(d[n][:, t0:t1]))
              for n in ("q", "k", "v", "g", "beta")}
        h0 = d["h0"]
        if opts.get("transpose_state_layout"):
            h0 = np.swapaxes(h0, -1, -2)
        fwd, apply = _oracle_ops(opts)
        o, s_out = cp.cp_fwd(sh["q"], sh["k"], sh["v"], sh["g"], sh["beta"],
                             initial_state=torch.from_numpy(np.ascontiguousarray(h0)),
                             fwd=fwd, apply=apply, A_log=torch.from_numpy(d["A_log"]),
                             dt_bias=torch.from_numpy(d["dt_bias"]), lower_bound=-5.0, scale=0.4,
                             **opts)
        out[rank] = (o.numpy(), s_out.numpy())
    finally:
        dist.destroy_process_group()


def _run(bounds, opts, port_off):
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    world = len(bounds) - 1
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = 31000 + port_off + (os.getpid() % 1500)
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, bounds, opts, out))
                 for r in range(world)]
        for p_ in procs:
            p_.start()
        for p_ in procs:
            p_.join(180)
            assert p_.exitcode == 0
        return dict(out)


@pytest.mark.parametrize("bounds,opts", [
    ((0, 23, 41), {}),
    ((0, 5, 30, 41), {"transpose_state_layout": True, "allow_neg_eigval": True}),
])
def test_sharded_ranks_equal_one_call_over_the_whole_sequence(bounds, opts):
    import oracle
    res = _run(bounds, opts, 17 * len(bounds))
    d = _inputs(7)
    h0 = np.swapaxes(d["h0"], -1, -2) if opts.get("transpose_state_layout") else d["h0"]
    ro, rfs = oracle.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], A_log=d["A_log"],
                         dt_bias=d["dt_bias"], gate_mode=oracle.GATE_SAFE, lower_bound=-5.0,
                         scale=0.4, initial_state=h0, **opts)
    world = len(bounds) - 1
    for r in range(world):
        o, s_out = res[r]
        t0, t1 = bounds[r], bounds[r + 1]
        assert np.max(np.abs(o - ro[:, t0:t1])) < 1e-10, r
    # the last rank ends with the whole sequences' final state
    assert np.max(np.abs(res[world - 1][1] - rfs)) < 1e-10


def test_chain_is_the_exclusive_prefix():
    """chain() on explicit maps: S_in(j+1) = P_j S_in(j) + R_j, S_in(0) = h0."""
    import torch
    from kimi_delta_attention_gate_gb300 import cp
    r = np.random.default_rng(3)
    P = [torch.from_numpy(r.standard_normal((2, 3, 3))) for _ in range(3)]
    R = [torch.from_numpy(r.standard_normal((2, 3, 4))) for _ in range(3)]
    h0 = torch.from_numpy(r.standard_normal((2, 3, 4)))
    _, apply = _oracle_ops({})
    st = cp.chain(P, R, h0, apply=apply)
    assert len(st) == 4 and st[0] is h0
    ref = h0.numpy()
    for j in range(3):
        ref = P[j].numpy() @ ref + R[j].numpy()
        assert np.allclose(st[j + 1].numpy(), ref, atol=1e-12)
    st0 = cp.chain(P[:1], R[:1], None, apply=apply)
    assert np.array_equal(st0[1].numpy(), R[0].numpy())
