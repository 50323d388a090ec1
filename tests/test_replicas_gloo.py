"""The multi-GPU path of bench.py is replicas only: each rank runs its own seeded copy of the
workload, the job's figure is every rank's tokens over the slowest rank's time, and only rank
0 prints.  These checks run that host logic as two gloo ranks on the CPU (no GPU)."""
import io
import os
import sys
import contextlib

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    from kimi_delta_attention_gate_gb300 import inputs as kin
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = kin.WORKLOADS["tiny_fp32"]
        inp = bench.replica_inputs(wl, rank)
        local_ms = 1.0 + 0.5 * rank                     # rank 1 is the slower one
        ms = bench.max_over_ranks(local_ms, dist)
        value = bench.job_throughput(inp.n_tokens, world, ms)
        # the replicas differ in values but not in shape
        digest = float(np.sum(inp.q[:, :4]))
        gathered = [None] * world
        dist.all_gather_object(gathered, (ms, value, inp.q.shape, digest))
        out[rank] = gathered
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_job_throughput():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = 29500 + (os.getpid() % 2000)
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p_ in procs:
            p_.start()
        for p_ in procs:
            p_.join(120)
            assert p_.exitcode == 0
        res = dict(out)
    for rank in range(2):
        (ms0, v0, shape0, d0), (ms1, v1, shape1, d1) = res[rank]
        assert ms0 == ms1 == 1.5                         # max over ranks, seen by both
        assert v0 == v1 == pytest.approx(256 * 2 / 1.5e-3)  # tiny_fp32: 256 tokens per rank
        assert shape0 == shape1 and d0 != d1             # replicas: same shapes, own seeds


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from kimi_delta_attention_gate_gb300 import inputs as kin
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    args = type("A", (), {"steps": 1, "warmup": 0, "gpus": 2})()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(args, kin.WORKLOADS["tiny_fp32"]) == 0
    assert buf.getvalue() == ""
