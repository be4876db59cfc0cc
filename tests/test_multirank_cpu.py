"""Multi-rank host logic of bench.py on CPU ranks (gloo, world size 2).

The operation shards over independent (sequence, head) replicas with no
collective on the data path; the only cross-rank steps are the barrier and the
max-over-ranks reduction of the timed region, which these tests exercise with
two real processes.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, local_ms, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        t = bench.max_over_ranks(local_ms[rank], world)
        v = bench.job_throughput(t, world, 8192, 4)
        q.put((rank, t, v, bench.replica_seed(1, rank)))
    finally:
        dist.destroy_process_group()


def _run(world, local_ms):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, local_ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def test_max_over_ranks_and_job_throughput_gloo_2():
    res = _run(2, [10.0, 15.0])
    assert [r[0] for r in res] == [0, 1]
    for _, t, v, _ in res:
        assert t == 15.0  # every rank sees the slowest rank's time
        assert v == pytest.approx(2 * 8192 * 4 / 0.015)
    assert res[0][3] != res[1][3]  # replicas draw different inputs


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1000.0, 1, 100, 10) == pytest.approx(1000.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import argparse

    import bench
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(workload="prefill_h32_t8192", warmup=3, steps=2, gpus=2, ref_tokens=64)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def _oracle_fns(scale, l2norm):
    import numpy as np
    import torch

    import oracle
    from gated_deltanet_linear_15_gb300 import cp

    def fwd(q, k, v, g, beta, S0):
        o, ST = oracle.fwd(q, k, v, g, beta, S0, None, scale=scale, l2norm=l2norm)
        return torch.from_numpy(o), torch.from_numpy(ST)

    def bwd(q, k, v, g, beta, dO, S0, dST):
        r = oracle.bwd(q, k, v, g, beta, dO, S0, dST, None, scale=scale, l2norm=l2norm)
        return tuple(torch.from_numpy(np.asarray(r[key])) for key in ("dq", "dk", "dv", "dg", "dbeta", "dS0"))

    return cp.ShardFns(fwd, bwd)


def _cp_worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import oracle
    from gated_deltanet_linear_15_gb300 import cp
    from gdn_inputs import make_inputs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = make_inputs("tiny_fp32", "cpu", T=96, H=2, B=1, with_S0=True, with_dST=True, seed=41)
        fns = _oracle_fns(x["scale"], x["l2norm"])
        cuts = [0, 40, 96]
        sh = {k: x[k][:, cuts[rank]:cuts[rank + 1]].contiguous() for k in ("q", "k", "v", "g", "beta", "dO")}
        o, S_end, S_start, M = cp.cp_forward(sh["q"], sh["k"], sh["v"], sh["g"], sh["beta"],
                                             x["S0"].double(), fns=fns)
        grads = cp.cp_backward(sh["q"], sh["k"], sh["v"], sh["g"], sh["beta"], sh["dO"], S_start, M,
                               x["dST"].double(), fns=fns)
        ref_o, ref_ST = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], None, scale=x["scale"],
                                   l2norm=x["l2norm"])
        ref = oracle.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["dO"], x["S0"], x["dST"], None,
                         scale=x["scale"], l2norm=x["l2norm"])
        a, b = cuts[rank], cuts[rank + 1]
        errs = {"o": float(abs(o.numpy() - ref_o[:, a:b]).max())}
        for i, key in enumerate(("dq", "dk", "dv", "dg", "dbeta")):
            errs[key] = float(abs(grads[i].numpy() - ref[key][:, a:b]).max())
        if rank == world - 1:
            errs["S_T"] = float(abs(S_end.numpy() - ref_ST).max())
        if rank == 0:
            errs["dS0"] = float(abs(grads[5].numpy() - ref["dS0"]).max())
        q.put((rank, errs))
    finally:
        dist.destroy_process_group()


def test_context_parallel_two_ranks_gloo():
    """Sequence split over two CPU ranks; the per-shard work is the fp64 oracle (test-only
    stand-in for the library), so the exchange and the composition must reproduce the oracle
    over the whole sequence to rounding."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_cp_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, errs in out:
        assert all(e < 1e-9 for e in errs.values()), (rank, errs)
    assert "S_T" in out[1][1] and "dS0" in out[0][1]
