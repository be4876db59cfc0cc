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
