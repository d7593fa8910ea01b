"""The multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

The decode step has no cross-sequence exchange, so N GPUs run N replicas of
the batch; the only collective is the timing reduction (max over ranks) used
for the whole-job throughput. This checks that logic without a GPU.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed_ms = [10.0, 12.5][rank]  # rank 1 is the slow one
    m = bench.reduce_max(elapsed_ms, world)
    results[rank] = (m, bench.job_tokens_per_s(256 * 100, m, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs)
        got = dict(results)
    assert got[0][0] == got[1][0] == 12.5
    assert got[0][1] == pytest.approx(2 * 256 * 100 / 12.5e-3)


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.reduce_max(3.0, 1) == 3.0
    assert bench.job_tokens_per_s(256, 1.0, 1) == pytest.approx(256_000.0)
