"""The bench's multi-rank host logic (replicas: barrier, max over ranks,
whole-job aggregation) on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench._dist = True
    ms = 2.0 + 3.0 * rank                      # rank 1 is the slow one
    bench.barrier()
    worst = bench.dist_max(ms)
    value = bench.whole_job_tflops(1e12, world, worst)
    q.put((rank, worst, value))
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_and_whole_job_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.0, 5.0]
    # 2 replicas x 1 TFLOP each in 5 ms
    assert res[0][2] == pytest.approx(2 * 1e12 / 5e-3 / 1e12)
    assert res[0][2] == res[1][2]


def test_single_process_helpers_are_identity():
    import bench
    bench._dist = False
    assert bench.dist_max(3.5) == 3.5
    assert bench.whole_job_tflops(2e12, 1, 1.0) == pytest.approx(2000.0)
