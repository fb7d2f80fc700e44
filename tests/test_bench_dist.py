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


def test_replica_launch_command_runs_ranks_on_cpu():
    # the command bench.py runs for --gpus N outside torchrun, here starting two
    # CPU replicas of a probe that uses the bench's barrier and max-over-ranks
    import json
    import subprocess
    import bench
    probe = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_replica_probe.py")
    cmd = bench.replica_command(2, probe, ["--steps", "3"], _free_port())
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"] and "--nproc-per-node=2" in cmd
    assert "--master-addr=127.0.0.1" in cmd
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(line) == 1, r.stdout
    got = json.loads(line[0])
    assert got["world"] == 2 and got["worst_ms"] == 2.0 and got["argv"] == ["--steps", "3"]
    assert got["value"] == pytest.approx(2 * 1e12 / 2e-3 / 1e12)
