"""The N > 1 path of bench.py on CPU: gloo, world size 2, no GPU.

Each rank runs an independent replica (heads are independent; no collective on the data path);
the job's time is the slowest rank's and the job's throughput sums the replicas' work.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [1.0 + rank, 10.0 - rank, 0.5 * (rank + 1)]
    agg = bench.aggregate_over_ranks(local, world)
    dist.barrier()
    out[rank] = agg
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == [2.0, 10.0, 1.0]


def test_job_throughput_sums_replicas():
    import bench
    one = bench.job_tflops(1, 2e12, 1.0)
    two = bench.job_tflops(2, 2e12, 1.0)
    assert one == pytest.approx(2000.0) and two == pytest.approx(2 * one)


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")

    class A:  # the parsed arguments the reference arm reads
        workload = bench.DEFAULT_WORKLOAD
        steps = 1
        warmup = 0
        gpus = 2
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
