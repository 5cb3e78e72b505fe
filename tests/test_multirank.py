"""Multi-rank host logic of bench.py on CPU: two gloo ranks (world_size 2, 127.0.0.1).

bench.py runs one independent replica of the decode workload per rank (weak scaling, no data-path
collective); the only collective is the max over ranks of the step time, from which the whole job's
throughput is world / max time.  The reference arm (the oracle on host cores) runs on rank 0 only.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, local_ms, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    value, ms = bench.job_throughput(local_ms[rank], world, dist, torch.device("cpu"))
    results[rank] = (value, ms)
    dist.barrier()
    dist.destroy_process_group()


def test_job_throughput_takes_the_slowest_rank():
    world, port = 2, _free_port()
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    local = [2.0, 5.0]   # ms per step measured on each rank
    mp.start_processes(_worker, args=(world, port, local, results), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        value, ms = results[r]
        assert ms == pytest.approx(5.0)
        assert value == pytest.approx(world * 1000.0 / 5.0)


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.job_throughput(4.0, 1)
    assert ms == 4.0 and value == pytest.approx(250.0)


def _ref_worker(rank, world, port, printed):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import argparse
    import contextlib
    import io

    import bench
    args = argparse.Namespace(gpus=world, steps=1, warmup=0, impl="reference", workload="tiny", B=0, T=0, layers=0,
                              no_e2e=True, no_cpu_baseline=True, dense=False)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, rank)
    printed[rank] = buf.getvalue()
    dist.barrier()
    dist.destroy_process_group()


def test_reference_arm_runs_on_rank_zero_only():
    import json
    world, port = 2, _free_port()
    manager = mp.get_context("spawn").Manager()
    printed = manager.dict()
    mp.start_processes(_ref_worker, args=(world, port, printed), nprocs=world, start_method="spawn", join=True)
    assert printed[1] == ""
    line = json.loads(printed[0].strip())
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
