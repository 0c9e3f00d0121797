"""The multi-GPU mode of the benchmark is replicas only: every rank runs the
whole path on its own inputs, and the only cross-rank step is the timing
(the slowest rank's step time).  Checked here with two gloo ranks on CPU."""
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


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [0.5, 0.8][rank]  # the second rank is slower
        ms = bench.replica_step_ms(local_ms, world, torch.device("cpu"))
        out[rank] = (ms, bench.replica_throughput(512, ms, world))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == out[1]                       # every rank agrees
    ms, value = out[0]
    assert ms == pytest.approx(0.8)               # the slowest rank's step time
    assert value == pytest.approx(512 * 2 / 0.8e-3)  # whole-job positions per second


def test_single_replica_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_step_ms(0.5, 1, torch.device("cpu")) == 0.5
    assert bench.replica_throughput(512, 0.5, 1) == pytest.approx(512 / 0.5e-3)
