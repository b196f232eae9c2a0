"""The multi-rank path of bench.py on CPU: two gloo ranks (127.0.0.1) reduce
their timed regions to the slowest one and report the weak-scaling aggregate;
no collective touches the data path."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [1.5, 4.0][rank]  # rank 1 is the slow one
    got = bench.max_over_ranks(ms, device="cpu")
    value = bench.weak_scaling_value(world, 2.0e9, got)
    out[rank] = (got, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        ms, value = out[r]
        assert ms == pytest.approx(4.0)
        assert value == pytest.approx(2 * 2.0e9 / 4.0e-3 / 1e9)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.weak_scaling_value(1, 1.0e9, 1.0) == pytest.approx(1000.0)


def test_launch_ranks_runs_torchrun_on_loopback(monkeypatch):
    """bench.py --gpus N (outside torchrun) re-launches itself as N ranks of one
    node, rendezvous on 127.0.0.1, and returns torchrun's exit code."""
    seen = {}

    def fake_call(cmd):
        seen["cmd"] = cmd
        return 3

    monkeypatch.setattr(bench.subprocess, "call", fake_call)
    rc = bench.launch_ranks(4, ["--gpus", "4", "--steps", "7"])
    cmd = seen["cmd"]
    assert rc == 3
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nnodes=1" in cmd and "--nproc-per-node=4" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert int(cmd[cmd.index("--master-port") + 1]) > 0
    assert cmd[-5].endswith("bench.py") and cmd[-4:] == ["--gpus", "4", "--steps", "7"]
