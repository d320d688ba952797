"""The multi-rank accounting of bench.py (replicas only): two gloo ranks on
CPU agree on the slowest rank's time and report all ranks' tokens over it."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = 2.0 + rank          # rank 1 is the slow one
    value, ms = bench.replica_throughput(256, ms_local, world)
    bench.barrier(world)
    out[rank] = (value, ms)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_total_tokens():
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1]
    value, ms = out[0]
    assert ms == 3.0
    assert value == pytest.approx(2 * 256 / 3.0e-3)


def test_single_rank_needs_no_process_group():
    import bench
    value, ms = bench.replica_throughput(100, 4.0, 1)
    assert ms == 4.0 and value == pytest.approx(100 / 4.0e-3)
