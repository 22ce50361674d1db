"""Multi-GPU runs of the layer are independent replicas (no data-path
collective): every rank runs the whole layer on its own tokens, and the job's
time is the slowest rank's.  The rank logic of bench.py is tested here with two
gloo processes on the CPU."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import importlib.util
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    # rank r "took" 10 * (r + 1) ms: the job time is the slowest rank's
    t = bench.max_over_ranks(10.0 * (rank + 1), world)
    v = bench.replica_throughput(world, 128, 5, t)
    dist.barrier()
    out[rank] = (t, v)
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_sum_the_tokens():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        t, v = res[rank]
        assert t == 20.0
        assert v == pytest.approx(2 * 128 * 5 / 0.020)


def test_single_rank_is_the_identity():
    import importlib.util
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.replica_throughput(1, 128, 10, 5.0) == pytest.approx(128 * 10 / 0.005)
