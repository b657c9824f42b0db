"""The N > 1 path of the benchmark: independent replicas whose whole-job figure
is the tokens of all ranks over the slowest rank's step time. Run as two gloo
ranks on CPU (no GPU, no data-path collective)."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [2.0, 3.0][rank]
    tok_local = [8192, 8192][rank]
    ms, tok, value = bench.replica_aggregate(ms_local, tok_local, dist, torch.device("cpu"))
    q.put((rank, ms, tok, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tok, value in res:
        assert ms == 3.0 and tok == 16384
        assert value == pytest.approx(16384 / 3e-3)


def test_single_replica_passthrough():
    import bench
    assert bench.replica_aggregate(4.0, 100) == (4.0, 100, 100 / 4e-3)
