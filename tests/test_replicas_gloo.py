"""Multi-GPU host logic on CPU: replicas with max-over-ranks timing (gloo, 2 ranks).

The path shards by token batch with no exchange, so N GPUs run N independent
replicas; the only cross-rank step is the timing reduction, checked here.
"""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = [120.0, 150.0][rank]  # ms; rank 1 is the slowest
    m = bench.max_over_ranks(elapsed)
    v = bench.aggregate_tokens_per_s(16384, 100, world, m)
    out[rank] = (m, v)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        m, v = out[r]
        assert m == 150.0
        assert abs(v - 16384 * 100 * 2 / 0.150) < 1e-6 * v


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.aggregate_tokens_per_s(1000, 10, 1, 10.0) == 1e6
