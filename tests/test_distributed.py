"""Host side of the multi-GPU benchmark on CPU: two gloo ranks.

The product path does not communicate between GPUs (each rank runs an
independent replica), so the only multi-process logic is the benchmark's
barrier and max-over-ranks timing, exercised here without a GPU.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (world, rank, rank)
    bench.barrier(world)
    slowest = bench.reduce_max_over_ranks(1.5 * (rank + 1), world)
    bench.barrier(world)
    q.put((rank, slowest))
    dist.destroy_process_group()


@pytest.mark.timeout(120) if hasattr(pytest.mark, "timeout") else (lambda f: f)
def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert results == {0: 3.0, 1: 3.0}


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max_over_ranks(2.5, 1) == 2.5
