"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks.

The path shards into independent replicas (no collective on the data path);
what bench.py does across ranks is a barrier around the timed region and the
maximum of the ranks' times. These run here with the gloo backend.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got == [(0, 2.5), (1, 2.5)]


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1, None) == 3.25
