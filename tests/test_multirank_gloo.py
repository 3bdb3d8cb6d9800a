"""The N > 1 path of the benchmark, on CPU: ranks are independent replicas
(the delta has no exchange step between tokens or batches), so a weak-scaled
run reports the slowest rank's time and the tokens of every rank. Two gloo
ranks check the reduction the benchmark uses."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, tok = bench.reduce_over_ranks(10.0 + 5.0 * rank, 100 * (rank + 1))
        dist.barrier()
        q.put((rank, ms, tok))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_benchmark():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0, 300), (1, 15.0, 300)]


def test_single_process_is_unchanged():
    import bench
    assert bench.reduce_over_ranks(3.5, 42) == (3.5, 42)
