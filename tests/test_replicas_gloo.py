"""The N > 1 path of bench.py on CPU: replicas time independently and rank 0
reports the maximum over ranks (gloo, world size 2, rendezvous on 127.0.0.1)."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist, r, w = bench.dist_init()
    assert (r, w) == (rank, world)
    bench.barrier(dist)
    got = bench.max_over_ranks(dist, 1.5 + rank)   # each replica's own time
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_world_size_2():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == 2.5 and out[1] == 2.5
