"""The replica aggregation of bench.py under torch.distributed (gloo, 2 ranks,
CPU): value = sum of tokens over ranks / the slowest rank's time."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    d = bench.Dist()
    assert d.pg is not None and d.world == world and d.rank == rank
    t = d.max(1.0 + rank)          # rank-local seconds: 1.0, 2.0
    tok = d.sum(100.0 * (rank + 1))  # tokens: 100, 200
    d.barrier()
    out[rank] = (t, tok, tok / t)
    d.pg.destroy_process_group()


def test_replica_aggregation_two_ranks():
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    for r in range(2):
        assert out[r] == (2.0, 300.0, 150.0)


def test_single_process_identity():
    import bench

    assert bench.reduce_scalar(None, 3.5, "max") == 3.5
    assert bench.reduce_scalar(None, 3.5, "sum") == 3.5
