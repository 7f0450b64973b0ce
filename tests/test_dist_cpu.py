"""Multi-process plumbing of bench.py on the CPU (gloo, world size 2): each
rank is an independent replica; timings are combined by a max over ranks,
and only rank 0 prints.  No GPU and no data-path collective is involved."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        bench.barrier(w)
        out[rank] = (r, w, local, bench.max_over_ranks(10.0 * (rank + 1), w))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True,
                       start_method="spawn")
    assert out[0] == (0, 2, 0, 20.0)
    assert out[1] == (1, 2, 1, 20.0)


def test_single_rank_defaults(monkeypatch):
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
