"""Host logic of bench.py across two gloo ranks on CPU: timings are maxed and token counts summed over
ranks, as the multi-replica run reports them."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    r, local, ws = bench.dist_setup()
    bench.barrier(ws)
    mx = bench.max_over_ranks(10.0 + r, ws)
    sm = bench.sum_over_ranks(8.0, ws)
    out[rank] = (r, ws, mx, sm)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_ranks_max_and_sum():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(port, out), nprocs=2, join=True)
    assert out[0] == (0, 2, 11.0, 16.0)
    assert out[1] == (1, 2, 11.0, 16.0)
