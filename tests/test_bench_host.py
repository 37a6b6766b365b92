"""Host logic of bench.py without a GPU: algorithmic byte counts and the
max-over-ranks timing reduction on world_size-2 gloo ranks."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench


def test_algorithmic_bytes_closed_form():
    total, attend = bench.algorithmic_bytes([16, 17])
    kv = 33 * 8 * 128 * 2
    scales = 33 * 8 * 4 * 2
    bt = (1 + 2) * 4
    q = 2 * 32 * 128 * 2
    assert attend == kv + scales + bt + q
    assert total == attend + 2 * 32 * (128 * 2 + 4) + 2 * 8 * (128 * 4 + 132 * 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(world)
    out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}
