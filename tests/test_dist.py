"""Multi-process host logic on CPU: two gloo ranks reduce step timing like bench.py does."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from kv_cache_quantization_witcert_gb300 import dist as wdist


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, lr, w = wdist.rank_env()
    ms, tok = wdist.reduce_timing(10.0 * (rank + 1), 1000.0 * (rank + 1))
    q.put((r, w, ms, tok, wdist.shard_seed(7, r)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_reduction_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got)
    assert all(g[2] == 20.0 and g[3] == 3000.0 for g in got)       # max time, total tokens
    assert got[0][4] != got[1][4]                                 # each rank serves other sequences


def test_single_process_reduction_is_identity():
    assert wdist.reduce_timing(3.5, 42) == (3.5, 42.0)
