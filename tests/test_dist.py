"""Multi-process host logic on CPU: two gloo ranks reduce step timing like bench.py does."""
import os
import socket

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


# ----------------------------------------------------------------------------- context-parallel exchange

def _pack(st, g):
    """Oracle partial state -> records [g, 136] (m, Z, S_A, S_B, S_V, 3 unused, acc)."""
    rec = torch.zeros((g, 136), dtype=torch.float64)
    rec[:, 0] = torch.from_numpy(st["m"])
    rec[:, 1] = torch.from_numpy(st["Z"])
    rec[:, 2] = torch.from_numpy(st["SA"])
    rec[:, 3] = torch.from_numpy(st["SB"])
    rec[:, 4] = torch.from_numpy(st["SV"])
    rec[:, 8:] = torch.from_numpy(st["acc"])
    return rec


def _cp_worker(rank, world, port, q):
    import numpy as np
    from oracle import meter
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(11)                      # same data on every rank
    S, g, d = 300, 4, 128
    qv = rng.standard_normal((g, d))
    kh = rng.standard_normal((S, d))
    vh = rng.standard_normal((S, d))
    ca = rng.uniform(0, 0.3, (g, S))
    cb = rng.uniform(0, 0.1, (g, S))
    wv = rng.uniform(0, 0.2, S)
    bounds = [0, 137, S]                                 # rank r holds positions bounds[r] .. bounds[r+1]-1
    local = _pack(meter.partial_state(qv, kh, vh, ca, cb, bounds[rank], bounds[rank + 1], wv), g)
    allp = wdist.gather_partials(local.unsqueeze(0)).squeeze(0)     # [g, world, 136]
    states = [dict(m=allp[:, r, 0].numpy(), Z=allp[:, r, 1].numpy(), SA=allp[:, r, 2].numpy(),
                   SB=allp[:, r, 3].numpy(), SV=allp[:, r, 4].numpy(), acc=allp[:, r, 8:].numpy())
              for r in range(world)]
    merged = meter.merge_states(states)
    whole = meter.merge_states([meter.partial_state(qv, kh, vh, ca, cb, 0, S, wv)])
    _, p, out = meter.attention(qv, kh, vh)
    ok = (torch.equal(allp[:, rank], local)
          and np.allclose(merged["out"], out, rtol=1e-12, atol=1e-12)
          and np.allclose(merged["D_a"], whole["D_a"], rtol=1e-12)
          and np.allclose(merged["D_b"], whole["D_b"], rtol=1e-12)
          and np.allclose(merged["meter_v"], p @ wv, rtol=1e-12))
    q.put((rank, bool(ok)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_context_parallel_exchange_and_merge_over_gloo():
    """Two ranks hold positions [0, 137) and [137, 300) of one context; their partial records,
    gathered over gloo, merge to the single-context attention output and meter sums."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_cp_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, True), (1, True)]


def test_single_process_gather_is_one_shard():
    x = torch.arange(12.0).reshape(1, 2, 6)
    assert wdist.gather_partials(x).shape == (1, 2, 1, 6)
