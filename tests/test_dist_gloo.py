"""Multi-process host logic of the benchmark on CPU (gloo, world size 2):
every rank draws its own independent batch (requests shard with no
collective on the data path) and the timing is the maximum over ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    w = W.custom(bench.rank_seed("large_batch_decode", r), q_lens=[1] * 4,
                 seq_lens=[300, 400, 500, 600], hq=4, di=64, topk=2)
    fake_ms = 10.0 * (rank + 1)
    t = torch.tensor([fake_ms])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    out[rank] = (float(t.item()), int(w.idx_q.astype(np.int64).sum()), w.num_rows)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_independent_batches_and_max_time():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    (t0, s0, n0), (t1, s1, n1) = out[0], out[1]
    assert t0 == t1 == 20.0          # both ranks see the max over ranks
    assert s0 != s1                  # different requests on each rank
    assert n0 == n1 == 4             # the same per-rank work (weak scaling)


def test_rank_seeds_are_distinct():
    import bench
    seeds = {bench.rank_seed(name, r) for name in bench.W_SEED for r in range(8)}
    assert len(seeds) == 8 * len(bench.W_SEED)
