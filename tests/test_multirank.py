"""Multi-process paths on CPU with gloo, world size 2 (no GPU).

* bench.py's timing reduction: every rank reports its step time and rank 0
  takes the maximum over ranks.
* Context-parallel verification (one long sequence split by key range over
  ranks): each rank computes softmax attention over its own key range, the
  (o, lse) partials are all-gathered, and the log-sum-exp merge reproduces
  single-pass attention over all keys.  Uses the oracle for the per-rank
  attention and the merge.
"""
import math
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _max_worker(rank, world, port, results):
    _init(rank, world, port)
    import bench

    value = bench.max_over_ranks(10.0 * (rank + 1), world, torch.device("cpu"))
    results[rank] = value
    dist.destroy_process_group()


def test_bench_takes_the_max_over_ranks():
    world, port = 2, _free_port()
    results = mp.Manager().dict()
    mp.spawn(_max_worker, args=(world, port, results), nprocs=world, join=True)
    assert dict(results) == {0: 20.0, 1: 20.0}


def _cp_worker(rank, world, port, results):
    _init(rank, world, port)
    import oracle

    g = torch.Generator().manual_seed(5)
    n, D = 1000, 64
    q = (torch.randn(D, generator=g) * 0.3).to(torch.bfloat16)
    k = torch.randn((n, D), generator=g).to(torch.bfloat16)
    v = torch.randn((n, D), generator=g).to(torch.bfloat16)
    lo, hi = rank * n // world, (rank + 1) * n // world
    member = np.zeros(n, dtype=bool)
    member[lo:hi] = True
    o, lse = oracle.attend_subset(q, k, v, member, 0.125)
    part = torch.tensor(np.concatenate([o, [lse]]), dtype=torch.float64)
    gathered = [torch.empty_like(part) for _ in range(world)]
    dist.all_gather(gathered, part)
    parts = torch.stack(gathered).numpy()
    out, out_lse = oracle.lse_merge(parts[None, :, :D], parts[None, :, D])
    full, full_lse = oracle.attend_subset(q, k, v, np.ones(n, dtype=bool), 0.125)
    results[rank] = (float(np.abs(out[0] - full).max()), abs(float(out_lse[0]) - full_lse))
    dist.destroy_process_group()


def test_context_parallel_merge_equals_single_pass():
    world, port = 2, _free_port()
    results = mp.Manager().dict()
    mp.spawn(_cp_worker, args=(world, port, results), nprocs=world, join=True)
    for r in range(world):
        err, lse_err = results[r]
        assert err < 1e-12 and lse_err < 1e-12
