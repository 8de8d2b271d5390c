"""The multi-rank host logic of bench.py on CPU with gloo (world size 2).

On GPUs every rank runs its own batch with no exchange step; the only
collectives are the barrier and the maximum of the step time.  This checks
that aggregation: the job's time is the slowest rank's and the value counts
every rank's work.
"""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [10.0, 12.5][rank]
    ms, value = bench.aggregate(world, 3.0e12, local_ms)
    bench.barrier(world)
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_weak_scaling_aggregation_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in out:
        assert ms == pytest.approx(12.5)
        assert value == pytest.approx(2 * 3.0e12 / 12.5e-3 / 1e12)


def test_valid_pair_count_matches_brute_force():
    import numpy as np
    import bench
    rng = np.random.default_rng(0)
    lq = rng.integers(0, 40, size=7)
    lkv = rng.integers(0, 40, size=7)
    for causal in (False, True):
        brute = sum(int(((np.arange(b)[None, :] <= np.arange(a)[:, None]) | (not causal)).sum())
                    for a, b in zip(lq, lkv))
        assert bench.valid_pairs(lq, lkv, causal) == brute
        for window in (1, 3, 17):
            brute_w = sum(int((((np.arange(b)[None, :] <= np.arange(a)[:, None]) | (not causal))
                               & (np.abs(np.arange(a)[:, None] - np.arange(b)[None, :]) < window)).sum())
                          for a, b in zip(lq, lkv))
            assert bench.valid_pairs(lq, lkv, causal, window) == brute_w
