"""Multi-process (world size 2, gloo on CPU) checks of the N > 1 host path.

Each rank owns a contiguous range of whole chunks and steps it alone; the
gathered result must equal one process stepping the whole buffer with the
same per-shard seeds, and the reported step time is the maximum over ranks.
"""

import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.demo_ref as ref
from decoupled_momentum_optimizer_gb300.sharding import CHUNK, max_over_ranks, shard_range, shard_seed


def test_shard_range_covers_exactly():
    for n in (32, 64, 32 * 7, 65536, 222903552):
        for world in (1, 2, 3, 4, 8):
            prev = 0
            sizes = []
            for r in range(world):
                lo, hi = shard_range(n, r, world)
                assert lo == prev and lo % CHUNK == 0 and hi % CHUNK == 0
                sizes.append(hi - lo)
                prev = hi
            assert prev == n
            assert max(sizes) - min(sizes) <= CHUNK
    with pytest.raises(ValueError):
        shard_range(33, 0, 1)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs(n, R, t):
    rng = np.random.default_rng(100 + t)
    return [rng.standard_normal(n).astype(np.float32).astype(np.float64) * 1e-2 for _ in range(R)]


def _worker(rank, world, port, n, R, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lo, hi = shard_range(n, rank, world)
    theta = (np.random.default_rng(1).standard_normal(n) * 2e-2)[lo:hi]
    ms = [np.zeros(hi - lo) for _ in range(R)]
    for t in range(3):
        gs = [g[lo:hi] for g in _inputs(n, R, t)]
        for mode, k in ((ref.MODE_DEMO, 4), (ref.MODE_RANDOM, 8)):
            theta, ms, _ = ref.step(theta, ms, gs, beta=0.9, lr=0.1, k=k, mode=mode, sign=True,
                                    seed=shard_seed(5, rank), step_idx=t)
    parts = [None] * world
    dist.all_gather_object(parts, (lo, hi, theta, ms))
    slowest = max_over_ranks(1.0 + rank, dist)
    if rank == 0:
        out_q.put((parts, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_shards_match_per_shard_reference():
    n, R, world = 32 * 37, 2, 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n, R, q)) for r in range(world)]
    for p in procs:
        p.start()
    parts, slowest = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert slowest == 2.0
    # one process, the same shards and seeds, stepped back to back
    theta_full = np.random.default_rng(1).standard_normal(n) * 2e-2
    for rank, (lo, hi, th, ms) in enumerate(parts):
        assert (lo, hi) == shard_range(n, rank, world)
        theta = theta_full[lo:hi]
        mm = [np.zeros(hi - lo) for _ in range(R)]
        for t in range(3):
            gs = [g[lo:hi] for g in _inputs(n, R, t)]
            for mode, k in ((ref.MODE_DEMO, 4), (ref.MODE_RANDOM, 8)):
                theta, mm, _ = ref.step(theta, mm, gs, beta=0.9, lr=0.1, k=k, mode=mode, sign=True,
                                        seed=shard_seed(5, rank), step_idx=t)
        assert np.abs(theta - th).max() <= 1e-15
        for a, b in zip(mm, ms):
            assert np.abs(a - b).max() <= 1e-15
    # DeMo chunks are independent of the shard split: rank-sharded DeMo equals the whole-buffer step
    th_full, _, _ = ref.step(theta_full, [np.zeros(n)] * R, _inputs(n, R, 0), beta=0.9, lr=0.1, k=4,
                             mode=ref.MODE_DEMO, sign=True)
    pieces = [ref.step(theta_full[lo:hi], [np.zeros(hi - lo)] * R, [g[lo:hi] for g in _inputs(n, R, 0)],
                       beta=0.9, lr=0.1, k=4, mode=ref.MODE_DEMO, sign=True)[0]
              for lo, hi in (shard_range(n, r, world) for r in range(world))]
    assert np.abs(np.concatenate(pieces) - th_full).max() <= 1e-15
