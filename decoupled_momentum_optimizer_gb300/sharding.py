"""Host-side sharding of a flat parameter buffer across GPUs (one process per GPU).

FlexDeMo shards the model inside a node (the shard group S) and replicates each
shard across nodes (the replication group R): accelerator i of every node holds
the same shard ("DeToNATION: Decoupled Torch Network-Aware Training on
Interlinked Online Nodes", Paper-Notes AAAI 2026, method section, "1. FlexDeMo"
implementation notes).  Every chunk of the step is independent, so a shard is
any contiguous range of whole 32-element chunks and the per-shard step needs no
data exchange between the GPUs of one node.  The chunk index that feeds the
Random scheme's position hash is local to the shard; ``shard_seed`` gives each
shard its own index seed so that shards do not repeat one selection pattern.
"""

CHUNK = 32


def shard_range(n, rank, world):
    """[lo, hi) element range of shard ``rank`` of ``world`` over a flat buffer of n.

    Whole chunks only; the first (nc mod world) shards get one extra chunk.
    """
    if n % CHUNK:
        raise ValueError("n must be a multiple of the chunk size")
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    nc = n // CHUNK
    base, extra = divmod(nc, world)
    lo_c = rank * base + min(rank, extra)
    hi_c = lo_c + base + (1 if rank < extra else 0)
    return lo_c * CHUNK, hi_c * CHUNK


def shard_seed(seed, rank):
    """Index seed of shard ``rank`` (shared by that shard's replicas)."""
    return (seed + 0x9E3779B97F4A7C15 * (rank + 1)) & ((1 << 64) - 1)


def max_over_ranks(value, dist=None, device=None):
    """Largest ``value`` over the process group (the step time every rank waits for)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()
