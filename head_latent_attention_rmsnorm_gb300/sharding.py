"""How the path partitions across ranks (host logic only, no arithmetic of the method).

LAGA's sequence-parallel rank owns a contiguous block of query positions over the
full gathered latent (LAGA, "What carries the argument": all-gather the latent,
rebuild K/V locally); the Ulysses-style view owns a block of heads over all
positions (the paper's section 3.3 "H_r slice"); Helix's KV parallelism owns a block
of the key splits of a decode ("What carries the argument"); TPLA's tensor-parallel
rank owns an equal shard of the latent dims with every head (TPLA, "The reading").  On
one GPU these are simulated by the calls' q_offset / head range / split / shard
arguments; under torchrun each rank takes its block, and the results concatenate (or,
for key splits, merge by the log-sum-exp rescale; for latent shards, add up: the
all-reduce).
"""
from __future__ import annotations


def block(n: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous block [begin, begin + count) of n items owned by `rank` of `world`."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(n, world)
    begin = rank * base + min(rank, extra)
    return begin, base + (1 if rank < extra else 0)


def query_shard(seq_len: int, world: int, rank: int) -> tuple[int, int]:
    """(q_offset, s_q) of a sequence-parallel rank."""
    return block(seq_len, world, rank)


def head_shard(n_heads: int, world: int, rank: int) -> tuple[int, int]:
    """(head_begin, head_count) of a head-parallel rank."""
    return block(n_heads, world, rank)


def latent_shard(d_kv: int, world: int, rank: int) -> tuple[int, int]:
    """(first latent dim, dims) of a TPLA rank: equal shards, so d_kv must divide."""
    if d_kv % world:
        raise ValueError("the latent dims must split evenly across the ranks")
    return block(d_kv, world, rank)


def split_shard(n_splits: int, world: int, rank: int) -> tuple[int, int]:
    """(first split, number of splits) of a KV-parallel decode rank."""
    return block(n_splits, world, rank)
