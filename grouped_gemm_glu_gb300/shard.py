"""Expert-parallel sharding of the layer across ranks (one GPU per rank).

Each rank owns a contiguous range of E local experts out of n_experts and
routes the same token batch; assignments to other ranks' experts are dropped
by its routing (row_of = -1).  There is no collective on the data path: the
all-to-all that would move tokens between ranks belongs to the
communication stack, so ranks are independent shards (weak scaling)."""
from __future__ import annotations


def shard_expert_begin(rank: int, E: int, n_experts: int) -> int:
    """First global expert id owned by `rank` when each rank holds E experts
    (ranks beyond n_experts / E wrap around and repeat a shard)."""
    if E <= 0 or n_experts <= 0 or E > n_experts:
        raise ValueError("need 0 < E <= n_experts")
    return (rank * E) % n_experts


def shards_cover(world: int, E: int, n_experts: int) -> bool:
    """True when the ranks' expert ranges tile [0, n_experts) exactly once."""
    begins = sorted(shard_expert_begin(r, E, n_experts) for r in range(world))
    return world * E == n_experts and begins == list(range(0, n_experts, E))
