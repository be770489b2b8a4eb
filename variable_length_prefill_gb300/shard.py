"""Head partition for running one attention call on several GPUs.

Every head of the operation is independent (each head's output rows depend
only on that head's q, k and v slices), so G processes, one per GPU, each
holding the packed tensors, split the heads between them and compute their
share in place with attn_varlen_fwd_heads: no exchange on the data path.
"""
from __future__ import annotations


def head_shard(num_heads: int, rank: int, world: int) -> tuple[int, int]:
    """(head_begin, head_count) of ``rank`` among ``world`` processes.

    Contiguous blocks in rank order; when ``world`` does not divide
    ``num_heads`` the first ``num_heads % world`` ranks take one head more.
    A rank beyond ``num_heads`` gets an empty range.
    """
    if num_heads < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad shard request: num_heads={num_heads} rank={rank} world={world}")
    base, extra = divmod(num_heads, world)
    count = base + (1 if rank < extra else 0)
    begin = rank * base + min(rank, extra)
    return begin, count
