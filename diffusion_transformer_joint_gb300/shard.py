"""How the joint attention is split across ranks, one GPU per rank
("Diffusers 中 Flux2Transformer2DModel 全面解析", section 并行化支持).

Head parallel (the tensor-parallel plan: Q, K and V are projected column-wise,
so a rank owns a contiguous range of heads): every (batch, head) pair is an
independent unit, so a rank calls flux_joint_rope_attention_heads on its heads
and nothing moves between ranks inside the attention.

Sequence parallel (the context-parallel plan, which splits the sequence
dimension): a rank owns a contiguous range of tokens. Its queries need every
key and value, so the ranks all-gather K and V (the one exchange step), then
each calls flux_joint_rope_attention_rows on its query rows.

The split itself and the gather are host logic; the kernels are the
library's.
"""
from __future__ import annotations


def even_range(rank: int, world: int, n: int) -> tuple[int, int]:
    """(start, count) of rank's share of n items in contiguous blocks whose
    sizes differ by at most one (the first n % world ranks take one more)."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError(f"bad split: rank {rank} of {world}, {n} items")
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def head_range(rank: int, world: int, H: int) -> tuple[int, int]:
    """(h0, n_heads) of a head-parallel rank."""
    return even_range(rank, world, H)


def seq_range(rank: int, world: int, S: int) -> tuple[int, int]:
    """(q0, n_rows) of a sequence-parallel rank's tokens."""
    return even_range(rank, world, S)


def gather_sequence(x_local, S: int, dist, out=None, group=None):
    """All-gather the sequence shards [B, n_r, H, D] of every rank (rank r owns
    the rows seq_range(r, world, S)) into the full [B, S, H, D] tensor.

    Shards are padded to the longest one so that every rank sends the same
    number of bytes (NCCL's all-gather requires it). With B = 1 and S a
    multiple of the world size the shards land in place in ``out`` (one
    all-gather into the full tensor); otherwise they are gathered into a
    scratch list and copied into place."""
    import torch

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    B, n, H, D = x_local.shape
    if n != seq_range(rank, world, S)[1]:
        raise ValueError(f"rank {rank} holds {n} rows, its share of {S} is "
                         f"{seq_range(rank, world, S)[1]}")
    if out is None:
        out = x_local.new_empty((B, S, H, D))
    L = -(-S // world)
    if B == 1 and S % world == 0:
        dist.all_gather_into_tensor(out.view(world * L, H, D), x_local[0].contiguous(), group=group)
        return out
    buf = x_local.new_zeros((B, L, H, D))
    buf[:, :n] = x_local
    parts = [torch.empty_like(buf) for _ in range(world)]
    dist.all_gather(parts, buf, group=group)
    for r, p in enumerate(parts):
        q0, m = seq_range(r, world, S)
        out[:, q0:q0 + m] = p[:, :m]
    return out
