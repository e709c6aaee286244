"""Split-KV of one long sequence across GPUs.

Each rank holds a contiguous range of every sequence's cache blocks,
decodes it with ``mla_decode_blocks`` (one split-KV piece: ``o_lat`` and
``lse`` over those keys alone), and the pieces are gathered to one rank,
which merges them with ``mla_combine_pieces``.  The merge is the
log-sum-exp combine of the on-GPU split (the softmax over the union of the
ranges, "From Vanilla Transformers to Modern LLMs -- Part 3" 2.a, 3.f); the
gather moves ``B * Hq * H * (d_c * 2 + 4)`` bytes per rank, about 132 KB per
query slot at H = 128.  Data-parallel decoding of a batch (one replica per
GPU, sequences sharded) needs none of this.
"""

from __future__ import annotations

import torch
import torch.distributed as dist


def block_range(rank: int, world: int, n_blocks: int) -> tuple[int, int]:
    """Rank ``rank``'s contiguous share ``[first, end)`` of the logical blocks
    ``[0, n_blocks)``: near-equal, in rank order, empty shares at the end
    when there are fewer blocks than ranks."""
    if world < 1 or not 0 <= rank < world or n_blocks < 0:
        raise ValueError("need 0 <= rank < world and n_blocks >= 0")
    per = (n_blocks + world - 1) // world
    first = min(n_blocks, rank * per)
    return first, min(n_blocks, first + per)


def gather_pieces(o_lat: torch.Tensor, lse: torch.Tensor, dst: int = 0, group=None):
    """Gather every rank's piece to rank ``dst``.

    Returns ``(o_pieces [world, ...], lse_pieces [world, ...])`` stacked in
    rank order on ``dst`` (the layout ``mla_combine_pieces`` takes) and
    ``(None, None)`` elsewhere.  The tensors must be on the device the
    process group's backend works on (CUDA for NCCL, host for gloo).
    """
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if rank == dst:
        o_all = torch.empty((world,) + tuple(o_lat.shape), dtype=o_lat.dtype,
                            device=o_lat.device)
        lse_all = torch.empty((world,) + tuple(lse.shape), dtype=lse.dtype, device=lse.device)
        dist.gather(o_lat.contiguous(), list(o_all.unbind(0)), dst=dst, group=group)
        dist.gather(lse.contiguous(), list(lse_all.unbind(0)), dst=dst, group=group)
        return o_all, lse_all
    dist.gather(o_lat.contiguous(), None, dst=dst, group=group)
    dist.gather(lse.contiguous(), None, dst=dst, group=group)
    return None, None
