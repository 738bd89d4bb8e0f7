"""Keys of one sequence sharded over ranks ("context" sharding), merged through the LSE.

Every rank holds the same queries and one contiguous range of the sequence's keys
and values. Each computes its shard's partial result on its own GPU
(``fa_fwd_kv_partial``: fp32 O normalised over the shard's keys, and the shard's
LSE, with the full sequence's causal diagonal); the partials are sent to the rank
that owns the output with a plain ``torch.distributed.gather`` (NCCL between GPUs:
every buffer a collective touches is this rank's own memory, and no kernel of this
library ever reads another device's memory); that rank merges them with
``lse_combine``:

    LSE = ln sum_r exp(LSE_r),   O = sum_r exp(LSE_r - LSE) O_r

("FlashAttention：一次前向计算", the two-round example: the results over two key
blocks are brought to one reference and divided once by the total denominator;
"Flash Attention 4", section "重缩放与结果写回": each part's LSE.)

The exchange moves 4·N_q·H·(d + 1) bytes per rank and batch entry, once per call;
this is the only collective of the path. The merge result equals the attention of
the queries over all keys (tests: shards computed one after another on one GPU and
merged, against the oracle over the whole sequence; the gather itself on CPU ranks
over gloo).
"""
from __future__ import annotations

from . import fa_fwd_kv_partial, lse_combine


def shard_range(n_kv_total: int, rank: int, world: int) -> tuple[int, int]:
    """Keys [lo, hi) of rank `rank` when n_kv_total keys are cut into `world` contiguous
    ranges whose sizes differ by at most one key."""
    if world < 1 or not 0 <= rank < world or n_kv_total < world:
        raise ValueError("need 0 <= rank < world <= n_kv_total")
    base, extra = divmod(n_kv_total, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def gather_partials(o_part, lse_part, dst: int = 0, group=None):
    """Send this rank's partial result to rank `dst`. On `dst` returns the partials of
    all ranks stacked in rank order, (o_parts [P, B, N_q, H, d], lse_parts [P, B, H, N_q]);
    on the other ranks returns (None, None). Tensors stay on their own device: CUDA
    tensors with the NCCL backend, CPU tensors with gloo."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    o_part = o_part.contiguous()
    lse_part = lse_part.contiguous()
    if rank == dst:
        o_parts = torch.empty((world,) + tuple(o_part.shape), dtype=o_part.dtype, device=o_part.device)
        lse_parts = torch.empty((world,) + tuple(lse_part.shape), dtype=lse_part.dtype, device=lse_part.device)
        dist.gather(o_part, gather_list=list(o_parts.unbind(0)), dst=dst, group=group)
        dist.gather(lse_part, gather_list=list(lse_parts.unbind(0)), dst=dst, group=group)
        return o_parts, lse_parts
    dist.gather(o_part, dst=dst, group=group)
    dist.gather(lse_part, dst=dst, group=group)
    return None, None


def fa_fwd_context_sharded(q, k_shard, v_shard, kv_offset: int, n_kv_total: int, *, dst: int = 0, group=None,
                           scale: float | None = None, causal: bool = False, dtype=None, stream=None):
    """Attention of q [B, N_q, H, d] over a sequence of n_kv_total keys of which this rank
    holds k_shard, v_shard [B, N_kv_shard, H_kv, d] = keys [kv_offset, kv_offset +
    N_kv_shard). Collective over `group`: every rank calls it with its own shard (the
    shards must cover the keys without overlap). Returns (o [B, N_q, H, d], lse
    [B, H, N_q]) on rank `dst`, (None, None) on the others."""
    import torch.distributed as dist
    o_part, lse_part = fa_fwd_kv_partial(q, k_shard, v_shard, kv_offset, n_kv_total, scale=scale, causal=causal,
                                         stream=stream)
    o_parts, lse_parts = gather_partials(o_part, lse_part, dst=dst, group=group)
    if dist.get_rank(group) != dst:
        return None, None
    return lse_combine(o_parts, lse_parts, dtype=dtype or q.dtype, stream=stream)
