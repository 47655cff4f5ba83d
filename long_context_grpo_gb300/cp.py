"""Context-parallel prompt sharding across ranks (LongStraw review, section 3-2 (2)
"Physical page ownership": each rank holds a slice of the prompt K/V pages and the local
attention results are combined by a cross-rank log-sum-exp and output merge).

Rank r owns prompt rows shard_bounds(P, world)[r] .. [r+1]-1 in its own prefix handle; the
last rank also owns the response's causal suffix.  Per response:
  forward   every rank computes its partial (o_r, lse_r); exchange_partials all-gathers
            them in rank order; the merge combines them (the same merged o, lse on every
            rank);
  backward  every rank runs its shard backward with the merged o, lse, which adds the
            exact gradient of its own keys into its accumulators and returns its part of
            dq; reduce_dq sums the parts in fp32 on every rank.
All arithmetic runs in the CUDA library (ls_attn_merge, ls_bf16_to_f32, ls_f32_to_bf16);
torch.distributed only moves the tensors.  The exchange helpers take tensors on any device
(gloo on CPU, NCCL on GPU) and an `ops` object with the merge and the two conversions, the
library's by default.
"""
from __future__ import annotations

import torch


class LibraryOps:
    """The CUDA library's partial-attention merge and the fp32 widening / bf16 rounding
    around the cross-rank dq sum."""

    @staticmethod
    def merge(o_parts, lse_parts):
        from . import _lib as ls
        return ls.attn_merge(o_parts, lse_parts)

    @staticmethod
    def to_f32(x):
        from . import _lib as ls
        return ls.bf16_to_f32(x)

    @staticmethod
    def to_bf16(x):
        from . import _lib as ls
        return ls.f32_to_bf16(x)


def shard_bounds(P: int, world: int) -> list:
    """Contiguous prompt slices, one per rank, sizes differing by at most one row."""
    if world < 1 or P < world:
        raise ValueError("need 1 <= world <= P")
    return [(P * r) // world for r in range(world + 1)]


def exchange_partials(o_r, lse_r, group=None):
    """All-gather the ranks' partial outputs and log-sum-exps; lists in rank order."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    o_all = [torch.empty_like(o_r) for _ in range(world)]
    lse_all = [torch.empty_like(lse_r) for _ in range(world)]
    dist.all_gather(o_all, o_r.contiguous(), group=group)
    dist.all_gather(lse_all, lse_r.contiguous(), group=group)
    return o_all, lse_all


def reduce_dq(dq_r, group=None, ops=LibraryOps):
    """Sum of the ranks' dq parts: widened to fp32, summed by the collective, rounded back
    to dq_r's dtype."""
    import torch.distributed as dist
    acc = ops.to_f32(dq_r)
    dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    return ops.to_bf16(acc)


def replay_response(pre, rank: int, world: int, q, k_suffix, v_suffix, d_out, group=None,
                    ops=LibraryOps):
    """One response's forward and backward on this rank's prompt shard (`pre`, a Prefix
    over the rank's rows).  Returns (o, lse, dq) -- identical on every rank -- and, on the
    last rank, the suffix key gradients (dk_suffix, dv_suffix); None elsewhere."""
    owner = rank == world - 1
    if owner:
        o_r, lse_r = pre.fwd(q, k_suffix, v_suffix)
    else:
        o_r, lse_r = pre.fwd_prompt_only(q)
    o_all, lse_all = exchange_partials(o_r, lse_r, group)
    o, lse = ops.merge(o_all, lse_all)
    if owner:
        dq_r, dks, dvs = pre.bwd(q, k_suffix, v_suffix, o, lse, d_out)
    else:
        dq_r = pre.bwd_prompt_only(q, o, lse, d_out)
        dks = dvs = None
    return o, lse, reduce_dq(dq_r, group, ops), dks, dvs
