"""Context-parallel prompt sharding across ranks (LongStraw review, section 3-2 (2)
"Physical page ownership": each rank holds a slice of the prompt K/V pages and the local
attention results are combined by a cross-rank log-sum-exp and output merge).

Rank r owns prompt rows shard_bounds(P, world)[r] .. [r+1]-1 in its own prefix handle; the
last rank also owns the response's causal suffix.  Per response:
  forward   every rank computes its partial (o_r, lse_r); exchange_partials all-gathers
            them in rank order; ls_attn_merge combines them (the same merged o, lse on
            every rank);
  backward  every rank runs its shard backward with the merged o, lse, which adds the
            exact gradient of its own keys into its accumulators and returns its part of
            dq; reduce_dq sums the parts (fp32) on every rank.
The exchange helpers take tensors on any device (gloo on CPU, NCCL on GPU); the replay
driver needs the CUDA library.
"""
from __future__ import annotations

import torch


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


def reduce_dq(dq_r, group=None):
    """Sum of the ranks' dq parts, accumulated in fp32, returned in dq_r's dtype."""
    import torch.distributed as dist
    acc = dq_r.to(torch.float32)
    dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    return acc.to(dq_r.dtype)


def replay_response(pre, rank: int, world: int, q, k_suffix, v_suffix, d_out, group=None):
    """One response's forward and backward on this rank's prompt shard (`pre`, a Prefix
    over the rank's rows).  Returns (o, lse, dq) -- identical on every rank -- and, on the
    last rank, the suffix key gradients (dk_suffix, dv_suffix); None elsewhere."""
    from . import _lib as ls
    owner = rank == world - 1
    if owner:
        o_r, lse_r = pre.fwd(q, k_suffix, v_suffix)
    else:
        o_r, lse_r = pre.fwd_prompt_only(q)
    o_all, lse_all = exchange_partials(o_r, lse_r, group)
    o, lse = ls.attn_merge(o_all, lse_all)
    if owner:
        dq_r, dks, dvs = pre.bwd(q, k_suffix, v_suffix, o, lse, d_out)
    else:
        dq_r = pre.bwd_prompt_only(q, o, lse, d_out)
        dks = dvs = None
    return o, lse, reduce_dq(dq_r, group), dks, dvs
