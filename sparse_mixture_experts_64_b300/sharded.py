"""Token-sharded routing: the exchange between the two phases of the sharded router.

One batch is split over the ranks of a process group in token order (rank 0 holds
the first tokens). The capacity rule is global ("Mixture of Experts (MoE)"
glossary, capacity-factor paragraph; GShard top-2 in its sparse-MoE list): the first
C selections of each expert are kept, in slot-major priority over the whole batch
(every token's first choice in token order, then every second choice, ...). So
each rank

  1. routes its own tokens (moe_router_shard_stats): selections per expert and slot
     [N][k], softmax sums per expert [N];
  2. all-gathers those statistics and its token count (exchange below: the one
     collective of the sharded layer);
  3. places its selections at their global priorities and takes the capacity
     decisions (moe_router_shard_assign); the aux loss uses the global sums.

Dispatch, the experts and combine then run on each rank's own rows, as in the
unsharded layer. The sums across ranks are taken on the host in rank order, so
every rank gets the same bits.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist


def slot_bases(counts) -> np.ndarray:
    """counts [R][N][k]: selections of expert e in slot j on rank r. Returns
    [R][N][k]: the global priority of rank r's first selection of (e, j) = all
    ranks' selections of e in earlier slots + the selections of (e, j) on earlier
    ranks."""
    c = np.asarray(counts, dtype=np.int64)
    totals = c.sum(axis=0)                       # [N][k] over all ranks
    before_slot = np.cumsum(totals, axis=1) - totals
    before_rank = np.cumsum(c, axis=0) - c
    return before_slot[None, :, :] + before_rank


def global_capacity(T_global: int, N: int, capacity_factor) -> int:
    """C = ceil(T_global * cf / N) for cf = (num, den); 0 = no limit."""
    if capacity_factor is None:
        return 0
    num, den = capacity_factor
    return (T_global * num + N * den - 1) // (N * den)


def exchange(slot_counts: torch.Tensor, prob_sums: torch.Tensor, T_local: int, group=None):
    """All-gather of the phase-1 statistics over `group` (any backend; tensors on
    the device that backend serves). Returns, for the calling rank and on the device
    of slot_counts: slot_base int32 [N][k], global_routed int32 [N],
    global_prob_sums fp32 [N] (summed in rank order) and T_global (int)."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    dev = slot_counts.device
    cnt = [torch.empty_like(slot_counts) for _ in range(world)]
    dist.all_gather(cnt, slot_counts.contiguous(), group=group)
    ps = [torch.empty_like(prob_sums) for _ in range(world)]
    dist.all_gather(ps, prob_sums.contiguous(), group=group)
    tl = [torch.empty(1, dtype=torch.int64, device=dev) for _ in range(world)]
    dist.all_gather(tl, torch.tensor([int(T_local)], dtype=torch.int64, device=dev), group=group)
    counts = torch.stack(cnt).cpu().numpy()               # [R][N][k]
    base = slot_bases(counts)[rank]
    g_routed = counts.sum(axis=(0, 2))
    g_psum = np.zeros(counts.shape[1], np.float32)
    for p in ps:                                          # rank order
        g_psum = (g_psum + p.cpu().numpy().astype(np.float32)).astype(np.float32)
    T_global = int(sum(int(t.item()) for t in tl))
    to = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a), dtype=dt).to(dev)  # noqa: E731
    return to(base, torch.int32), to(g_routed, torch.int32), to(g_psum, torch.float32), T_global


def route_sharded(cfg, x, w_r, b_r, capacity_factor, ws, group=None, stream=None) -> dict:
    """Phase 1, exchange, phase 2 for this rank's tokens x [T_local][d] on its GPU.
    cfg: this rank's shard (T = T_local, no capacity of its own). Returns the
    routing outputs of this rank (as moe_router_topk) plus the global capacity,
    the global token count and the global aux loss."""
    from . import (moe_max_rows, moe_router_shard_assign, moe_router_shard_stats)
    T, k, N = cfg.T, cfg.k, cfg.N
    dev = x.device
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(topk_idx=torch.empty((T, k), **i32), topk_gate=torch.empty((T, k), device=dev),
               slot_counts=torch.empty((N, k), **i32), prob_sums=torch.empty(N, device=dev),
               counts_kept=torch.empty(N, **i32), expert_offsets=torch.empty(N + 1, **i32),
               slot_row=torch.empty((T, k), **i32), perm_token=torch.empty(moe_max_rows(cfg), **i32),
               aux=torch.empty(2, device=dev))
    moe_router_shard_stats(cfg, x, w_r, b_r, out["topk_idx"], out["topk_gate"], out["slot_counts"],
                           out["prob_sums"], ws, stream)
    base, g_routed, g_psum, T_global = exchange(out["slot_counts"], out["prob_sums"], T, group)
    C = global_capacity(T_global, N, capacity_factor)
    moe_router_shard_assign(cfg, out["topk_idx"], base, C, g_routed, g_psum, T_global,
                            out["counts_kept"], out["expert_offsets"], out["slot_row"],
                            out["perm_token"], out["aux"], ws, stream)
    out.update(slot_base=base, capacity=C, T_global=T_global, counts_routed_global=g_routed)
    return out
