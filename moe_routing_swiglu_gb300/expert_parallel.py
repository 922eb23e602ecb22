"""Expert-parallel sharding of the local MoE chain: the exchange plan.

Each rank routes and dispatches its own tokens with the local chain
(moe_route, moe_dispatch). Experts are split into contiguous blocks over the
ranks (``expert_range``), so the dispatched layout, which is sorted by
expert, already holds the rows bound for each rank as one contiguous slice:
x_dispatched itself is the send buffer of the row exchange. One step:

  1. counts exchange: rank s sends rank d the per-expert row counts of d's
     experts (an all-to-all of E counts in total);
  2. rows exchange: an all-to-all-v of dispatched rows; rank d receives, from
     every source s in turn, s's rows of d's experts in s's dispatched order;
  3. the received rows are put in expert-major order (within an expert:
     by source rank, then in the source's order) and the owned experts run as
     one grouped GEMM over them (moe_experts_forward_dispatched with a handle
     on the owned experts' weights, or any function of the same contract);
  4. the expert outputs go back by the inverse permutation and the reverse
     all-to-all-v, landing in each source's own dispatched order;
  5. each source combines locally (moe_combine: slot order, FP32), so the
     result does not depend on the rank count or the arrival order.

The pages describe the local chain only; this sharding is the expert-parallel
extension of its dispatch and combine contract (ruDNN user guide, section 5
"Expert weights and dispatch" and section 6 "Call MoE"). The plan and the
exchanges here use torch.distributed collectives (NCCL on GPUs, gloo on the
CPU); on CUDA tensors the two reorders (steps 3 and 4) run the library's
row-move kernel (moe_permute_rows), and the experts and the combine are the
library's kernels too. On CPU tensors (the plan's gloo tests) the reorders
are torch indexing.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable

import torch
import torch.distributed as dist


def _moe():
    """The library's Python binding (imported on first use: the plan itself
    needs no GPU)."""
    import moe_routing_swiglu_gb300 as moe

    return moe


def expert_range(E: int, world: int, rank: int) -> tuple[int, int]:
    """Experts [lo, hi) owned by ``rank``: contiguous blocks, the first
    E % world ranks holding one expert more than the others."""
    if not (1 <= world and 0 <= rank < world and E >= 1):
        raise ValueError("need E >= 1 and 0 <= rank < world")
    base, extra = divmod(E, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


@dataclass
class EpPlan:
    """The exchange plan of one step on one rank."""

    send_splits: list[int]        # rows sent to each rank (this rank's rows of that rank's experts)
    recv_splits: list[int]        # rows received from each rank
    recv_counts: torch.Tensor     # [world, n_local] rows per (source rank, owned expert), int64
    local_offsets: torch.Tensor   # [n_local + 1] int64: expert-major layout of the received rows
    perm: torch.Tensor            # [n_recv] int64: received row i sits at local row perm[i]
    experts: tuple[int, int]      # owned experts [lo, hi)


def ep_plan(counts: torch.Tensor, E: int, group=None) -> EpPlan:
    """Exchange the per-expert counts (this rank's ``counts`` [E], from its
    dispatch) and derive the send/receive splits and the permutation of the
    received rows into expert-major order."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    counts = counts.reshape(-1).to(torch.int64)
    if counts.numel() != E:
        raise ValueError("counts must hold one entry per expert")
    ranges = [expert_range(E, world, r) for r in range(world)]
    lo, hi = ranges[rank]
    n_local = hi - lo
    send_splits = [int(counts[a:b].sum()) for a, b in ranges]
    # Counts exchange: rank d receives [world, n_local(d)] counts.
    cdev = counts.device
    recv = torch.empty(world * n_local, dtype=torch.int64, device=cdev)
    dist.all_to_all_single(recv, counts.contiguous(), [n_local] * world, [b - a for a, b in ranges], group=group)
    recv_counts = recv.view(world, n_local).cpu()
    recv_splits = [int(x) for x in recv_counts.sum(dim=1)]
    local_counts = recv_counts.sum(dim=0)
    local_offsets = torch.zeros(n_local + 1, dtype=torch.int64)
    local_offsets[1:] = torch.cumsum(local_counts, dim=0)
    # Received row order: source s, then expert e, then the source's order.
    # Local order: expert e, then source s, then the source's order.
    seg_base = torch.cumsum(recv_counts, dim=0) - recv_counts        # rows of (s', e) for s' < s
    perm_parts = []
    for s in range(world):
        for e in range(n_local):
            n = int(recv_counts[s, e])
            if n:
                start = int(local_offsets[e] + seg_base[s, e])
                perm_parts.append(torch.arange(start, start + n, dtype=torch.int64))
    perm = torch.cat(perm_parts) if perm_parts else torch.empty(0, dtype=torch.int64)
    return EpPlan(send_splits, recv_splits, recv_counts, local_offsets, perm.to(cdev), (lo, hi))


def ep_dispatch_rows(x_dispatched: torch.Tensor, plan: EpPlan, group=None) -> torch.Tensor:
    """Send each rank its slice of x_dispatched [rows, H] and return the
    received rows in expert-major order [n_recv, H]."""
    if x_dispatched.shape[0] != sum(plan.send_splits):
        raise ValueError("x_dispatched must hold exactly the dispatched rows")
    H = x_dispatched.shape[1]
    recv = x_dispatched.new_empty(sum(plan.recv_splits), H)
    dist.all_to_all_single(recv, x_dispatched.contiguous(), plan.recv_splits, plan.send_splits, group=group)
    if recv.is_cuda:  # the library's row-move kernel
        return _moe().moe_permute_rows(recv, plan.perm, scatter=True)
    local = torch.empty_like(recv)
    local[plan.perm] = recv
    return local


def ep_return_rows(y_local: torch.Tensor, plan: EpPlan, group=None) -> torch.Tensor:
    """Send the owned experts' outputs [n_recv, H] (expert-major) back to
    their sources; returns this rank's expert outputs in its own dispatched
    order [rows, H]."""
    if y_local.is_cuda:  # the library's row-move kernel
        back = _moe().moe_permute_rows(y_local.contiguous(), plan.perm)
    else:
        back = y_local[plan.perm].contiguous()
    out = y_local.new_empty(sum(plan.send_splits), y_local.shape[1])
    dist.all_to_all_single(out, back, plan.send_splits, plan.recv_splits, group=group)
    return out


def ep_experts_forward(x_dispatched: torch.Tensor, counts: torch.Tensor, E: int,
                       experts_fn: Callable[[torch.Tensor, torch.Tensor, tuple[int, int]], torch.Tensor],
                       group=None) -> torch.Tensor:
    """Steps 1-4: the expert outputs of this rank's dispatched rows, in its
    dispatched order, computed by the ranks that own the experts.
    ``experts_fn(x_local, local_offsets, (lo, hi))`` runs the owned experts
    lo..hi-1 on the expert-major rows (offsets relative to expert lo)."""
    plan = ep_plan(counts, E, group)
    x_local = ep_dispatch_rows(x_dispatched, plan, group)
    y_local = experts_fn(x_local, plan.local_offsets, plan.experts)
    if y_local.shape[0] != x_local.shape[0]:
        raise ValueError("experts_fn must return one row per received row")
    return ep_return_rows(y_local, plan, group)
