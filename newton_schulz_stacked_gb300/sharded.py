"""The Muon step sharded over data-parallel ranks by bank slot.

Each rank holds every bank's weights in full (the model needs them) and, for the
slots it owns, the optimizer state: the fp32 momentum buffer, the uint16 low
mantissa and, with NorMuon, the per-row second moment.  One step is three passes
("Muon Custom Sizing" write-up, record 2025-09-23, section 4; the mixed-precision
form in the "GPT-2 Medium track record 7" write-up, section 4.2):

  1. the ranks' bf16 gradients are reduced and scattered by slot, averaged, so
     that each rank gets the mean gradient of the slots it owns;
  2. each rank runs the whole Muon step (momentum, normalisation, Newton-Schulz,
     update) on its own slots, through the library's muon_multi_step;
  3. the updated bf16 weights of every rank's slots are gathered to all ranks.

Only bf16 weights and gradients cross ranks: momentum, mantissa and row state
never leave their owner.  A bank's leading dimension is padded to a multiple of
the world size; the padding slots are dead (zero gradient, zero weight and
state), so their update is exactly zero and they stay zero.

The collectives are torch.distributed calls on the caller's process group, on
plain device memory (no multicast): reduce_scatter_tensor with AVG where the
backend has it (NCCL), else SUM followed by a division by the world size
(the gloo backend of the CPU tests).  The local step is injectable so that the
data movement can be tested on CPU ranks; by default it is the library's
CUDA path, which raises without the built library.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional, Sequence

import torch
import torch.distributed as dist


@dataclass(frozen=True)
class ShardPlan:
    """Ownership of a bank's slots: `per` consecutive slots per rank, the bank padded to
    `padded` = per * world slots; rank r owns slots [r * per, (r + 1) * per)."""
    batch: int
    world: int

    @property
    def per(self) -> int:
        return -(-self.batch // self.world)

    @property
    def padded(self) -> int:
        return self.per * self.world

    def owned(self, rank: int):
        """The slot range [lo, hi) of `rank`, including any padding slots it holds."""
        if not 0 <= rank < self.world:
            raise ValueError(f"rank {rank} outside a world of {self.world}")
        return rank * self.per, (rank + 1) * self.per

    def live(self, rank: int):
        """The owned slots that belong to the bank (padding excluded): [lo, hi), empty (hi == lo)
        for a rank that owns only padding."""
        lo, hi = self.owned(rank)
        return lo, max(lo, min(hi, self.batch))


class ShardedBank:
    """One bank of a sharded step, as held by one rank.

    weights   : bf16 bits (int16 or bfloat16) [plan.padded, rows, cols], every rank's copy of the
                whole bank; rows past `batch` are padding and must be zero
    momentum  : fp32 [plan.per, rows, cols], this rank's slots
    mantissa  : uint16 bits (int16) [plan.per, rows, cols], this rank's slots
    row_state : fp32 [plan.per, rows] with NorMuon, else None
    """

    def __init__(self, plan: ShardPlan, rank: int, weights, momentum, mantissa, row_state=None):
        rows, cols = weights.shape[1:]
        if weights.shape[0] != plan.padded:
            raise ValueError(f"weights must hold {plan.padded} slots (padded), not {weights.shape[0]}")
        for name, t, shape in (("momentum", momentum, (plan.per, rows, cols)),
                               ("mantissa", mantissa, (plan.per, rows, cols))):
            if tuple(t.shape) != shape:
                raise ValueError(f"{name} must be {shape}, not {tuple(t.shape)}")
        if row_state is not None and tuple(row_state.shape) != (plan.per, rows):
            raise ValueError(f"row_state must be {(plan.per, rows)}")
        self.plan, self.rank = plan, rank
        self.weights, self.momentum, self.mantissa, self.row_state = weights, momentum, mantissa, row_state

    @property
    def shard(self):
        """This rank's slots of the weights (a view)."""
        lo, hi = self.plan.owned(self.rank)
        return self.weights[lo:hi]


def _reduce_scatter_mean(out: torch.Tensor, full: torch.Tensor, world: int, group) -> None:
    """out = the mean over ranks of this rank's slots of `full` (bf16 bits)."""
    bf_full = full.view(torch.bfloat16) if full.dtype == torch.int16 else full
    bf_out = out.view(torch.bfloat16) if out.dtype == torch.int16 else out
    if dist.get_backend(group) == "nccl":
        dist.reduce_scatter_tensor(bf_out, bf_full, op=dist.ReduceOp.AVG, group=group)
    else:
        dist.reduce_scatter_tensor(bf_out, bf_full, op=dist.ReduceOp.SUM, group=group)
        bf_out.div_(world)


def library_local_step(banks, grads, lr, wd, mu, normuon, beta2, ns_steps, workspace):
    """The default local step: the library's muon_multi_step on this rank's slots."""
    from . import BankState, muon_multi_step
    states = [BankState(b.shard, g, b.momentum, b.mantissa, b.row_state) for b, g in zip(banks, grads)]
    return muon_multi_step(states, lr, wd, mu, normuon=normuon, beta2=beta2, ns_steps=ns_steps, workspace=workspace)


def sharded_step(banks: Sequence[ShardedBank], grads: Sequence[torch.Tensor], lr: float, wd: float, mu: float,
                 normuon: bool = False, beta2: float = 0.95, ns_steps: int = 5, group=None,
                 local_step: Optional[Callable] = None, workspace=None):
    """One data-parallel Muon step over `banks`.

    grads[i] is this rank's bf16 gradient of bank i, [plan.padded, rows, cols] (padding slots
    zero).  After the call every rank's banks[i].weights holds the updated bank, and each rank's
    momentum, mantissa and row state are those of its slots.  Returns what the local step
    returns (the library's workspace by default)."""
    if len(banks) != len(grads) or not banks:
        raise ValueError("one gradient per bank, at least one bank")
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    for b, g in zip(banks, grads):
        if b.plan.world != world or b.rank != rank:
            raise ValueError("the banks' plans were made for another rank or world size")
        if tuple(g.shape) != tuple(b.weights.shape):
            raise ValueError(f"gradient shape {tuple(g.shape)} is not the padded bank's {tuple(b.weights.shape)}")
    # 1. mean gradient of this rank's slots
    shard_grads = []
    for b, g in zip(banks, grads):
        out = torch.empty_like(b.shard)
        _reduce_scatter_mean(out, g, world, group)
        shard_grads.append(out)
    # 2. the whole step on this rank's slots
    step = local_step or library_local_step
    ret = step(banks, shard_grads, lr, wd, mu, normuon, beta2, ns_steps, workspace)
    # 3. every rank's updated slots to every rank (the send buffer is a copy of this rank's slots,
    #    so the gather never reads a region it writes)
    for b in banks:
        send = b.shard.clone()
        full = b.weights.view(torch.bfloat16) if b.weights.dtype == torch.int16 else b.weights
        dist.all_gather_into_tensor(full, send.view(torch.bfloat16) if send.dtype == torch.int16 else send,
                                    group=group)
    return ret
