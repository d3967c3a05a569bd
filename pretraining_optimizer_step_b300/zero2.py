"""ZeRO-2-style sharded Muon step over torch.distributed ranks.

The apidog.com page (section "2. Pengoptimal Muon", paragraph "Pelatihan
Terdistribusi") describes the multi-GPU optimizer as three asynchronous
phases: reduce-scatter the gradients, compute the updates (each rank for the
matrices it owns) while the weights' all-gather is launched, then copy the
gathered weights back.  This module is that data-parallel plumbing around the
library: the ownership comes from muon_partition (C), the collectives are
torch.distributed's (NCCL on GPUs), and the update of the owned matrices is
muon_step (or any callable with its signature, e.g. a CPU reference in tests).

Layout: every rank packs the gradients into one flat buffer of `world` shards
of equal length; shard r holds, in index order, the flattened matrices rank r
owns (padded to the longest shard).  One reduce_scatter_tensor leaves each
rank the summed gradients of its matrices, which are averaged; each rank keeps
momentum only for the matrices it owns (the sharded optimizer state); after the
update its weights go into its shard of a second flat buffer and one
all_gather_into_tensor gives every rank every matrix.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence

import torch

from . import muon_partition, muon_step


class ShardedMuon:
    """Sharded Muon steps for one process group.

    params: this rank's full list of weight matrices (same shapes on every rank,
    updated in place).  compute(params, grads, moms, **hyper) updates the owned
    matrices; the default runs muon_step on `stream`."""

    def __init__(self, params: Sequence[torch.Tensor], group=None, compute: Optional[Callable] = None,
                 stream=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.params = list(params)
        self.shapes = [tuple(p.shape) for p in self.params]
        self.owner = muon_partition(self.shapes, self.world)
        self.owned = [i for i, r in enumerate(self.owner) if r == self.rank]
        sizes = [p.numel() for p in self.params]
        self.shard_len = max(sum(sizes[i] for i, r in enumerate(self.owner) if r == k) for k in range(self.world))
        self.shard_len = max(self.shard_len, 1)
        # offset of every matrix inside its owner's shard
        self.offset = [0] * len(sizes)
        fill = [0] * self.world
        for i, r in enumerate(self.owner):
            self.offset[i] = fill[r]
            fill[r] += sizes[i]
        dev = self.params[0].device
        self.momentum = {i: torch.zeros_like(self.params[i]) for i in self.owned}
        self.send = torch.zeros(self.world * self.shard_len, dtype=torch.float32, device=dev)
        self.mine = torch.zeros(self.shard_len, dtype=torch.float32, device=dev)
        self.gathered = torch.zeros(self.world * self.shard_len, dtype=torch.float32, device=dev)
        self.stream = stream
        self.compute = compute if compute is not None else self._gpu_compute

    def _gpu_compute(self, params, grads, moms, **hyper):
        muon_step(params, grads, moms, stream=self.stream, **hyper)

    def _view(self, flat: torch.Tensor, i: int) -> torch.Tensor:
        base = self.owner[i] * self.shard_len + self.offset[i]
        return flat[base:base + self.params[i].numel()].view(self.shapes[i])

    def step(self, grads: Sequence[torch.Tensor], **hyper) -> None:
        """One sharded step with this rank's local gradients (averaged over the group)."""
        dist = self.dist
        # phase 1: reduce-scatter of the gradient shards
        for i, g in enumerate(grads):
            self._view(self.send, i).copy_(g)
        work = dist.reduce_scatter_tensor(self.mine, self.send, op=dist.ReduceOp.SUM, group=self.group,
                                          async_op=True)
        work.wait()
        self.mine.mul_(1.0 / self.world)
        # phase 2: update the owned matrices, then publish them
        if self.owned:
            own_g = [self.mine[self.offset[i]:self.offset[i] + self.params[i].numel()].view(self.shapes[i])
                     for i in self.owned]
            self.compute([self.params[i] for i in self.owned], own_g, [self.momentum[i] for i in self.owned],
                         **hyper)
        for i in self.owned:
            self.mine[self.offset[i]:self.offset[i] + self.params[i].numel()].copy_(self.params[i].reshape(-1))
        work = dist.all_gather_into_tensor(self.gathered, self.mine, group=self.group, async_op=True)
        # phase 3: copy the gathered weights back
        work.wait()
        for i, p in enumerate(self.params):
            if self.owner[i] != self.rank:
                p.copy_(self._view(self.gathered, i))
