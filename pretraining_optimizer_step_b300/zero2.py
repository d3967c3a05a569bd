"""ZeRO-2-style sharded Muon step over torch.distributed ranks, with its three
phases overlapped.

The apidog.com page (section "2. Pengoptimal Muon", paragraph "Pelatihan
Terdistribusi") describes the multi-GPU optimizer as three asynchronous
phases: reduce-scatter the gradients so that each rank holds the summed
gradients of the matrices it owns, compute the updates (each rank for its own
matrices) while the weights' all-gather is already under way, and gather the
updated weights on every rank.  This module is that data-parallel plumbing
around the library: ownership comes from muon_partition (C; largest matrix
first to the least-loaded rank), the collectives are torch.distributed's (NCCL
on GPUs), and the update of the owned matrices is muon_step (or any callable
with its signature, e.g. a CPU reference in tests).

Buckets.  The matrices are split, in index order, into at most `buckets`
groups of about equal size (a group is closed once it reaches its share).  Each bucket has a flat gradient buffer of `world` equal
shards (shard r holds the matrices of the bucket that rank r owns, each at a
fixed offset) and a flat weight buffer of the same layout.  A step posts the
reduce-scatter of bucket 0 and 1, then for every bucket b: waits for its
reduce-scatter, averages, runs the update of the owned matrices of b, posts
the reduce-scatter of bucket b + 2 and the all-gather of bucket b.  With NCCL
the waits only order the compute stream after the collective, so bucket b's
update overlaps the reduce-scatter of the next buckets and the all-gather of
the previous one; the host never blocks until the end of the step.

No copies of the weights.  Every weight tensor is re-pointed (``Tensor.set_``)
at its place in its bucket's weight buffer, so the owner's update writes its
shard in place and the all-gather (in place: each rank's input is its own shard
of the output) delivers the other ranks' matrices straight into the weights.
Gradients are copied into the bucket buffers by ``step(grads)``; a caller that
writes them there itself (``grad_view(i)``) calls ``step()`` without copies.
Momentum is kept only by owners (the sharded optimizer state).
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence

import torch

from . import muon_partition, muon_step


class _Bucket:
    def __init__(self, index: List[int], sizes: Sequence[int], owner: Sequence[int], world: int, dtype, dev):
        self.index = index
        self.offset = {}
        fill = [0] * world
        for i in index:
            self.offset[i] = fill[owner[i]]
            fill[owner[i]] += sizes[i]
        self.shard_len = max(max(fill), 1)
        self.grads = torch.zeros(world * self.shard_len, dtype=dtype, device=dev)
        self.mine = torch.zeros(self.shard_len, dtype=dtype, device=dev)
        self.weights = torch.zeros(world * self.shard_len, dtype=dtype, device=dev)


class ShardedMuon:
    """Sharded Muon steps for one process group.

    params: this rank's full list of weight matrices (same shapes and values on
    every rank).  Each is re-pointed at its place in a flat bucket buffer (its
    values are kept), so references to the tensors stay valid and always hold
    the current weights.  compute(params, grads, moms, **hyper) updates the owned
    matrices of one bucket; the default runs muon_step on `stream` (the current
    CUDA stream if None).  buckets: at most how many groups the matrices are
    split into (more buckets overlap more, but each update launch then holds
    fewer matrices)."""

    def __init__(self, params: Sequence[torch.Tensor], group=None, compute: Optional[Callable] = None,
                 stream=None, buckets: int = 2):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.params = list(params)
        if not self.params:
            raise ValueError("no parameters")
        self.shapes = [tuple(p.shape) for p in self.params]
        self.owner = muon_partition(self.shapes, self.world)
        self.owned = [i for i, r in enumerate(self.owner) if r == self.rank]
        sizes = [p.numel() for p in self.params]
        dev, dtype = self.params[0].device, self.params[0].dtype
        # buckets: consecutive matrices, cut at about equal element counts
        nb = max(1, min(int(buckets), len(self.params)))
        total = sum(sizes)
        cuts, acc, b = [[]], 0, 0
        for i, n in enumerate(sizes):
            if b < nb - 1 and acc >= total * (b + 1) / nb and cuts[-1]:
                cuts.append([])
                b += 1
            cuts[-1].append(i)
            acc += n
        self.buckets = [_Bucket(ix, sizes, self.owner, self.world, dtype, dev) for ix in cuts]
        self.bucket_of = {}
        for k, bk in enumerate(self.buckets):
            for i in bk.index:
                self.bucket_of[i] = k
                # the weight tensor now lives in the bucket's weight buffer (value kept)
                view = self._slot(bk.weights, bk, i)
                with torch.no_grad():
                    view.copy_(self.params[i])
                    self.params[i].set_(view)
        self.momentum = {i: torch.zeros_like(self.params[i]) for i in self.owned}
        self.stream = stream
        self.compute = compute if compute is not None else self._gpu_compute

    def _slot(self, flat: torch.Tensor, bk: _Bucket, i: int) -> torch.Tensor:
        base = self.owner[i] * bk.shard_len + bk.offset[i]
        return flat[base:base + self.params[i].numel()].view(self.shapes[i])

    def grad_view(self, i: int) -> torch.Tensor:
        """Where step() reads matrix i's local gradient from (write it there to skip the copy)."""
        bk = self.buckets[self.bucket_of[i]]
        return self._slot(bk.grads, bk, i)

    def _gpu_compute(self, params, grads, moms, **hyper):
        stream = self.stream if self.stream is not None else torch.cuda.current_stream()
        muon_step(params, grads, moms, stream=stream, **hyper)

    def _post_reduce_scatter(self, bk: _Bucket):
        return self.dist.reduce_scatter_tensor(bk.mine, bk.grads, op=self.dist.ReduceOp.SUM, group=self.group,
                                               async_op=True)

    def step(self, grads: Optional[Sequence[torch.Tensor]] = None, **hyper) -> None:
        """One sharded step with this rank's local gradients (averaged over the group)."""
        if grads is not None:
            for i, g in enumerate(grads):
                self.grad_view(i).copy_(g)
        nb = len(self.buckets)
        rs = [None] * nb
        ag = []
        for b in range(min(2, nb)):
            rs[b] = self._post_reduce_scatter(self.buckets[b])
        for b, bk in enumerate(self.buckets):
            rs[b].wait()
            bk.mine.mul_(1.0 / self.world)
            own = [i for i in bk.index if self.owner[i] == self.rank]
            if own:
                own_g = [bk.mine[bk.offset[i]:bk.offset[i] + self.params[i].numel()].view(self.shapes[i])
                         for i in own]
                self.compute([self.params[i] for i in own], own_g, [self.momentum[i] for i in own], **hyper)
            if b + 2 < nb:
                rs[b + 2] = self._post_reduce_scatter(self.buckets[b + 2])
            # in place: this rank's input is its own shard of the weight buffer
            shard = bk.weights[self.rank * bk.shard_len:(self.rank + 1) * bk.shard_len]
            ag.append(self.dist.all_gather_into_tensor(bk.weights, shard, group=self.group, async_op=True))
        for w in ag:
            w.wait()
