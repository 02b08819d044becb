"""The LM head split by vocabulary across ranks: rank r holds the contiguous rows
[v_r, v_{r+1}) of W, every rank the whole batch (hidden rows, labels, the CSR support).
Pull request #4233 ("What changes": the ragged support is sharded and gathered with the
head across context-parallel ranks) is the setting; this module is the rank logic only.
Every step of the arithmetic runs in librlhead's kernels (the `LibraryOps` below); what is
here is the partition, the order of the collectives and which buffers they carry.

Forward, per rank, then two collectives:
  1. the labels' and support ids' local numbering (ids the rank does not own fall outside
     its columns);
  2. the rank's statistics over its columns, per token (m = max z, s = sum e^(z - m),
     u = sum e^(z - m)(z - m)), and the label / support logits it owns (0 elsewhere);
  3. all-gather of the statistics, in rank order; all-reduce (sum) of the owned logits,
     which routes every logit from its owner to all ranks;
  4. on every rank, the loss, log-probs, masks, metrics and saved state from the gathered
     statistics, combined as the single-GPU forward combines its vocabulary splits: the
     same bits on every rank.
Backward, per rank, then one collective:
  5. the rank's slice of the logit gradient (its columns: the dense part against the global
     logsumexp, the spikes at the ids it owns): dW for its rows, no exchange, and its part
     of dX;
  6. all-reduce (sum) of the dX parts.
Traffic per step: 3 N floats gathered from each rank, N + nnz floats and N H floats summed.

The ops and the exchange are passed in, so the same rank logic runs on GPUs (LibraryOps,
TorchExchange over NCCL) and in the CPU tests (an fp64 stand-in for the ops, gloo).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


def vocab_partition(V: int, world: int, align: int = 256):
    """[(begin, end)] for each rank: contiguous ranges covering [0, V), boundaries at
    multiples of `align` (the forward GEMM's column tile), tile counts as equal as they can
    be (the earlier ranks take one more tile when they do not divide evenly)."""
    if world < 1 or V < 1:
        raise ValueError("need V >= 1 and world >= 1")
    tiles = -(-V // align)
    if tiles < world:
        raise ValueError(f"{V} ids in tiles of {align} cannot be split over {world} ranks")
    per, extra = divmod(tiles, world)
    out, t = [], 0
    for r in range(world):
        n = per + (1 if r < extra else 0)
        out.append((min(V, t * align), min(V, (t + n) * align)))
        t += n
    return out


@dataclasses.dataclass
class Shard:
    rank: int
    world: int
    begin: int
    end: int

    @property
    def size(self) -> int:
        return self.end - self.begin


class TorchExchange:
    """The two collectives, over a torch.distributed process group."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group

    def all_gather(self, x: torch.Tensor) -> torch.Tensor:
        world = self.dist.get_world_size(self.group)
        out = torch.empty((world * x.shape[0],) + tuple(x.shape[1:]), dtype=x.dtype, device=x.device)
        self.dist.all_gather_into_tensor(out, x.contiguous(), group=self.group)
        return out.view((world,) + tuple(x.shape))

    def all_reduce_sum_(self, x: torch.Tensor) -> torch.Tensor:
        self.dist.all_reduce(x, op=self.dist.ReduceOp.SUM, group=self.group)
        return x


class LibraryOps:
    """The per-rank steps on the GPU, through librlhead (lm_head_gb300)."""

    def __init__(self):
        import lm_head_gb300 as rh
        self.rh = rh

    def local_batch(self, batch, w_shard: torch.Tensor, shard: Shard):
        rh = self.rh
        return dataclasses.replace(batch, weight=w_shard,
                                   labels=rh.rl_head_shard_remap(batch.labels, shard.begin, shard.end),
                                   ids=rh.rl_head_shard_remap(batch.ids, shard.begin, shard.end))

    def stats(self, local, params):
        return self.rh.rl_head_shard_stats(local, params)

    def loss(self, batch, params, stats_all, zlab, zsup, V: int):
        return self.rh.rl_head_loss_from_shard_stats(batch, params, stats_all, zlab, zsup, V=V)

    def backward(self, local, params, fwd, dloss):
        dX, dW, status = self.rh.rl_head_loss_bwd(local, params, fwd.saved, dloss)
        return dX, dW

    def dx_to_sum(self, dX_part: torch.Tensor) -> torch.Tensor:
        return dX_part.float()        # the parts are summed in fp32

    def dx_from_sum(self, dX_sum: torch.Tensor) -> torch.Tensor:
        return dX_sum.to(torch.bfloat16)


def forward(batch, w_shard, shard: Shard, V: int, params, ops, exch):
    """Steps 1-4: returns (the loss outputs as ops.loss gives them, the local batch)."""
    local = ops.local_batch(batch, w_shard, shard)
    stats, zlab, zsup = ops.stats(local, params)
    stats_all = exch.all_gather(stats)              # [R, 3, N], rank order
    exch.all_reduce_sum_(zlab)                      # each logit nonzero on its owner only
    exch.all_reduce_sum_(zsup)
    return ops.loss(batch, params, stats_all, zlab, zsup, V), local


def backward(local, params, fwd, dloss, ops, exch):
    """Steps 5-6: returns (dX summed over the ranks, this rank's rows of dW)."""
    dX_part, dW = ops.backward(local, params, fwd, dloss)
    total = exch.all_reduce_sum_(ops.dx_to_sum(dX_part))
    return ops.dx_from_sum(total), dW
