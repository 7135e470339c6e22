"""Data-parallel sharding of one Parallax layer problem across ranks.

Every (batch, head) of the layer is independent in the forward pass and for
dq, dk and dv.  The projector gradient is the one quantity shared across the
batch: dP_h = sum over b and t of du_t delta_t^T.  So:

* sharding by batch: rank r runs the whole layer on its contiguous slice of
  the batch, and the ranks sum their partial dP with one all-reduce
  ([H, d, d] float32) -- the only exchange step the layer has;
* sharding by head: rank r runs its slice of the heads and P; no exchange.

The arithmetic runs in the library's kernels (``parallax_fwd`` /
``parallax_bwd`` on the local slice); this module only splits the work and
issues the collective through ``torch.distributed`` on the caller's process
group.
"""
from __future__ import annotations

import torch

__all__ = ["shard_range", "allreduce_dP", "batch_sharded_step"]


def shard_range(n: int, rank: int, world: int) -> tuple[int, int]:
    """[lo, hi) of the rank's contiguous share of n items (the first n % world
    ranks take one more), so every item belongs to exactly one rank."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError("need 0 <= rank < world and n >= 0")
    base, extra = divmod(n, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def allreduce_dP(dP: torch.Tensor, group=None) -> torch.Tensor:
    """Sums the ranks' partial projector gradients in place (the batch-shard
    exchange step); a no-op without an initialised process group of size > 1."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(dP, op=dist.ReduceOp.SUM, group=group)
    return dP


def batch_sharded_step(q, k, v, P, dout, group=None, fwd_workspace=None, bwd_workspace=None, stream=None):
    """Forward and backward of the local batch slice, then the dP all-reduce.

    q, k, v, dout: this rank's [B_local, H, T, d] slice; P: the full [H, d, d]
    projector (replicated).  Returns (out, lse, mu_k, dq, dk, dv, dP) with dP
    summed over every rank's batch slice.
    """
    import parallax_local_linear_fwd_b300 as plx
    B, H, T, d = (int(x) for x in q.shape)
    if fwd_workspace is None:
        out, lse, mu = plx.parallax_fwd(q, k, v, P, stream=stream)
    else:
        out = torch.empty_like(q)
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
        mu = torch.empty((B, H, T, d), dtype=torch.float32, device=q.device)
        plx.parallax_fwd_ws(q, k, v, P, out, lse, mu, fwd_workspace, stream=stream)
    dq, dk, dv, dP = plx.parallax_bwd(q, k, v, P, lse, mu, dout, workspace=bwd_workspace, stream=stream)
    allreduce_dP(dP, group)
    return out, lse, mu, dq, dk, dv, dP
