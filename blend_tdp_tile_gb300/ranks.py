"""Round-robin TDP across ranks: the collective around the library's partial blend.

"Tiled Data Parallelism (TDP)", section "What it is": tiles are assigned to ranks
round-robin (tile t to rank t % world; 16 tiles on 4 GPUs is 4 tiles per rank), every
rank blends its own tiles, and a single all_reduce sums the blended tiles into the final
result.  Here each rank runs ``tdp_blend_partial`` (its tiles into an fp32 partial
latent, on its own GPU) and the ranks' partials are summed by torch.distributed:

  mode "all_reduce"      one all_reduce(sum) of the fp32 partial, then every rank stores
                         the sum in the plan's dtype (``tdp_blend_store``);
  mode "reduce_scatter"  a reduce_scatter of the partial over slabs of whole latent rows
                         (each rank sums one slab), each rank stores its slab in the plan's
                         dtype, and an all_gather of the stored slabs rebuilds the latent on
                         every rank: 4 + 2 bytes per bf16 element on the wire per rank
                         instead of all_reduce's 2 x 4.  Used when the rows divide evenly
                         among the ranks, else "all_reduce".

This module is host-side plumbing only: the arithmetic runs in the library's kernels
and in the collective.  The collective reads and writes this GPU's own buffers; no
kernel of the library waits on another rank.
"""
from __future__ import annotations

from typing import Callable, Optional

__all__ = ["rows_per_rank", "reduce_partials", "blend_across_ranks"]


def rows_per_rank(n_rows: int, world: int) -> Optional[int]:
    """Latent rows (b, f, h) each rank sums under "reduce_scatter", or None when they do not
    divide evenly (the all_reduce form is used then)."""
    if world < 1:
        raise ValueError("world must be >= 1")
    return n_rows // world if n_rows % world == 0 else None


def reduce_partials(Zp, Z, row_elems: int, store: Callable, group=None, mode: str = "reduce_scatter") -> str:
    """Sum the ranks' fp32 partial latents and leave the sum, in Z's dtype, in Z on every rank.

    Zp         this rank's fp32 partial latent (contiguous; overwritten).
    Z          the output latent (contiguous, same element count).
    row_elems  elements per latent row (W * C): the reduce_scatter slabs are whole rows.
    store      store(src_fp32, dst): write src into dst in dst's dtype (tdp_blend_store on a GPU).
    Returns the mode used ("all_reduce" or "reduce_scatter")."""
    import torch.distributed as dist
    if mode not in ("all_reduce", "reduce_scatter"):
        raise ValueError(f"unknown mode {mode!r}")
    if Zp.numel() != Z.numel() or Zp.numel() % row_elems != 0:
        raise ValueError("Zp and Z must hold the same whole number of latent rows")
    world = dist.get_world_size(group)
    zp, z = Zp.view(-1), Z.view(-1)
    per = rows_per_rank(zp.numel() // row_elems, world) if mode == "reduce_scatter" else None
    if per is None:
        dist.all_reduce(zp, op=dist.ReduceOp.SUM, group=group)
        store(zp, z)
        return "all_reduce"
    n = per * row_elems
    mine = zp.new_empty(n)
    dist.reduce_scatter_tensor(mine, zp, op=dist.ReduceOp.SUM, group=group)
    slab = z.new_empty(n)                 # this rank's rows in Z's dtype
    store(mine, slab)
    dist.all_gather_into_tensor(z, slab, group=group)
    return "reduce_scatter"


def blend_across_ranks(plan, Yout, Z, group=None, mode: str = "reduce_scatter", Zp=None, stream=None) -> str:
    """The blend of a round-robin TDP step on this rank's GPU, summed over the ranks of `group`.

    Yout  this rank's tile outputs in tdp_split's tile-major layout; only its own tiles
          (t % world == rank) are read.
    Z     [B,F,H,W,C] latent (plan dtype), written on every rank.
    Zp    optional fp32 [B,F,H,W,C] work buffer for the partial (allocated if None).
    Returns the mode used."""
    import torch
    import torch.distributed as dist

    from . import tdp_blend_partial, tdp_blend_store
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    if Zp is None:
        Zp = torch.empty(Z.shape, dtype=torch.float32, device=Z.device)
    s = stream if stream is not None else torch.cuda.current_stream(Z.device)
    with torch.cuda.stream(s):
        tdp_blend_partial(plan, rank, world, Yout, Zp, stream=s)
        return reduce_partials(Zp, Z, plan.W * plan.C,
                               lambda src, dst: tdp_blend_store(plan, src, dst, stream=s), group=group, mode=mode)
