"""A long context split across GPUs (context parallelism): host-side marshalling only.

Rank r of W holds, for every request, a contiguous block of its logical pages and
decodes just that block: a sparse selected-page pa_decode over the block (fp32 output
and lse), so each position keeps its place in the sequence and the causal cutoff stays
exact.  The ranks' partials are all-gathered with torch.distributed (NCCL on GPUs, gloo
on CPUs) and combined by pa_lse_merge, the log-sum-exp merge of the split-K partition
triple (ROCm/ATOM PR 2710, "Smaller": max logits, exp sums, partial outputs), here one
partition per GPU.  Every arithmetic step runs in libpagedfp8's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B


def rank_pages(context_lens, page_size: int, world: int, rank: int, stride: int | None = None):
    """The logical pages of every request that rank `rank` of `world` owns: request r's n
    pages are cut into `world` contiguous blocks, block k = [k n // world, (k + 1) n // world).
    Returns (selected int32 [B, stride], -1 padded; num_selected int32 [B]) for a sparse
    pa_decode.  stride defaults to the most pages one rank owns (at least 1)."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world {world}")
    L = np.asarray(context_lens, dtype=np.int64)
    n = (L + page_size - 1) // page_size
    lo, hi = n * rank // world, n * (rank + 1) // world
    cnt = (hi - lo).astype(np.int32)
    width = max(int(cnt.max()) if cnt.size else 0, 1)
    if stride is None:
        stride = width
    if stride < width:
        raise ValueError(f"stride {stride} below the {width} pages this rank owns")
    sel = np.full((L.size, stride), -1, dtype=np.int32)
    for r in range(L.size):
        sel[r, :cnt[r]] = np.arange(lo[r], hi[r], dtype=np.int32)
    return sel, cnt


def max_rank_pages(max_context_len: int, page_size: int, world: int) -> int:
    """The most pages one rank owns for any request of up to max_context_len tokens (the
    plan's max_selected_pages)."""
    n = (max_context_len + page_size - 1) // page_size
    return max(1, -(-n // world))


def gather_partials(out: torch.Tensor, lse: torch.Tensor, group=None):
    """All-gather of every rank's partial (out fp32 [rows, heads, D], lse fp32 [rows, heads]):
    returns (part_out [world, rows, heads, D], part_lse [world, rows, heads]), rank order."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    outs = [torch.empty_like(out) for _ in range(world)]
    lses = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(outs, out.contiguous(), group=group)
    dist.all_gather(lses, lse.contiguous(), group=group)
    return torch.stack(outs), torch.stack(lses)


def merge(part_out: torch.Tensor, part_lse: torch.Tensor, out_dtype=torch.bfloat16,
          with_lse: bool = False, stream=None):
    """pa_lse_merge of gathered partials (device tensors); returns out (and the lse)."""
    if part_out.dtype != torch.float32 or part_lse.dtype != torch.float32:
        raise TypeError("partials are fp32")
    out = torch.empty(part_out.shape[1:], dtype=out_dtype, device=part_out.device)
    lse = (torch.empty(part_lse.shape[1:], dtype=torch.float32, device=part_out.device)
           if with_lse else None)
    B.lse_merge(part_out.contiguous(), part_lse.contiguous(), out, lse, stream=stream)
    return (out, lse) if with_lse else out


def decode_shard(plan, q, k_cache, v_cache, block_table, context_lens_host, world: int,
                 rank: int, stream=None, **kw):
    """This rank's partial: a sparse pa_decode over its block of every request's pages.
    `plan` must be created with out_dtype "f32" and max_selected_pages >= the pages a rank
    owns (max_rank_pages).  context_lens_host is the host copy of context_lens; kw are
    pa_decode's other arguments (scales, cu_seqlens_q, sm_scale, ...).  Returns
    (out fp32 [rows, heads, D], lse fp32 [rows, heads])."""
    if plan.out_dtype != "f32":
        raise ValueError("the partials must be fp32: create the plan with out_dtype='f32'")
    sel, nsel = rank_pages(context_lens_host, plan.desc.page_size, world, rank,
                           stride=plan.desc.max_selected_pages)
    dev = q.device
    sel_d = torch.from_numpy(sel).to(dev)
    nsel_d = torch.from_numpy(nsel).to(dev)
    ctx = torch.as_tensor(np.asarray(context_lens_host, dtype=np.int32)).to(dev)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    out = plan.decode(q, k_cache, v_cache, block_table, ctx, lse=lse, selected_pages=sel_d,
                      num_selected=nsel_d, stream=stream, **kw)
    return out, lse
