"""Moves a seeded problem (synth.Problem) to the device and runs it through a Plan.

Marshalling only: tensors are copied as they are, and every step of the attention runs
in libpagedfp8's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from .binding import Plan


def to_device(p, device="cuda") -> dict:
    dev = torch.device(device)
    t = lambda a, dt=None: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    d = {
        "q": torch.from_numpy(p.q.view(np.int16)).view(torch.bfloat16).to(dev),
        "block_table": t(p.block_table), "context_lens": t(p.context_lens),
        "cu_seqlens_q": t(p.cu_seqlens_q),
    }
    if p.kv_dtype == "fp8":
        d["k_cache"] = t(p.k_cache)
        d["v_cache"] = t(p.v_cache)
    else:
        d["k_cache"] = torch.from_numpy(p.k_cache.view(np.int16)).view(torch.bfloat16).to(dev)
        d["v_cache"] = torch.from_numpy(p.v_cache.view(np.int16)).view(torch.bfloat16).to(dev)
    if p.scale_mode == "per_token":
        d["k_scale"] = t(p.k_scale)
        d["v_scale"] = t(p.v_scale)
    if p.selected is not None:
        d["selected_pages"] = t(p.selected)
        d["num_selected"] = t(p.num_selected)
    return d


def plan_for(p, *, out_dtype="bf16", partition_tokens=0, ragged=None, device="cuda",
             max_context_len=None, q_len=None, max_selected_pages=None, **kw) -> Plan:
    """A plan sized exactly for problem p (its capacity bucket)."""
    rag = ragged if ragged is not None else (p.uniform_q_len is None)
    ql = q_len if q_len is not None else (p.max_q_len if rag else int(p.uniform_q_len))
    if max_selected_pages is None:
        max_selected_pages = 0 if p.selected is None else p.selected.shape[1]
    return Plan(device=device, num_kv_heads=p.num_kv_heads, group_size=p.group_size,
                head_dim=p.head_dim, page_size=p.page_size, kv_dtype=p.kv_dtype,
                scale_mode=p.scale_mode, q_mode="ragged" if rag else "uniform",
                q_len=max(ql, 1), max_batch=max(p.num_seqs, 1), max_rows=max(p.num_rows, 1),
                max_context_len=max_context_len or max(int(p.context_lens.max()), 1),
                max_selected_pages=max_selected_pages,
                partition_tokens=partition_tokens, out_dtype=out_dtype, **kw)


def call_kwargs(p, d: dict, *, with_cu=True, host_mirror=True) -> dict:
    kw = dict(k_scale=d.get("k_scale"), v_scale=d.get("v_scale"),
              k_scale_scalar=p.k_scale_scalar, v_scale_scalar=p.v_scale_scalar,
              sm_scale=p.sm_scale, selected_pages=d.get("selected_pages"),
              num_selected=d.get("num_selected"))
    if with_cu:
        kw["cu_seqlens_q"] = d["cu_seqlens_q"]
        if host_mirror:
            kw["cu_seqlens_q_host"] = p.cu_seqlens_q
    return kw


def run(plan: Plan, p, d: dict, *, lse=False, **kw):
    """Decodes problem p (already on the device as d); returns (out, lse or None)."""
    l = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=d["q"].device) if lse else None
    ck = call_kwargs(p, d)
    ck.update(kw)
    out = plan.decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["context_lens"],
                      lse=l, **ck)
    return out, l
