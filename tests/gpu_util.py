"""Shared helpers of the GPU tests: sub-problems for the oracle and the tolerances."""
from __future__ import annotations

import dataclasses

import numpy as np

# bf16 outputs against the fp64 oracle (max-abs and cosine); LSE in natural-log units.
MAX_ABS = 1e-2
MIN_COS = 0.9999
LSE_ABS = 2e-3
# split-K against single pass, both fp32 outputs, relative to the output's scale
SPLIT_REL = 1e-3


def subset(p, idx):
    """The same problem restricted to requests idx (caches and block tables shared)."""
    idx = np.asarray(idx, dtype=np.int64)
    ql = p.q_lens[idx]
    cu = np.zeros(len(idx) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    rows = np.concatenate([np.arange(p.cu_seqlens_q[r], p.cu_seqlens_q[r + 1]) for r in idx]) \
        if len(idx) else np.zeros(0, np.int64)
    uni = int(ql[0]) if len(idx) and np.all(ql == ql[0]) else None
    return dataclasses.replace(
        p, num_seqs=len(idx), q=p.q[rows], block_table=p.block_table[idx],
        context_lens=p.context_lens[idx], cu_seqlens_q=cu, uniform_q_len=uni,
        selected=None if p.selected is None else p.selected[idx],
        num_selected=None if p.num_selected is None else p.num_selected[idx])


def rows_of(p, idx):
    return np.concatenate([np.arange(p.cu_seqlens_q[r], p.cu_seqlens_q[r + 1]) for r in idx])


def compare(got, ref, what="", max_abs=MAX_ABS, min_cos=MIN_COS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    den = np.linalg.norm(got) * np.linalg.norm(ref)
    cos = float((got * ref).sum() / den) if den > 0 else 1.0
    assert err <= max_abs, f"{what}: max abs {err:.3e} > {max_abs}"
    assert cos >= min_cos, f"{what}: cosine {cos:.7f} < {min_cos}"
    return err, cos


def compare_lse(got, ref, what="", tol=LSE_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: lse finiteness differs"
    if fin.any():
        err = float(np.abs(got[fin] - ref[fin]).max())
        assert err <= tol, f"{what}: lse err {err:.3e}"
