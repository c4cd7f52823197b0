"""Seeded synthetic inputs for paged decode attention over an FP8 (e4m3) KV cache.

This module only makes data: it holds none of the attention arithmetic, so that the
CUDA path and the fp64 CPU oracle can both consume the very same bytes.  Every array
is a numpy array on the host; callers copy what they need to the device.

Workload recipe (the shapes and value distributions of the MiniMax-M3 decode
workloads on the source pages: one KV head per tensor-parallel rank, 16 query heads
per KV head, head_dim 128, pages of 128 tokens, ROCm/ATOM PR 2122 section 2 and
vLLM PR 52060 "Serve command"):

* Q is bf16, drawn N(0, 1) in fp32 and rounded to bf16 (round to nearest even).
* K and V are drawn N(0, 1) in fp32.  Per-token mode quantises every (page, KV head,
  slot) row of head_dim values to e4m3 with scale = amax / 448 (fp32 scale, codes
  from x / scale clamped to +-448 and rounded to nearest even by the torch cast);
  an all-zero row gets scale 0 and codes 0.  Scalar mode draws one K and one V scale
  uniform in [0.005, 0.05] and quantises x / scale the same way (saturation at +-448
  is part of the data).  The BF16 control stores the dequantised values code * scale
  rounded to bf16.
* Block tables map every logical page of every request to a distinct physical page
  of a shared pool, through a seeded random permutation of the pool.
* Ragged speculative-decode batches carry cu_seqlens_q; uniform batches also carry
  it (row r * q_len), so both sides see one row map.
* Sparse batches carry a per-request list of logical page indices (sampled without
  replacement, always holding the request's last page), padded with -1.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclasses.dataclass
class Problem:
    num_seqs: int
    num_kv_heads: int
    group_size: int
    head_dim: int
    page_size: int
    kv_dtype: str                      # "fp8" | "bf16"
    scale_mode: str                    # "none" | "scalar" | "per_token"
    q: np.ndarray                      # uint16 bf16 bits [rows, Hq, D]
    k_cache: np.ndarray                # uint8 codes or uint16 bf16 bits [P, Hkv, ps, D]
    v_cache: np.ndarray
    k_scale: Optional[np.ndarray]      # float32 [P, Hkv, ps] (per-token mode)
    v_scale: Optional[np.ndarray]
    k_scale_scalar: float
    v_scale_scalar: float
    block_table: np.ndarray            # int32 [B, stride]
    context_lens: np.ndarray           # int32 [B]
    cu_seqlens_q: np.ndarray           # int32 [B + 1]
    uniform_q_len: Optional[int]       # q_len when every request has the same count
    selected: Optional[np.ndarray]     # int32 [B, sel_stride], -1 padded
    num_selected: Optional[np.ndarray]  # int32 [B]
    sm_scale: float
    name: str = ""

    @property
    def num_rows(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q).astype(np.int32)

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max()) if self.num_seqs else 0


# ----------------------------------------------------------------------------- data

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 values -> bf16 bit patterns (torch cast, round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    """fp32 values (already in code units) -> e4m3fn codes, clamped to +-448."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).clamp_(-E4M3_MAX, E4M3_MAX)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    """e4m3fn codes -> fp32 values via the torch dtype (used only to build the BF16 control)."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy()


def quantize_per_token(x: np.ndarray):
    """Per-row quantisation over the last axis: scale = amax / 448."""
    amax = np.abs(x).max(axis=-1).astype(np.float32)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    codes = e4m3_codes(x / safe[..., None])
    codes[scale == 0] = 0
    return codes, scale


def quantize_scalar(x: np.ndarray, scale: float):
    return e4m3_codes(x / np.float32(scale))


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def _fill_pages(rng, pages: np.ndarray, Hkv, ps, D, scale_mode, kv_dtype, k_out, v_out,
                ks_out, vs_out, kss, vss, chunk=1024, kv_mag_log2=0.0):
    """Draw N(0,1) K/V for the listed physical pages and store their encoding.  With
    kv_mag_log2 = M > 0 every (page, KV head, slot) row is first multiplied by its own
    2^u, u uniform in [-M, M] (K and V drawn independently)."""
    for i in range(0, len(pages), chunk):
        idx = pages[i:i + chunk]
        for which, out, sout, ss in ((0, k_out, ks_out, kss), (1, v_out, vs_out, vss)):
            x = _normal(rng, (len(idx), Hkv, ps, D))
            if kv_mag_log2 > 0:
                u = rng.uniform(-kv_mag_log2, kv_mag_log2, size=(len(idx), Hkv, ps, 1))
                x = (x * np.exp2(u)).astype(np.float32)
            if scale_mode == "per_token":
                codes, sc = quantize_per_token(x)
            elif scale_mode == "scalar":
                codes, sc = quantize_scalar(x, ss), None
            else:
                codes, sc = None, None
            if kv_dtype == "fp8":
                out[idx] = codes
                if sc is not None:
                    sout[idx] = sc
            else:
                if codes is None:
                    out[idx] = bf16_bits(x)
                else:
                    val = e4m3_values(codes)
                    val = val * (sc[..., None] if sc is not None else np.float32(ss))
                    out[idx] = bf16_bits(val)


def make_problem(seed: int, *, num_seqs: int, context_lens: Sequence[int],
                 q_lens: Sequence[int], num_kv_heads: int = 1, group_size: int = 16,
                 head_dim: int = 128, page_size: int = 128, kv_dtype: str = "fp8",
                 scale_mode: str = "per_token", pool_pages: Optional[int] = None,
                 selected_pages: Optional[int] = None, block_table_pad: int = 0,
                 only_selected_data: bool = False, kv_mag_log2: float = 0.0,
                 q_mag_log2: float = 0.0, name: str = "") -> Problem:
    """General seeded problem.  kv_dtype "bf16" with scale_mode "none" draws bf16 values
    directly; "bf16" with another scale_mode stores the dequantised e4m3 values.
    kv_mag_log2 = M gives every K and V token row its own magnitude 2^u, u uniform in
    [-M, M], before quantisation; q_mag_log2 = Mq does the same for every query element."""
    rng = np.random.default_rng(seed)
    B, Hkv, g, D, ps = num_seqs, num_kv_heads, group_size, head_dim, page_size
    L = np.asarray(context_lens, dtype=np.int64)
    ql = np.asarray(q_lens, dtype=np.int64)
    assert L.shape == (B,) and ql.shape == (B,)
    npg = (L + ps - 1) // ps
    need = int(npg.sum())
    P = max(need, 1) if pool_pages is None else int(pool_pages)
    assert P >= need, "pool too small"
    perm = rng.permutation(P).astype(np.int32)
    stride = max(int(npg.max()) if B else 1, 1) + block_table_pad
    bt = np.full((B, stride), -1, dtype=np.int32)
    off = 0
    for r in range(B):
        bt[r, :npg[r]] = perm[off:off + npg[r]]
        off += int(npg[r])

    sel = nsel = None
    if selected_pages is not None:
        sel = np.full((B, selected_pages), -1, dtype=np.int32)
        nsel = np.zeros(B, dtype=np.int32)
        for r in range(B):
            n = int(npg[r])
            k = min(selected_pages, n)
            if n == 0:
                continue
            others = rng.choice(n - 1, size=k - 1, replace=False) if k > 1 else np.zeros(0, int)
            pick = np.concatenate([others, [n - 1]]).astype(np.int32)
            rng.shuffle(pick)
            sel[r, :k] = pick
            nsel[r] = k

    kss = float(rng.uniform(0.005, 0.05)) if scale_mode == "scalar" else 1.0
    vss = float(rng.uniform(0.005, 0.05)) if scale_mode == "scalar" else 1.0
    cdt = np.uint8 if kv_dtype == "fp8" else np.uint16
    k_cache = np.zeros((P, Hkv, ps, D), dtype=cdt)
    v_cache = np.zeros((P, Hkv, ps, D), dtype=cdt)
    per_tok = scale_mode == "per_token" and kv_dtype == "fp8"
    k_scale = np.zeros((P, Hkv, ps), dtype=np.float32) if per_tok else None
    v_scale = np.zeros((P, Hkv, ps), dtype=np.float32) if per_tok else None
    if only_selected_data and sel is not None:
        used = np.unique(np.concatenate(
            [bt[r, sel[r, :nsel[r]]] for r in range(B) if nsel[r] > 0] or [np.zeros(0, np.int32)]))
    else:
        used = np.arange(P, dtype=np.int64)
    used = np.asarray(used, dtype=np.int64)
    _fill_pages(rng, used, Hkv, ps, D, scale_mode, kv_dtype, k_cache, v_cache,
                k_scale, v_scale, kss, vss, kv_mag_log2=kv_mag_log2)

    rows = int(ql.sum())
    qf = _normal(rng, (rows, Hkv * g, D))
    if q_mag_log2 > 0:
        qf = (qf * np.exp2(rng.uniform(-q_mag_log2, q_mag_log2, size=qf.shape))).astype(np.float32)
    q = bf16_bits(qf)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    uni = int(ql[0]) if B and np.all(ql == ql[0]) else None
    eff_mode = scale_mode if kv_dtype == "fp8" else "none"
    return Problem(num_seqs=B, num_kv_heads=Hkv, group_size=g, head_dim=D, page_size=ps,
                   kv_dtype=kv_dtype, scale_mode=eff_mode, q=q, k_cache=k_cache,
                   v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                   k_scale_scalar=kss if eff_mode == "scalar" else 1.0,
                   v_scale_scalar=vss if eff_mode == "scalar" else 1.0,
                   block_table=bt, context_lens=L.astype(np.int32), cu_seqlens_q=cu,
                   uniform_q_len=uni, selected=sel, num_selected=nsel,
                   sm_scale=1.0 / float(np.sqrt(D)), name=name)


def subset(p: Problem, idx) -> Problem:
    """The same problem restricted to requests idx (caches and block tables shared)."""
    idx = np.asarray(idx, dtype=np.int64)
    ql = p.q_lens[idx]
    cu = np.zeros(len(idx) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    rows = rows_of(p, idx) if len(idx) else np.zeros(0, np.int64)
    uni = int(ql[0]) if len(idx) and np.all(ql == ql[0]) else None
    return dataclasses.replace(
        p, num_seqs=len(idx), q=p.q[rows], block_table=p.block_table[idx],
        context_lens=p.context_lens[idx], cu_seqlens_q=cu, uniform_q_len=uni,
        selected=None if p.selected is None else p.selected[idx],
        num_selected=None if p.num_selected is None else p.num_selected[idx])


def rows_of(p: Problem, idx) -> np.ndarray:
    """The query rows of requests idx, in order."""
    return np.concatenate([np.arange(p.cu_seqlens_q[r], p.cu_seqlens_q[r + 1]) for r in idx])


# --------------------------------------------------------------------- named workloads

def tiny_dense(seed: int = 0) -> Problem:
    """4 requests, Hkv 1, group 16, D 128, page 16, context uniform in [1, 300], q_len 1,
    block table a random permutation of a 128-page pool."""
    rng = np.random.default_rng(seed + 1000)
    L = rng.integers(1, 301, size=4)
    return make_problem(seed, num_seqs=4, context_lens=L, q_lens=[1] * 4, page_size=16,
                        pool_pages=128, name="tiny dense decode")


def dense_8k(seed: int = 1, kv_dtype: str = "fp8", num_seqs: int = 32) -> Problem:
    """Batch 32, every context 8192, page 128, q_len 1, per-token e4m3 K/V (or the BF16
    control with the same dequantised values)."""
    return make_problem(seed, num_seqs=num_seqs, context_lens=[8192] * num_seqs,
                        q_lens=[1] * num_seqs, page_size=128, kv_dtype=kv_dtype,
                        scale_mode="per_token", name="dense decode 8K")


def long_128k(seed: int = 2, scale_mode: str = "scalar", num_seqs: int = 8,
              context: int = 131072) -> Problem:
    """Batch 8, every context 131072, page 128, q_len 1, scalar or per-token scales."""
    return make_problem(seed, num_seqs=num_seqs, context_lens=[context] * num_seqs,
                        q_lens=[1] * num_seqs, page_size=128, scale_mode=scale_mode,
                        name="long-context decode 128K")


def ragged_spec(seed: int = 3, batch: str = "A") -> Problem:
    """(A) 31 requests, 30 with q_len 4 and one (seeded position) with q_len 1 (121 rows);
    (B) 4 requests with q_len [4, 4, 6, 2] (16 rows).  Contexts uniform in [1024, 32768]."""
    rng = np.random.default_rng(seed + 1000 + (0 if batch == "A" else 1))
    if batch == "A":
        ql = [4] * 31
        ql[int(rng.integers(0, 31))] = 1
    else:
        ql = [4, 4, 6, 2]
    L = rng.integers(1024, 32769, size=len(ql))
    return make_problem(seed + (0 if batch == "A" else 100), num_seqs=len(ql), context_lens=L,
                        q_lens=ql, page_size=128, name=f"ragged speculative decode {batch}")


def sparse_selected(seed: int = 4, num_seqs: int = 32, context: int = 131072,
                    selected: int = 64, only_selected_data: bool = True) -> Problem:
    """Batch 32, context 131072 (1024 pages), 64 selected pages per request (always the
    last page), q_len 1 for the first half of the requests and 4 for the second half."""
    ql = [1] * (num_seqs // 2) + [4] * (num_seqs - num_seqs // 2)
    return make_problem(seed, num_seqs=num_seqs, context_lens=[context] * num_seqs,
                        q_lens=ql, page_size=128, selected_pages=selected,
                        only_selected_data=only_selected_data, name="sparse selected-page decode")


def prefill_as_decode(seed: int = 6, num_tokens: int = 2048, prefix: int = 0,
                      page_size: int = 128, selected_pages: Optional[int] = None,
                      scale_mode: str = "per_token", name: str = "") -> Problem:
    """A prefill chunk of one sequence run through the decode contract, one request per new
    token (ROCm/ATOM PR 2614, "Change": per-token-as-decode prefill reuses the paged-decode
    contract).  The sequence holds prefix + num_tokens tokens; request t is the query row of
    token prefix + t, with context prefix + t + 1 and q_len 1, and every request shares the
    sequence's block table, so row t attends exactly the causal prefix of its token.  With
    selected_pages, request t attends that many of its prefix's pages instead (always its
    own last page), as the sparse prefill does."""
    L = prefix + num_tokens
    base = make_problem(seed, num_seqs=1, context_lens=[L], q_lens=[1], page_size=page_size,
                        scale_mode=scale_mode, name=name or "prefill as decode")
    rng = np.random.default_rng(seed + 500)
    T = num_tokens
    ctx = (prefix + np.arange(1, T + 1)).astype(np.int32)
    bt = np.repeat(base.block_table, T, axis=0)
    q = bf16_bits(_normal(rng, (T, base.num_kv_heads * base.group_size, base.head_dim)))
    sel = nsel = None
    if selected_pages is not None:
        sel = np.full((T, selected_pages), -1, dtype=np.int32)
        nsel = np.zeros(T, dtype=np.int32)
        for t in range(T):
            n = (int(ctx[t]) + page_size - 1) // page_size
            k = min(selected_pages, n)
            others = rng.choice(n - 1, size=k - 1, replace=False) if k > 1 else np.zeros(0, int)
            pick = np.concatenate([others, [n - 1]]).astype(np.int32)
            rng.shuffle(pick)
            sel[t, :k] = pick
            nsel[t] = k
    return dataclasses.replace(base, num_seqs=T, q=q, block_table=bt, context_lens=ctx,
                               cu_seqlens_q=np.arange(T + 1, dtype=np.int32), uniform_q_len=1,
                               selected=sel, num_selected=nsel)


@dataclasses.dataclass
class IndexProblem:
    """Inputs of the indexer's block score and top-k: index queries, the e4m3 index cache
    (num_pages, page_size, 128) with optional per-token scales, and the decode row map."""
    q: np.ndarray                 # bf16 bits [rows, index_heads, 128]
    k_cache: np.ndarray           # uint8 e4m3 codes [num_pages, page_size, 128]
    k_scale: Optional[np.ndarray]  # fp32 [num_pages, page_size] or None
    block_table: np.ndarray       # int32 [B, stride]
    context_lens: np.ndarray      # int32 [B]
    cu_seqlens_q: np.ndarray      # int32 [B + 1]
    sm_scale: float
    topk: int
    name: str = ""

    @property
    def num_rows(self) -> int:
        return int(self.cu_seqlens_q[-1])


def index_problem(seed: int, context_lens: Sequence[int], q_lens: Sequence[int],
                  index_heads: int = 1, page_size: int = 128, topk: int = 64,
                  per_token_scale: bool = True, hot_pages: int = 8, pool_pages=None,
                  zero_q: bool = False, name: str = "") -> IndexProblem:
    """Seeded indexer inputs.  Index keys are N(0, 1) quantised per token (scale amax/448)
    or, without per-token scales, quantised at a fixed scale of 1/64; each request has
    `hot_pages` pages whose keys lean towards its first query row, so that the selection
    has a clear top; block tables are a random permutation of the pool."""
    rng = np.random.default_rng(seed)
    L = np.asarray(context_lens, dtype=np.int64)
    ql = np.asarray(q_lens, dtype=np.int64)
    B, D, ps, H = len(L), 128, page_size, index_heads
    npg = (L + ps - 1) // ps
    P = int(npg.sum()) if pool_pages is None else int(pool_pages)
    perm = rng.permutation(P).astype(np.int32)
    stride = max(int(npg.max()), 1)
    bt = np.full((B, stride), -1, dtype=np.int32)
    off = 0
    for r in range(B):
        bt[r, :npg[r]] = perm[off:off + npg[r]]
        off += int(npg[r])
    rows = int(ql.sum())
    qf = np.zeros((rows, H, D), np.float32) if zero_q else _normal(rng, (rows, H, D))
    x = _normal(rng, (P, ps, D))
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    for r in range(B):
        if npg[r] == 0 or zero_q:
            continue
        hot = rng.choice(int(npg[r]), size=min(hot_pages, int(npg[r])), replace=False)
        dirn = qf[cu[r], 0] / max(float(np.linalg.norm(qf[cu[r], 0])), 1e-6)
        for b in hot:
            x[bt[r, b]] += (rng.uniform(0.5, 3.0) * np.sqrt(D) * 0.25) * dirn
    if per_token_scale:
        codes, sc = quantize_per_token(x)
    else:
        codes, sc = quantize_scalar(x, 1.0 / 64.0), None
    return IndexProblem(q=bf16_bits(qf), k_cache=codes, k_scale=sc, block_table=bt,
                        context_lens=L.astype(np.int32), cu_seqlens_q=cu,
                        sm_scale=1.0 / float(np.sqrt(D)), topk=topk, name=name)


def index_decode_128k(seed: int = 8) -> IndexProblem:
    """The sparse decode's indexer step: batch 32, context 131072 (1024 pages of 128),
    q_len 1 for the first 16 requests and 4 for the others (80 rows), one index head,
    per-token e4m3 index keys, top 64 pages."""
    ql = [1] * 16 + [4] * 16
    return index_problem(seed, [131072] * 32, ql, index_heads=1, page_size=128, topk=64,
                         name="indexer block score + top-64, batch 32, context 131072")


@dataclasses.dataclass
class KvWriteCase:
    """New K/V rows (bf16 bits [T, Hkv, D]), their slots, and sentinel-filled caches."""
    k_new: np.ndarray
    v_new: np.ndarray
    slot_mapping: np.ndarray      # int64 [T]
    k_cache: np.ndarray           # uint8 [P, Hkv, ps, D]
    v_cache: np.ndarray
    k_scale: np.ndarray           # fp32 [P, Hkv, ps]
    v_scale: np.ndarray
    name: str = ""
    block_table: Optional[np.ndarray] = None   # int32 [B, pages]: where a prefill layout put each sequence
    context_lens: Optional[np.ndarray] = None  # int32 [B]


def kv_write_case(seed: int, num_tokens: int, num_kv_heads: int = 1, page_size: int = 128,
                  num_pages: int = 64, skip: int = 0, past_end: int = 0,
                  special_rows: bool = True, name: str = "") -> KvWriteCase:
    """Seeded new-token K/V rows for the quantise-and-write step.

    Rows are N(0, 1) times a per-row magnitude drawn log-uniformly from 2^-20 .. 2^20;
    with special_rows, a few rows are all zero, e4m3 values times a power of two (with
    +-448 among them), or one nonzero value, and one row mixes magnitudes 2^-40 .. 2^10.
    Slots are distinct and drawn without replacement from the cache; `skip` tokens get
    slot -1 and `past_end` tokens a slot past the cache.  Caches hold sentinel bytes."""
    rng = np.random.default_rng(seed)
    T, Hkv, D, ps, P = num_tokens, num_kv_heads, 128, page_size, num_pages
    assert T <= P * ps
    mag = np.exp2(rng.uniform(-20, 20, size=(T, Hkv, 1))).astype(np.float32)
    x = (_normal(rng, (T, Hkv, D)) * mag).astype(np.float32)
    y = (_normal(rng, (T, Hkv, D)) * mag[::-1]).astype(np.float32)
    if special_rows and T >= 4:
        x[0, 0] = 0.0
        codes = rng.integers(0, 0x7F, size=D).astype(np.uint8) | \
            (rng.integers(0, 2, size=D).astype(np.uint8) << 7)
        codes[codes & 0x7F == 0x7F] = 0x7E
        codes[5] = 0x7E
        x[1, 0] = e4m3_values(codes) * np.float32(2.0 ** -7)
        y[2, 0] = 0.0
        y[2, 0, 77] = np.float32(-0.3125)
        x[3, 0] = (_normal(rng, (D,)) * np.exp2(rng.uniform(-40, 10, size=D))).astype(np.float32)
    slots = rng.choice(P * ps, size=T, replace=False).astype(np.int64)
    idx = rng.permutation(T)
    slots[idx[:skip]] = -1
    slots[idx[skip:skip + past_end]] = P * ps + rng.integers(0, 1000, size=past_end)
    return KvWriteCase(
        k_new=bf16_bits(x), v_new=bf16_bits(y), slot_mapping=slots,
        k_cache=np.full((P, Hkv, ps, D), 0xC3, dtype=np.uint8),
        v_cache=np.full((P, Hkv, ps, D), 0x3C, dtype=np.uint8),
        k_scale=np.full((P, Hkv, ps), -1.0, dtype=np.float32),
        v_scale=np.full((P, Hkv, ps), -2.0, dtype=np.float32), name=name)


def kv_write_prefill_8k(seed: int = 5) -> KvWriteCase:
    """The whole dense-8K batch written at once: 32 sequences x 8192 tokens = 262144 tokens,
    Hkv 1, page 128, into a 2048-page pool.  Each sequence owns 64 pages of a random
    permutation of the pool (its block table) and its tokens fill them in order, as a
    prefill writes them."""
    c = kv_write_case(seed, 32 * 8192, 1, 128, 2048, special_rows=True,
                      name="KV quantise-and-write, 262144 tokens (dense 8K batch)")
    rng = np.random.default_rng(seed + 77)
    pages = rng.permutation(2048).astype(np.int64).reshape(32, 64)
    pos = np.arange(8192, dtype=np.int64)
    c.slot_mapping = (pages[:, pos // 128] * 128 + pos % 128).reshape(-1)
    c.block_table = pages.astype(np.int32)
    c.context_lens = np.full(32, 8192, dtype=np.int32)
    return c


def kv_bytes_per_token(p: Problem) -> int:
    """Algorithmic bytes of one attended (token, KV head): K and V rows plus scales."""
    if p.kv_dtype == "bf16":
        return 4 * p.head_dim
    return 2 * p.head_dim + (8 if p.scale_mode == "per_token" else 0)
