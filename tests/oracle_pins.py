"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each pin takes an OracleLib (the real build, or a mutated copy) and raises
AssertionError when the oracle disagrees with
  * a library routine (torch's float8_e4m3fn / bfloat16 decoding, torch's fp64
    scaled_dot_product_attention and logsumexp over a gather built with torch
    indexing),
  * a closed form (equal keys give the mean of V, q = 0 gives the uniform mean and
    log n, one key gives that key's V, two keys give a logistic weight),
  * an invariant stated by the source pages (folded scales equal per-element
    dequantisation, unit scales with bf16-exact values equal bf16 attention, a ragged
    batch equals its uniform pieces row by row, a sparse run over every page equals
    the dense run, scalar mode equals per-token mode with equal scales), or
  * a worked example printed on the pages (the [4, 4, 6, 2] ragged batch, 121 rows).
"""
from __future__ import annotations

import dataclasses
import os

import numpy as np
import torch
import torch.nn.functional as F

from paged_fp8_kv_04_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TOL = 1e-11


# ------------------------------------------------------------------ independent brute force

def _dequant_cache(p, which):
    cache = p.k_cache if which == "k" else p.v_cache
    if p.kv_dtype == "fp8":
        x = torch.from_numpy(np.ascontiguousarray(cache)).view(torch.float8_e4m3fn).to(torch.float64)
    else:
        x = torch.from_numpy(np.ascontiguousarray(cache).view(np.int16)).view(torch.bfloat16)
        x = x.to(torch.float64)
    if p.scale_mode == "per_token":
        s = p.k_scale if which == "k" else p.v_scale
        x = x * torch.from_numpy(s).to(torch.float64)[..., None]
    elif p.scale_mode == "scalar":
        x = x * float(p.k_scale_scalar if which == "k" else p.v_scale_scalar)
    return x


def _q64(p):
    return torch.from_numpy(p.q.view(np.int16)).view(torch.bfloat16).to(torch.float64)


def _positions(p, r):
    """Candidate positions of request r (before the causal cutoff), in gather order."""
    L, ps = int(p.context_lens[r]), p.page_size
    if p.selected is None:
        return torch.arange(L, dtype=torch.int64)
    pages = [int(x) for x in p.selected[r, :p.num_selected[r]] if x >= 0]
    if not pages:
        return torch.zeros(0, dtype=torch.int64)
    pos = (torch.tensor(pages)[:, None] * ps + torch.arange(ps)[None, :]).reshape(-1)
    return pos[pos < L]


def brute_force(p):
    """fp64 torch attention: gather with tensor indexing, SDPA with a boolean mask."""
    K, V, Q = _dequant_cache(p, "k"), _dequant_cache(p, "v"), _q64(p)
    g, D = p.group_size, p.head_dim
    out = torch.zeros(Q.shape, dtype=torch.float64)
    lse = torch.full(Q.shape[:2], float("-inf"), dtype=torch.float64)
    bt = torch.from_numpy(p.block_table).to(torch.int64)
    for r in range(p.num_seqs):
        r0, r1 = int(p.cu_seqlens_q[r]), int(p.cu_seqlens_q[r + 1])
        ql = r1 - r0
        if ql == 0:
            continue
        pos = _positions(p, r)
        phys = bt[r, pos // p.page_size]
        slot = pos % p.page_size
        tok = torch.arange(ql)[:, None]
        mask = pos[None, :] < (int(p.context_lens[r]) - ql + tok + 1)       # [ql, n]
        for h in range(p.num_kv_heads):
            Kr, Vr = K[phys, h, slot], V[phys, h, slot]                    # [n, D]
            Qr = Q[r0:r1, h * g:(h + 1) * g].transpose(0, 1)                # [g, ql, D]
            if pos.numel() == 0:
                continue
            o = F.scaled_dot_product_attention(Qr, Kr[None].expand(g, -1, -1),
                                               Vr[None].expand(g, -1, -1),
                                               attn_mask=mask[None].expand(g, -1, -1),
                                               scale=p.sm_scale)
            s = (Qr @ Kr.T) * p.sm_scale
            s = s.masked_fill(~mask[None], float("-inf"))
            lz = torch.logsumexp(s, dim=-1)                                 # [g, ql]
            empty = ~mask.any(dim=-1)                                       # [ql]
            o = torch.where(empty[None, :, None], torch.zeros_like(o), o)
            out[r0:r1, h * g:(h + 1) * g] = o.transpose(0, 1)
            lse[r0:r1, h * g:(h + 1) * g] = lz.transpose(0, 1)
    return out.numpy(), lse.numpy()


def _close(a, b, tol=TOL, what=""):
    a, b = np.asarray(a), np.asarray(b)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: finiteness differs"
    assert np.array_equal(a[~fin], b[~fin]), f"{what}: infinities differ"
    err = np.max(np.abs(a[fin] - b[fin])) if fin.any() else 0.0
    assert err <= tol, f"{what}: max abs diff {err}"


# ----------------------------------------------------------------------------- problems

def _small(seed, **kw):
    base = dict(num_seqs=3, context_lens=[37, 5, 20], q_lens=[1, 1, 1], page_size=16,
                head_dim=32, group_size=4)
    base.update(kw)
    return synth.make_problem(seed, **base)


def _mutate(p, **kw):
    return dataclasses.replace(p, **kw)


# --------------------------------------------------------------------------------- pins

def pin_e4m3_all_codes(lib):
    """Every one of the 256 e4m3fn codes decodes as torch.float8_e4m3fn does."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([lib.dec_e4m3(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "NaN codes differ"
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m]), "e4m3 values differ"
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def pin_bf16_all_patterns(lib):
    """Every bf16 bit pattern decodes as torch.bfloat16 does (NaNs as NaN)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([lib.dec_bf16(int(b)) for b in bits[::7]])
    r = ref[::7]
    assert np.array_equal(np.isnan(got), np.isnan(r))
    m = ~np.isnan(r)
    assert np.array_equal(got[m], r[m]), "bf16 values differ"


def pin_brute_dense_per_token(lib):
    p = _small(11)
    _close(lib.decode(p)[0], brute_force(p)[0], what="out")
    _close(lib.decode(p)[1], brute_force(p)[1], what="lse")


def pin_brute_dense_scalar(lib):
    p = _small(12, scale_mode="scalar")
    o, l = lib.decode(p)
    bo, bl = brute_force(p)
    _close(o, bo, what="out")
    _close(l, bl, what="lse")


def pin_brute_bf16_kv(lib):
    p = _small(13, kv_dtype="bf16", scale_mode="none")
    o, l = lib.decode(p)
    bo, bl = brute_force(p)
    _close(o, bo, what="out")
    _close(l, bl, what="lse")


def pin_brute_two_kv_heads(lib):
    """Hkv = 2 so that the head -> KV-head map and the cache's head stride both matter."""
    p = _small(14, num_kv_heads=2, context_lens=[40, 17, 3])
    o, l = lib.decode(p)
    bo, bl = brute_force(p)
    _close(o, bo, what="out")
    _close(l, bl, what="lse")


def pin_brute_ragged_causal(lib):
    """Ragged q_len [4, 4, 6, 2] with the cutoff L - q_len + tok + 1 (and one L < q_len)."""
    p = _small(15, num_seqs=5, context_lens=[50, 9, 33, 18, 3], q_lens=[4, 4, 6, 2, 5])
    o, l = lib.decode(p)
    bo, bl = brute_force(p)
    _close(o, bo, what="out")
    _close(l, bl, what="lse")


def pin_brute_sparse(lib):
    p = _small(16, num_seqs=3, context_lens=[100, 60, 77], q_lens=[1, 3, 2], selected_pages=3)
    sel = p.selected.copy()
    sel[1, 2] = -1                                   # padding inside the count
    p = _mutate(p, selected=sel)
    o, l = lib.decode(p)
    bo, bl = brute_force(p)
    _close(o, bo, what="out")
    _close(l, bl, what="lse")


def pin_closed_form_equal_keys(lib):
    """All keys equal: uniform weights, out = mean of V^ over the causal key set."""
    p = _small(17, num_seqs=2, context_lens=[30, 19], q_lens=[3, 1])
    k = p.k_cache.copy()
    k[:] = k[0, 0, 0]
    ks = np.full_like(p.k_scale, 0.01)
    p = _mutate(p, k_cache=k, k_scale=ks)
    o, l = lib.decode(p)
    V = _dequant_cache(p, "v").numpy()
    for r in range(p.num_seqs):
        ql = p.q_lens[r]
        for tok in range(ql):
            n = int(p.context_lens[r]) - ql + tok + 1
            pos = np.arange(n)
            vh = V[p.block_table[r, pos // p.page_size], 0, pos % p.page_size]
            row = p.cu_seqlens_q[r] + tok
            for i in range(p.group_size):
                assert np.max(np.abs(o[row, i] - vh.mean(axis=0))) < TOL


def pin_closed_form_zero_query(lib):
    """q = 0: every score is 0, out = mean of V^, lse = log(n)."""
    p = _small(18, context_lens=[23, 1, 64], q_lens=[2, 1, 1])
    p = _mutate(p, q=np.zeros_like(p.q))
    o, l = lib.decode(p)
    V = _dequant_cache(p, "v").numpy()
    for r in range(p.num_seqs):
        ql = p.q_lens[r]
        for tok in range(ql):
            n = int(p.context_lens[r]) - ql + tok + 1
            pos = np.arange(n)
            vh = V[p.block_table[r, pos // p.page_size], 0, pos % p.page_size].mean(axis=0)
            row = p.cu_seqlens_q[r] + tok
            assert np.max(np.abs(o[row] - vh[None])) < TOL
            assert np.max(np.abs(l[row] - np.log(n))) < TOL


def pin_closed_form_one_and_two_keys(lib):
    """One key: out = V^[0], lse = its score.  Two keys: logistic weights."""
    p = _small(19, num_seqs=2, context_lens=[1, 2], q_lens=[1, 1])
    o, l = lib.decode(p)
    K, V, Q = (_dequant_cache(p, "k").numpy(), _dequant_cache(p, "v").numpy(),
               _q64(p).numpy())
    b0 = p.block_table[0, 0]
    s = Q[0] @ K[b0, 0, 0] * p.sm_scale
    assert np.max(np.abs(o[0] - V[b0, 0, 0][None])) < TOL
    assert np.max(np.abs(l[0] - s)) < TOL
    b1 = p.block_table[1, 0]
    s0 = Q[1] @ K[b1, 0, 0] * p.sm_scale
    s1 = Q[1] @ K[b1, 0, 1] * p.sm_scale
    w1 = 1.0 / (1.0 + np.exp(s0 - s1))
    want = (1 - w1)[:, None] * V[b1, 0, 0][None] + w1[:, None] * V[b1, 0, 1][None]
    assert np.max(np.abs(o[1] - want)) < TOL
    assert np.max(np.abs(l[1] - np.logaddexp(s0, s1))) < TOL


def pin_invariant_folded_scales(lib):
    """Per-token K scale folded into the score column and V scale into P (vLLM PR 52060,
    "Suggested Fix") equals explicit per-element dequantisation."""
    p = _small(20, context_lens=[45, 12, 31], q_lens=[1, 2, 1])
    o, _ = lib.decode(p)
    codes_k = torch.from_numpy(p.k_cache).view(torch.float8_e4m3fn).to(torch.float64)
    codes_v = torch.from_numpy(p.v_cache).view(torch.float8_e4m3fn).to(torch.float64)
    ks = torch.from_numpy(p.k_scale).to(torch.float64)
    vs = torch.from_numpy(p.v_scale).to(torch.float64)
    Q = _q64(p)
    for r in range(p.num_seqs):
        ql = p.q_lens[r]
        L = int(p.context_lens[r])
        pos = torch.arange(L)
        phys = torch.from_numpy(p.block_table[r]).long()[pos // p.page_size]
        sl = pos % p.page_size
        for tok in range(ql):
            n = L - ql + tok + 1
            row = p.cu_seqlens_q[r] + tok
            raw = Q[row] @ codes_k[phys[:n], 0, sl[:n]].T                  # [g, n]
            s = raw * (ks[phys[:n], 0, sl[:n]] * p.sm_scale)[None]
            w = torch.softmax(s, dim=-1) * vs[phys[:n], 0, sl[:n]][None]
            want = w @ codes_v[phys[:n], 0, sl[:n]]
            assert np.max(np.abs(o[row] - want.numpy())) < TOL


def pin_invariant_unit_scales_bf16(lib):
    """Unit per-token scales with bf16-exact values equal the BF16-KV run exactly."""
    p = _small(21, context_lens=[29, 16, 8], q_lens=[1, 1, 2])
    p8 = _mutate(p, k_scale=np.ones_like(p.k_scale), v_scale=np.ones_like(p.v_scale))
    kb = synth.bf16_bits(synth.e4m3_values(p.k_cache))
    vb = synth.bf16_bits(synth.e4m3_values(p.v_cache))
    pb = _mutate(p8, kv_dtype="bf16", scale_mode="none", k_cache=kb, v_cache=vb,
                 k_scale=None, v_scale=None)
    o8, l8 = lib.decode(p8)
    ob, lb = lib.decode(pb)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def pin_invariant_ragged_equals_uniform(lib):
    """A ragged batch equals, row by row, the uniform batches of its pieces."""
    p = _small(22, num_seqs=4, context_lens=[40, 33, 51, 20], q_lens=[4, 4, 6, 2])
    o, l = lib.decode(p)
    for r in range(p.num_seqs):
        one = _mutate(p, num_seqs=1, block_table=p.block_table[r:r + 1],
                      context_lens=p.context_lens[r:r + 1],
                      cu_seqlens_q=np.array([0, p.q_lens[r]], dtype=np.int32),
                      q=p.q[p.cu_seqlens_q[r]:p.cu_seqlens_q[r + 1]], uniform_q_len=p.q_lens[r])
        o1, l1 = lib.decode(one)
        a, b = p.cu_seqlens_q[r], p.cu_seqlens_q[r + 1]
        assert np.array_equal(o[a:b], o1) and np.array_equal(l[a:b], l1)


def pin_invariant_sparse_all_pages_is_dense(lib):
    p = _small(23, context_lens=[70, 16, 33], q_lens=[1, 2, 1])
    npg = (p.context_lens + p.page_size - 1) // p.page_size
    sel = np.full((p.num_seqs, int(npg.max())), -1, dtype=np.int32)
    rng = np.random.default_rng(5)
    for r in range(p.num_seqs):
        sel[r, :npg[r]] = rng.permutation(npg[r])
    ps = _mutate(p, selected=sel, num_selected=npg.astype(np.int32))
    _close(lib.decode(ps)[0], lib.decode(p)[0], tol=1e-13, what="out")
    _close(lib.decode(ps)[1], lib.decode(p)[1], tol=1e-13, what="lse")


def pin_invariant_prefill_as_decode_is_one_ragged_request(lib):
    """A prefill chunk run as one q_len-1 request per token (contexts prefix + t + 1, the
    sequence's block table shared) equals the same chunk as one request with q_len T and
    context prefix + T, row by row: the cutoff L - q_len + tok + 1 gives each row the
    same keys (ROCm/ATOM PR 2614, per-token-as-decode prefill on the decode contract)."""
    pa = synth.prefill_as_decode(51, 40, 30, page_size=16)
    T = pa.num_seqs
    pb = _mutate(pa, num_seqs=1, block_table=pa.block_table[:1],
                 context_lens=np.array([30 + T], dtype=np.int32),
                 cu_seqlens_q=np.array([0, T], dtype=np.int32), uniform_q_len=None)
    oa, la = lib.decode(pa, threads=2)
    ob, lb = lib.decode(pb, threads=2)
    _close(oa, ob, what="prefill rows vs one ragged request")
    _close(la, lb, what="lse")


def pin_invariant_scalar_is_uniform_per_token(lib):
    p = _small(24, scale_mode="scalar")
    ks = np.full((p.num_pages, 1, p.page_size), np.float32(p.k_scale_scalar), dtype=np.float32)
    vs = np.full((p.num_pages, 1, p.page_size), np.float32(p.v_scale_scalar), dtype=np.float32)
    p2 = _mutate(p, scale_mode="per_token", k_scale=ks, v_scale=vs,
                 k_scale_scalar=float(np.float32(p.k_scale_scalar)),
                 v_scale_scalar=float(np.float32(p.v_scale_scalar)))
    p1 = _mutate(p, k_scale_scalar=float(np.float32(p.k_scale_scalar)),
                 v_scale_scalar=float(np.float32(p.v_scale_scalar)))
    assert np.array_equal(lib.decode(p1)[0], lib.decode(p2)[0])


def _golden_rowmap():
    path = os.path.join(GOLDEN, "rowmap_4_4_6_2.txt")
    rows = []
    meta = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if "=" in line:
                k, v = line.split("=", 1)
                meta[k.strip()] = [int(x) for x in v.split(",")]
                continue
            rows.append([int(x) for x in line.split()])
    return meta, np.array(rows)


def pin_golden_ragged_4_4_6_2(lib):
    """The page's ragged batch [4, 4, 6, 2]: 16 rows, divisible by 4 yet ragged.  The
    oracle's key sets follow the fixture's (request, tok, cutoff) per row."""
    meta, rows = _golden_rowmap()
    ql, L = meta["q_lens"], meta["context_lens"]
    p = _small(25, num_seqs=4, context_lens=L, q_lens=ql)
    assert p.num_rows == 16 and p.num_rows % 4 == 0
    for row, r, tok, cut in rows:
        assert p.cu_seqlens_q[r] + tok == row
        keys = lib.key_positions(p, r, tok)
        assert np.array_equal(keys, np.arange(cut)), (row, r, tok, cut)
    # the division map the page warns about disagrees on some rows of this batch
    div = [(row // 4, row % 4) for row in range(16)]
    assert any((r, t) != d for (_, r, t, _), d in zip(rows, div))


def pin_golden_row_map(lib):
    """oracle.row_map (the reference of the device row-map test) against the fixture's
    hand-written (request, tok, cutoff) rows of the page's [4, 4, 6, 2] batch, and, on a
    seeded ragged batch with an empty request, every row's cutoff against the length of
    the key set the C oracle attends for that row."""
    from oracle import oracle as O
    meta, rows = _golden_rowmap()
    ql, L = np.array(meta["q_lens"]), np.array(meta["context_lens"])
    cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    rm = O.row_map(cu, L)
    assert np.array_equal(rm, rows[:, 1:]), "row map differs from the fixture"
    assert np.array_equal(np.arange(len(rows)), rows[:, 0])
    ql2 = [3, 0, 1, 5, 2]
    p = _small(28, num_seqs=5, context_lens=[9, 4, 40, 17, 2], q_lens=ql2)
    rm2 = O.row_map(p.cu_seqlens_q, p.context_lens)
    assert rm2.shape == (sum(ql2), 3)
    for row, (r, tok, cut) in enumerate(rm2):
        assert p.cu_seqlens_q[r] <= row < p.cu_seqlens_q[r + 1] and row - p.cu_seqlens_q[r] == tok
        assert cut == lib.key_positions(p, int(r), int(tok)).size, (row, r, tok, cut)


def pin_golden_121_rows(lib):
    """30 requests with q_len 4 plus one with q_len 1 give 121 rows (121 = 30*4 + 1);
    each row's key set ends at its own cutoff."""
    ql = [4] * 30 + [1]
    ql[7], ql[30] = 1, 4
    L = [20 + 3 * i for i in range(31)]
    p = synth.make_problem(26, num_seqs=31, context_lens=L, q_lens=ql, page_size=16,
                           head_dim=16, group_size=2)
    assert p.num_rows == 121
    for r in (6, 7, 8, 30):
        for tok in range(ql[r]):
            keys = lib.key_positions(p, r, tok)
            assert keys.size == L[r] - ql[r] + tok + 1 and keys[-1] == keys.size - 1


def pin_golden_q_shape_225280(lib):
    """110 rows of [Hkv=1, g=16, D=128] is the 225280-element query of the page, which
    a [27, 4, 1, 16, 128] reshape (108 rows) cannot hold."""
    assert 110 * 1 * 16 * 128 == 225280 and 27 * 4 * 16 * 128 != 225280
    ql = [4] * 26 + [6]
    assert sum(ql) == 110
    p = synth.make_problem(27, num_seqs=27, context_lens=[8] * 27, q_lens=ql, page_size=16,
                           head_dim=128, group_size=16)
    assert p.q.size == 225280
    o, _ = lib.decode(p)
    assert o.shape == (110, 16, 128)


# ------------------------------------------------ log-sum-exp merge of a split context

def _split_parts(p, nparts, rng):
    """Each request's logical pages cut into nparts contiguous blocks (some may be empty):
    one sparse problem per block, selecting exactly that block."""
    npg = (p.context_lens.astype(np.int64) + p.page_size - 1) // p.page_size
    stride = max(int(npg.max()), 1)
    cuts = []
    for r in range(p.num_seqs):
        c = np.sort(rng.integers(0, npg[r] + 1, size=nparts - 1))
        cuts.append(np.concatenate([[0], c, [npg[r]]]))
    parts = []
    for i in range(nparts):
        sel = np.full((p.num_seqs, stride), -1, dtype=np.int32)
        ns = np.zeros(p.num_seqs, dtype=np.int32)
        for r in range(p.num_seqs):
            pages = np.arange(cuts[r][i], cuts[r][i + 1], dtype=np.int32)
            sel[r, :pages.size] = rng.permutation(pages)
            ns[r] = pages.size
        parts.append(_mutate(p, selected=sel, num_selected=ns))
    return parts


def pin_lse_merge_split_equals_whole(lib):
    """Attention over a request's whole key set equals the log-sum-exp merge of the
    attentions over disjoint parts of it (contiguous page blocks, some empty, with ragged
    q_len, the causal cutoff, partial last pages and two KV heads), for the outputs and
    the lse."""
    p = _small(29, num_seqs=4, context_lens=[70, 33, 5, 100], q_lens=[3, 1, 2, 4],
               num_kv_heads=2)
    rng = np.random.default_rng(3)
    for nparts in (2, 3, 5):
        parts = _split_parts(p, nparts, rng)
        outs, lses = zip(*[lib.decode(q) for q in parts])
        mo, ml = lib.lse_merge(np.stack(outs), np.stack(lses))
        wo, wl = lib.decode(p)
        _close(mo, wo, 1e-12, f"merged output ({nparts} parts)")
        _close(ml, wl, 1e-12, f"merged lse ({nparts} parts)")


def pin_lse_merge_closed_forms(lib):
    """One part is returned as it is; a part with lse -inf is ignored; two parts with equal
    lse give the mean and lse + log 2, also at lse 1000 (the maximum is taken out before
    exp); parts weighted e^1 : 1 give that mix; no finite part gives zeros and -inf."""
    rng = np.random.default_rng(8)
    o = rng.standard_normal((3, 2, 5, 8))
    l = rng.standard_normal((3, 2, 5)) * 3
    mo, ml = lib.lse_merge(o[:1], l[:1])
    _close(mo, o[0], 0.0, "one part")
    _close(ml, l[0], 0.0, "one part lse")
    l2 = l.copy()
    l2[1] = -np.inf
    mo, ml = lib.lse_merge(o[:2], l2[:2])
    _close(mo, o[0], 1e-15, "empty part ignored")
    for base in (0.0, 1000.0):
        le = np.full((2, 2, 5), base)
        mo, ml = lib.lse_merge(o[:2], le)
        _close(mo, (o[0] + o[1]) / 2, 1e-14, f"equal lse {base}")
        _close(ml, le[0] + np.log(2.0), 1e-12, f"equal lse {base}: lse")
    lw = np.stack([np.full((2, 5), 1.0), np.zeros((2, 5))])
    mo, _ = lib.lse_merge(o[:2], lw)
    e = np.e
    _close(mo, (e * o[0] + o[1]) / (e + 1), 1e-14, "weights e : 1")
    mo, ml = lib.lse_merge(o[:2], np.full((2, 2, 5), -np.inf))
    assert np.all(mo == 0) and np.all(np.isneginf(ml)), "no finite part"


# ---------------------------------------------------------- KV quantise-and-write (producer)

def _finite_code_values():
    """Values of the 254 finite e4m3fn codes, through torch's decoding (pinned above)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    fin = ~np.isnan(vals)
    return np.arange(256)[fin], vals[fin]


def _brute_nearest_code(x, codes, vals):
    """Nearest finite code of x's sign by exhaustive search; ties go to the even code."""
    if abs(x) > 448.0:
        return 0x7E | (0x80 if x < 0 else 0)
    neg = np.signbit(x)
    m = ((codes & 0x80) != 0) == neg
    c, v = codes[m], vals[m]
    d = np.abs(v - x)
    best = d.min()
    cand = c[d == best]
    even = cand[(cand & 1) == 0]
    return int(even[0] if even.size else cand[0])


def _encode_probe_values():
    codes, vals = _finite_code_values()
    pos = np.unique(vals[vals >= 0])
    mids = (pos[:-1] + pos[1:]) / 2                       # exact ties
    ulp = np.spacing(mids.astype(np.float32)).astype(np.float64)
    rng = np.random.default_rng(11)
    rand = np.exp2(rng.uniform(-12, 9.2, 3000)).astype(np.float32).astype(np.float64)
    xs = np.concatenate([pos, mids, mids - ulp, mids + ulp, rand, [449.0, 463.9, 1e6]])
    xs = xs.astype(np.float32).astype(np.float64)
    return np.concatenate([xs, -xs])


def pin_e4m3_encode_is_nearest(lib):
    """The encoder returns the nearest e4m3fn code (ties to even, saturating at 448),
    checked by exhaustive search over the 254 finite codes."""
    codes, vals = _finite_code_values()
    for x in _encode_probe_values():
        want = _brute_nearest_code(float(x), codes, vals)
        got = lib.enc_e4m3(float(x))
        assert got == want, f"enc({x!r}) = {got:#x}, nearest is {want:#x}"


def pin_e4m3_encode_matches_torch(lib):
    """Within [-464, 464] the encoder agrees with torch's float32 -> float8_e4m3fn cast."""
    xs = _encode_probe_values()
    xs = xs[np.abs(xs) <= 464.0]
    ref = torch.from_numpy(xs.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    got = np.array([lib.enc_e4m3(float(x)) for x in xs], dtype=np.uint8)
    assert np.array_equal(got, ref.numpy()), "encoder differs from torch's cast"


def _kv_case(T=6, Hkv=2, D=128, ps=16, P=5, seed=21):
    rng = np.random.default_rng(seed)
    k = synth.bf16_bits(rng.standard_normal((T, Hkv, D)).astype(np.float32) * 3)
    v = synth.bf16_bits(rng.standard_normal((T, Hkv, D)).astype(np.float32) * 0.01)
    kc = np.full((P, Hkv, ps, D), 0xA5, dtype=np.uint8)
    vc = np.full((P, Hkv, ps, D), 0x5A, dtype=np.uint8)
    ks = np.full((P, Hkv, ps), -7.0, dtype=np.float32)
    vs = np.full((P, Hkv, ps), -9.0, dtype=np.float32)
    return k, v, kc, vc, ks, vs


def _bf16_of(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def pin_quantize_write_closed_forms(lib):
    """Closed forms of the per-token quantiser and the slot placement:
    - a row of e4m3 values times a power of two, whose largest magnitude is 448 times it,
      comes back as exactly those codes, with that power of two as its scale;
    - an all-zero row gives scale 0 and zero codes;
    - a row with one nonzero value a gives scale |a| / 448 (fp32) and the code of +-448;
    - slot s lands at page s // page_size, offset s % page_size, for every KV head; a slot
      of -1 and a slot past the cache change nothing, and the latter is counted."""
    T, Hkv, D, ps, P = 6, 2, 128, 16, 5
    k, v, kc, vc, ks, vs = _kv_case(T, Hkv, D, ps, P)
    codes, vals = _finite_code_values()
    rng = np.random.default_rng(5)
    exact_codes = rng.choice(codes[np.abs(vals) < 448], size=D).astype(np.uint8)
    exact_codes[17] = 0xFE                                # -448 somewhere in the row
    s = 2.0 ** -5
    row = np.array([lib.dec_e4m3(int(c)) for c in exact_codes]) * s
    k[0, 1] = synth.bf16_bits(row.astype(np.float32))
    k[1, 0] = 0
    one = np.zeros(D, dtype=np.float32)
    one[40] = -3.140625                                   # bf16-exact
    v[2, 1] = synth.bf16_bits(one)
    # exact midpoints between neighbouring e4m3 values (times 2^-7, with 448 * 2^-7 as the
    # row maximum): the quotient is the midpoint itself, so each code is the even neighbour
    pos = np.unique(vals[(vals > 0) & (vals < 448)])
    mids = ((pos[:-1] + pos[1:]) / 2)[::3][:D - 1]
    mid_row = np.zeros(D, dtype=np.float64)
    mid_row[:mids.size] = mids * np.where(np.arange(mids.size) % 2 == 0, 1.0, -1.0)
    mid_row[D - 1] = 448.0
    mid_codes = np.array([_brute_nearest_code(float(x), codes, vals) for x in mid_row], np.uint8)
    k[5, 0] = synth.bf16_bits((mid_row * 2.0 ** -7).astype(np.float32))
    assert np.array_equal(_bf16_of(k[5, 0]).astype(np.float64), mid_row * 2.0 ** -7)
    slots = np.array([3 * ps + 7, 0, 4 * ps + ps - 1, -1, P * ps + 2, ps + 1], dtype=np.int64)
    kc0, vc0, ks0, vs0 = kc.copy(), vc.copy(), ks.copy(), vs.copy()
    bad = lib.kv_quantize_write(k, v, slots, kc, vc, ks, vs)
    assert bad == 1, "the slot past the cache is not counted"
    # token 0, head 1: exact codes and scale
    assert np.array_equal(kc[3, 1, 7], exact_codes), "exact e4m3 row not reproduced"
    assert ks[3, 1, 7] == np.float32(s), "power-of-two scale not reproduced"
    # token 1, head 0: zero row
    assert ks[0, 0, 0] == 0.0 and not kc[0, 0, 0].any(), "zero row"
    # token 5, head 0: midpoints go to the even neighbour
    assert np.array_equal(kc[1, 0, 1], mid_codes), "ties not rounded to the even code"
    # token 2, head 1: one nonzero V value
    assert vs[4, 1, ps - 1] == np.float32(np.float32(3.140625) / np.float32(448.0))
    want = np.zeros(D, dtype=np.uint8)
    want[40] = 0xFE
    assert np.array_equal(vc[4, 1, ps - 1], want), "single-value row"
    # placement: exactly the rows of the written slots changed
    written = {(3, 7), (0, 0), (4, ps - 1), (1, 1)}
    for pg in range(P):
        for o in range(ps):
            for h in range(Hkv):
                same = (np.array_equal(kc[pg, h, o], kc0[pg, h, o]) and
                        np.array_equal(vc[pg, h, o], vc0[pg, h, o]) and
                        ks[pg, h, o] == ks0[pg, h, o] and vs[pg, h, o] == vs0[pg, h, o])
                assert same == ((pg, o) not in written), f"placement at page {pg} slot {o}"


def pin_quantize_write_round_trip(lib):
    """Dequantised codes (code value x scale) lie within half an e4m3 step of the input,
    every row's largest magnitude maps to +-448, and K and V rows are kept apart."""
    T, Hkv, D, ps, P = 6, 2, 128, 16, 5
    k, v, kc, vc, ks, vs = _kv_case(T, Hkv, D, ps, P, seed=33)
    slots = np.arange(T, dtype=np.int64) * 3 + 1
    lib.kv_quantize_write(k, v, slots, kc, vc, ks, vs)
    dec = np.array([lib.dec_e4m3(c) if c not in (0x7F, 0xFF) else np.nan for c in range(256)])
    for t in range(T):
        pg, o = divmod(int(slots[t]), ps)
        for h in range(Hkv):
            for new, cache, sc in ((k, kc, ks), (v, vc, vs)):
                x = _bf16_of(new[t, h]).astype(np.float64)
                scale = float(sc[pg, h, o])
                y = dec[cache[pg, h, o]] * scale
                amax = np.abs(x).max()
                assert np.isclose(scale, amax / 448.0, rtol=2 ** -23), "scale is not amax / 448"
                assert abs(np.abs(y).max() - amax) <= amax * 2 ** -20, "amax element not at 448"
                # e4m3 has 3 mantissa bits: error <= 2^-4 relative, or half a subnormal step
                err = np.abs(y - x)
                bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scale) * (1 + 1e-6)
                assert np.all(err <= bound), "dequantised value too far from the input"


def _nearest_code_exact(q, neg):
    """Nearest finite e4m3fn code to the non-negative rational q (a Fraction), with the
    sign bit `neg`, by exact comparison against all 127 non-negative finite codes; ties
    go to the even code, and q above 448 saturates to 448."""
    from fractions import Fraction
    codes, vals = _finite_code_values()
    sgn = 0x80 if neg else 0x00
    if q > 448:
        return 0x7E | sgn
    best, cand = None, []
    for c, v in zip(codes, vals):
        if c & 0x80:
            continue
        d = abs(Fraction(float(v)) - q)
        if best is None or d < best:
            best, cand = d, [int(c)]
        elif d == best:
            cand.append(int(c))
    even = [c for c in cand if (c & 1) == 0]
    return (even[0] if even else cand[0]) | sgn


def _near_tie_rows():
    """(amax, x) pairs of bf16 values, x <= amax, for which 448 x / amax is exactly an
    e4m3 rounding midpoint.  With the stored scale s = fl32(amax / 448) the quotient x / s
    is then a hair above or below that midpoint (as s was rounded up or down), so the
    code is decided by s's rounding error: exactly where the fp32 product
    x * fl32(448 / amax) and the fp32 quotient fl32(x / s) can land on the midpoint, or
    on its other side, and pick the other neighbour."""
    from fractions import Fraction
    _, vals = _finite_code_values()
    pos = sorted({Fraction(float(v)) for v in vals if 0 < v <= 448})
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    out = []
    for A in range(128, 256):                       # amax mantissas (exponent 0: amax in [1, 2))
        amax = Fraction(A, 128)
        for m in mids:
            x = m * amax / 448
            num, den = x.numerator, x.denominator
            if den & (den - 1) or num.bit_length() > 8 or x > amax:
                continue                            # not a bf16 value below amax
            out.append((amax, x))
    return out


def pin_quantize_write_exact_quotient(lib):
    """Each code is the e4m3 rounding of the exact real quotient x / scale, with scale the
    stored fp32 amax / 448 (the recipe scale = amax / 448), checked with exact rational
    arithmetic on rows built so that x / scale sits next to a rounding midpoint.  The
    cases must include some where the fp32 product with 448 / amax and the fp32 quotient
    each pick the other code, so that both shortcuts are told apart from the reading."""
    from fractions import Fraction
    pairs = _near_tie_rows()
    assert len(pairs) >= 64, "too few near-tie rows"
    D, ps = 128, 16
    # one row per amax: its pairs' x values, and amax itself as the row's maximum
    rows = {}
    for i, (amax, x) in enumerate(pairs):
        rows.setdefault(amax, []).append((i, x))
    xs = np.zeros((len(rows), 1, D), dtype=np.float32)
    meta = []
    for t, (amax, items) in enumerate(sorted(rows.items())):
        items = items[:D - 1]
        for d, (i, x) in enumerate(items):
            xs[t, 0, d] = float(x) * (-1.0 if i % 3 == 1 else 1.0)
        xs[t, 0, D - 1] = float(amax)
        meta.append(amax)
    T = xs.shape[0]
    k = synth.bf16_bits(xs)
    assert np.array_equal(_bf16_of(k).astype(np.float64), xs.astype(np.float64)), "not bf16-exact"
    v = k.copy()
    P = (T + ps - 1) // ps
    kc = np.zeros((P, 1, ps, D), np.uint8)
    vc, ks, vs = kc.copy(), np.zeros((P, 1, ps), np.float32), np.zeros((P, 1, ps), np.float32)
    slots = np.arange(T, dtype=np.int64)
    lib.kv_quantize_write(k, v, slots, kc, vc, ks, vs)
    prod_differs = quot32_differs = 0
    for t in range(T):
        pg, o = divmod(t, ps)
        x = xs[t, 0].astype(np.float64)
        s32 = np.float32(np.float32(meta[t]) / np.float32(448.0))
        assert ks[pg, 0, o] == s32, "stored scale is not fl32(amax / 448)"
        S = Fraction(float(s32))
        inv32 = np.float32(np.float32(448.0) / np.float32(meta[t]))
        for d in range(D):
            if x[d] == 0.0:
                continue
            want = _nearest_code_exact(abs(Fraction(float(x[d])) / S), x[d] < 0)
            got = int(kc[pg, 0, o, d])
            assert got == want, f"row {t} d {d}: code {got:#x}, exact quotient gives {want:#x}"
            prod = float(np.float32(np.float32(x[d]) * inv32))
            quot = float(np.float32(np.float32(x[d]) / s32))
            prod_differs += _nearest_code_exact(abs(Fraction(prod)), prod < 0) != want
            quot32_differs += _nearest_code_exact(abs(Fraction(quot)), quot < 0) != want
    assert prod_differs > 0 and quot32_differs > 0, (prod_differs, quot32_differs)


# ------------------------------------------------ indexer block score and top-k selection

def _index_brute(ip):
    """Scores and selection by materialised fp64 torch: the keys decoded through torch's
    float8_e4m3fn, s = sm_scale * log2(e) * q . k, a block's score the base-2 log-sum-exp of
    its attended (head, token) scores, and the selection by Python's sort."""
    q = torch.from_numpy(ip.q.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    kc = torch.from_numpy(ip.k_cache).view(torch.float8_e4m3fn).to(torch.float64)
    if ip.k_scale is not None:
        kc = kc * torch.from_numpy(ip.k_scale).to(torch.float64)[..., None]
    ps = ip.k_cache.shape[1]
    sel_all, n_all, S_all = [], [], []
    for r in range(len(ip.context_lens)):
        L = int(ip.context_lens[r])
        r0, r1 = int(ip.cu_seqlens_q[r]), int(ip.cu_seqlens_q[r + 1])
        ql = r1 - r0
        for tok in range(ql):
            lim = max(0, min(L, L - ql + tok + 1))
            nb = (lim + ps - 1) // ps
            S = {}
            for b in range(nb):
                keys = kc[int(ip.block_table[r, b])][: min(ps, lim - b * ps)]   # [n, D]
                sc = (q[r0 + tok] @ keys.T) * ip.sm_scale / np.log(2.0)       # [H, n], log2 units
                S[b] = float(torch.logsumexp(sc.reshape(-1) * np.log(2.0), 0) / np.log(2.0))
            order = ([nb - 1] if nb else []) + sorted((b for b in S if b != nb - 1),
                                                       key=lambda b: (-S[b], b))
            sel = order[: ip.topk]
            sel_all.append(sel + [-1] * (ip.topk - len(sel)))
            n_all.append(len(sel))
            S_all.append(S)
    return np.array(sel_all, dtype=np.int32).reshape(-1, ip.topk), np.array(n_all), S_all


def pin_index_topk_brute_force(lib):
    """Indexer scores and selection against a materialised torch computation (two index
    heads, per-token key scales, ragged q_len with the causal cutoff, a partial last page)."""
    ip = synth.index_problem(31, [300, 1000, 37, 129], [1, 3, 2, 1], index_heads=2,
                             page_size=16, topk=8)
    sel, n, S = lib.index_topk(ip)
    bsel, bn, bS = _index_brute(ip)
    assert np.array_equal(n, bn), "selection counts differ"
    assert np.array_equal(sel, bsel), "selected pages differ"
    for row, Sr in enumerate(bS):
        for b, v in Sr.items():
            assert abs(S[row, b] - v) <= 1e-9 * max(1.0, abs(v)), f"score row {row} page {b}"
        assert np.all(np.isneginf(np.delete(S[row], list(Sr.keys())))), "non-candidate scored"


def pin_index_topk_scalar_keys(lib):
    """The same without per-token key scales (codes read at scale 1)."""
    ip = synth.index_problem(32, [500, 64], [2, 1], index_heads=1, page_size=32, topk=5,
                             per_token_scale=False)
    sel, n, _ = lib.index_topk(ip)
    bsel, bn, _ = _index_brute(ip)
    assert np.array_equal(sel, bsel) and np.array_equal(n, bn)


def pin_index_topk_closed_forms(lib):
    """q = 0: every attended (head, token) scores 0, so a page's score is log2 of its count
    of attended pairs; the full pages tie and the selection is the last attended page, then
    pages 0, 1, 2, ...  A page count below topk selects every page."""
    ip = synth.index_problem(33, [16 * 10 + 5, 40], [1, 2], index_heads=3, page_size=16,
                             topk=4, zero_q=True)
    sel, n, S = lib.index_topk(ip)
    assert list(sel[0]) == [10, 0, 1, 2] and n[0] == 4
    assert S[0, 0] == np.log2(3 * 16) and S[0, 10] == np.log2(3 * 5)
    # request 1: L 40, q_len 2 -> limits 39 and 40 -> 3 pages each
    assert list(sel[1]) == [2, 0, 1, -1] and n[1] == 3
    assert list(sel[2]) == [2, 0, 1, -1] and S[1, 2] == np.log2(3 * 7) and S[2, 2] == np.log2(3 * 8)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
