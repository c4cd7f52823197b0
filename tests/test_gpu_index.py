"""The indexer's block score and top-k selection against the oracle (needs a GPU).

Page scores are fp32 sums on the GPU and fp64 in the oracle, so they are compared within
a tolerance in log2 units.  The selection is an integer result decided by those scores:
where the oracle's order has no near-tie the pages must match exactly; otherwise the
GPU's choice must be a valid top-k under the tolerance (the forced last page first, no
page left out that scores clearly above one taken, an order that never rises by more
than the tolerance).
"""
import dataclasses

import numpy as np
import pytest
import torch

from gpu_util import compare
from oracle import oracle as O
from paged_fp8_kv_04_gb300 import binding as B
from paged_fp8_kv_04_gb300 import device as dv
from paged_fp8_kv_04_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 2e-3  # log2 units


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def run_gpu(ip, status=True, scales_4b_aligned=False):
    """scales_4b_aligned: k_scale starts 4 bytes past a 16-byte boundary (the contract asks
    for 4-byte alignment only)."""
    dev = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q = dev(ip.q.view(np.int16))
    kc = dev(ip.k_cache)
    ks = None if ip.k_scale is None else dev(ip.k_scale)
    if ks is not None and scales_4b_aligned:
        buf = torch.empty(ks.numel() + 4, dtype=torch.float32, device="cuda")
        ks = buf[1:1 + ks.numel()].view(ks.shape)
        ks.copy_(dev(ip.k_scale))
        assert ks.data_ptr() % 16 == 4
    bt, L, cu = dev(ip.block_table), dev(ip.context_lens), dev(ip.cu_seqlens_q)
    R, stride = ip.num_rows, ip.block_table.shape[1]
    sel = torch.full((R, ip.topk), -7, dtype=torch.int32, device="cuda")
    nsel = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((R, stride), 12345.0, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    maxq = int(np.diff(ip.cu_seqlens_q).max())
    a = B.index_args(q, kc, ks, bt, L, cu, sel, nsel, scores, topk=ip.topk, max_q_len=maxq,
                     sm_scale=ip.sm_scale, status=st)
    B.index_topk(a, device=torch.device("cuda"))
    torch.cuda.synchronize()
    return sel.cpu().numpy(), nsel.cpu().numpy(), scores.cpu().numpy(), int(st.item())


def sub(ip, reqs):
    """The same index problem restricted to requests `reqs` (shared cache and tables)."""
    reqs = np.asarray(reqs)
    ql = np.diff(ip.cu_seqlens_q)[reqs]
    cu = np.zeros(len(reqs) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    rows = np.concatenate([np.arange(ip.cu_seqlens_q[r], ip.cu_seqlens_q[r + 1]) for r in reqs])
    return dataclasses.replace(ip, q=ip.q[rows], block_table=ip.block_table[reqs],
                               context_lens=ip.context_lens[reqs], cu_seqlens_q=cu), rows


def check_row(g, o, gS, oS, n, what):
    cand = np.isfinite(oS)
    assert np.all(np.isneginf(gS[~cand])), f"{what}: non-candidate pages scored"
    err = np.abs(gS[cand] - oS[cand]).max() if cand.any() else 0.0
    assert err <= TOL, f"{what}: page score off by {err}"
    g, o = list(g[:n]), list(o[:n])
    if g == o:
        return
    assert g[0] == o[0], f"{what}: forced page {g[0]} != {o[0]}"
    assert len(set(g)) == n and all(cand[b] for b in g), f"{what}: invalid selection {g}"
    rest_g = [b for b in g[1:]]
    taken = set(g)
    lowest = min(oS[b] for b in rest_g) if rest_g else np.inf
    left = [oS[b] for b in np.flatnonzero(cand) if b not in taken]
    assert not left or max(left) <= lowest + TOL, f"{what}: a clearly better page left out"
    sc = [oS[b] for b in rest_g]
    assert all(sc[i + 1] <= sc[i] + TOL for i in range(len(sc) - 1)), f"{what}: order rises"


def check(ip, reqs=None, what="", **kw):
    gsel, gn, gS, st = run_gpu(ip, **kw)
    assert st == 0, f"{what}: device flags {st:#x}"
    q, rows = (ip, np.arange(ip.num_rows)) if reqs is None else sub(ip, reqs)
    osel, on, oS = O.index_topk(q)
    assert np.array_equal(gn[rows], on), f"{what}: counts {gn[rows]} vs {on}"
    for i, row in enumerate(rows):
        assert np.all(gsel[row, on[i]:] == -1), f"{what}: padding"
        check_row(gsel[row], osel[i], gS[row], oS[i], on[i], f"{what} row {row}")


@pytest.mark.parametrize("case", ["ragged_two_heads", "page128", "scalar_keys_rh16",
                                  "topk_above_pages"])
def test_index_topk(case):
    if case == "ragged_two_heads":
        ip = synth.index_problem(41, [300, 1000, 37, 129], [1, 3, 2, 1], index_heads=2,
                                 page_size=16, topk=8)
    elif case == "page128":
        ip = synth.index_problem(42, [9000, 131, 20000, 128], [1, 1, 1, 1], page_size=128, topk=16)
    elif case == "scalar_keys_rh16":
        ip = synth.index_problem(43, [2000, 777], [4, 3], index_heads=4, page_size=32, topk=12,
                                 per_token_scale=False)
    else:
        ip = synth.index_problem(44, [100, 64, 16], [1, 2, 1], page_size=16, topk=64)
    check(ip, what=case)


@pytest.mark.parametrize("case", ["ragged_two_heads", "page128"])
def test_index_topk_scales_4b_aligned(case):
    """The same results when the scales are only 4-byte aligned."""
    if case == "ragged_two_heads":
        ip = synth.index_problem(41, [300, 1000, 37, 129], [1, 3, 2, 1], index_heads=2,
                                 page_size=16, topk=8)
    else:
        ip = synth.index_problem(42, [9000, 131, 20000, 128], [1, 1, 1, 1], page_size=128, topk=16)
    check(ip, what=case + " (4-byte aligned scales)", scales_4b_aligned=True)
    a, an, aS, _ = run_gpu(ip)
    b, bn, bS, _ = run_gpu(ip, scales_4b_aligned=True)
    assert np.array_equal(an, bn) and np.array_equal(a, b) and np.array_equal(aS, bS)


def test_index_topk_full_size_sampled():
    """The bench's workload (batch 32, context 131072, q_len 1 and 4, top 64): requests
    0, 5, 17 and 31 (q_len 1, 1, 4, 4) against the oracle."""
    check(synth.index_decode_128k(8), reqs=[0, 5, 17, 31], what="indexer 128K")


def test_index_bad_page_is_flagged():
    ip = synth.index_problem(45, [300, 200], [1, 1], page_size=16, topk=4)
    bt = ip.block_table.copy()
    bt[1, 3] = 10 ** 6
    _, _, _, st = run_gpu(dataclasses.replace(ip, block_table=bt))
    assert st & 0x01, "bad page id not flagged"


def test_selection_feeds_sparse_decode():
    """The indexer's pages, as chosen on the GPU, drive pa_decode's sparse path: the decode
    over them equals the oracle's attention over the same lists."""
    p = synth.make_problem(46, num_seqs=4, context_lens=[700, 333, 1024, 90], q_lens=[1] * 4,
                           page_size=16)
    ip = synth.index_problem(47, p.context_lens, [1] * 4, page_size=16, topk=6,
                             pool_pages=p.k_cache.shape[0])
    ip = dataclasses.replace(ip, block_table=p.block_table)
    gsel, gn, _, st = run_gpu(ip)
    assert st == 0
    q = dataclasses.replace(p, selected=gsel, num_selected=gn)
    d = dv.to_device(q)
    plan = dv.plan_for(q)
    out, _ = dv.run(plan, q, d, lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ref, _ = O.decode(q)
    compare(out.float().cpu().numpy(), ref, "indexer -> sparse decode")


def test_index_degenerate_rows():
    """A request without rows between others (equal cu_seqlens_q entries), a context
    shorter than one page, and a single-page request whose only candidate is forced."""
    ip = synth.index_problem(49, [300, 5, 77, 16], [2, 1, 1, 1], page_size=16, topk=4)
    ql = [2, 0, 1, 1, 1]
    L = np.array([300, 40, 5, 77, 16], dtype=np.int32)
    cu = np.zeros(6, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    bt = np.full((5, ip.block_table.shape[1]), -1, dtype=np.int32)
    bt[[0, 2, 3, 4]] = ip.block_table
    bt[1, :3] = ip.block_table[0, :3]
    ip = dataclasses.replace(ip, block_table=bt, context_lens=L, cu_seqlens_q=cu)
    check(ip, what="degenerate rows")
    sel, n, _ = O.index_topk(ip)
    assert list(n) == [4, 4, 1, 4, 1]
