"""Host side of a context split across GPUs, on CPU (no GPU): the page partition, and the
exchange of the ranks' partials on two gloo ranks.  Each rank's partial is the oracle's
attention over the pages rank_pages gives it (what pa_decode computes there on a GPU);
after gather_partials the oracle's log-sum-exp merge must reproduce the oracle's
attention over the whole context, on every rank."""
import dataclasses
import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

from paged_fp8_kv_04_gb300 import context_parallel as cp  # noqa: E402
from paged_fp8_kv_04_gb300 import synth  # noqa: E402


def test_rank_pages_cover_every_page_once_in_contiguous_blocks():
    L = np.array([0, 1, 127, 128, 129, 5000, 131072, 300])
    for ps in (16, 128):
        for world in (1, 2, 3, 4, 8):
            n = (L + ps - 1) // ps
            seen = [[] for _ in L]
            for rank in range(world):
                sel, cnt = cp.rank_pages(L, ps, world, rank)
                assert sel.dtype == np.int32 and cnt.dtype == np.int32
                assert sel.shape[1] >= max(int(cnt.max()), 1)
                for r in range(L.size):
                    got = sel[r, :cnt[r]]
                    assert np.all(sel[r, cnt[r]:] == -1)
                    if got.size:
                        assert np.array_equal(got, np.arange(got[0], got[0] + got.size))
                    seen[r].extend(got.tolist())
                    assert cnt[r] <= cp.max_rank_pages(int(L.max()), ps, world)
            for r in range(L.size):
                assert sorted(seen[r]) == list(range(n[r])), (ps, world, r)
                sizes = [((n[r] * (k + 1)) // world) - (n[r] * k) // world for k in range(world)]
                assert max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    return synth.make_problem(90, num_seqs=3, context_lens=[700, 129, 2000], q_lens=[1, 3, 2],
                              page_size=16, num_kv_heads=2)


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from oracle import oracle as O
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = _problem()
        sel, cnt = cp.rank_pages(p.context_lens, p.page_size, world, rank)
        shard = dataclasses.replace(p, selected=sel, num_selected=cnt)
        out, lse = O.decode(shard)                      # this rank's partial
        po, pl = cp.gather_partials(torch.from_numpy(out.astype(np.float32)),
                                    torch.from_numpy(lse.astype(np.float32)))
        mo, ml = O.lse_merge(po.numpy().astype(np.float64), pl.numpy().astype(np.float64))
        ref, ref_lse = O.decode(p)
        q.put((rank, tuple(po.shape), float(np.abs(mo - ref).max()),
               float(np.abs(ml - ref_lse)[np.isfinite(ref_lse)].max())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_gather_partials_that_merge_to_the_whole_context():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(300)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    p = _problem()
    for rank, (r, shape, err, lerr) in enumerate(got):
        assert r == rank
        assert shape == (2, p.num_rows, p.num_kv_heads * p.group_size, p.head_dim)
        # fp32 partials on the wire: the merge is as exact as their rounding allows
        assert err <= 1e-6 and lerr <= 1e-5, (err, lerr)
