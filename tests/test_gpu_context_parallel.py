"""A context split across GPUs, emulated on one GPU (needs a GPU): every rank's shard is
decoded here in turn (a sparse pa_decode over its block of pages, fp32 output and lse),
the shards are stacked as the all-gather would deliver them, and pa_lse_merge combines
them.  The merged output must match the oracle's attention over the whole context
(bf16 within max-abs 1e-2, cosine >= 0.9999 per (row, head); lse within 2e-3) and the
one-GPU decode element by element within 1e-3 relative in fp32."""
import numpy as np
import pytest
import torch

from gpu_util import compare, compare_lse, compare_split
from oracle import oracle as O
from paged_fp8_kv_04_gb300 import binding as B
from paged_fp8_kv_04_gb300 import context_parallel as cp
from paged_fp8_kv_04_gb300 import device as dv
from paged_fp8_kv_04_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def split_decode(p, world):
    """(merged bf16, merged fp32, merged lse) of p decoded as `world` shards."""
    d = dv.to_device(p)
    plan = dv.plan_for(p, out_dtype="f32", ragged=True,
                       max_selected_pages=cp.max_rank_pages(int(p.context_lens.max()),
                                                            p.page_size, world))
    kw = dv.call_kwargs(p, d)
    kw.pop("selected_pages"), kw.pop("num_selected")
    outs, lses = [], []
    for rank in range(world):
        o, l = cp.decode_shard(plan, d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                               p.context_lens, world, rank, **kw)
        outs.append(o)
        lses.append(l)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    po, pl = torch.stack(outs), torch.stack(lses)
    bf, lse = cp.merge(po, pl, out_dtype=torch.bfloat16, with_lse=True)
    f32 = cp.merge(po, pl, out_dtype=torch.float32)
    torch.cuda.synchronize()
    return bf.float().cpu().numpy(), f32.cpu().numpy(), lse.cpu().numpy()


def one_gpu(p):
    d = dv.to_device(p)
    plan = dv.plan_for(p, out_dtype="f32")
    out, _ = dv.run(plan, p, d)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("world", [2, 3])
def test_long_context_split_over_ranks(world):
    p = synth.make_problem(91, num_seqs=3, context_lens=[40000, 131072, 9000], q_lens=[1] * 3)
    bf, f32, lse = split_decode(p, world)
    ref, ref_lse = O.decode(p)
    compare(bf, ref, f"{world} shards")
    compare_lse(lse, ref_lse, f"{world} shards")
    compare_split(f32, one_gpu(p), f"{world} shards vs one GPU")


def test_ragged_causal_split_with_empty_shards():
    """Ragged q_len up to 6 with the causal cutoff, pages of 16, short requests whose
    shards are empty on some ranks (their lse is -inf and they are skipped)."""
    p = synth.make_problem(92, num_seqs=5, context_lens=[3000, 6, 700, 33, 16], q_lens=[4, 1, 6, 2, 3],
                           page_size=16, num_kv_heads=2)
    bf, f32, lse = split_decode(p, 4)
    ref, ref_lse = O.decode(p)
    compare(bf, ref, "ragged split")
    compare_lse(lse, ref_lse, "ragged split")
    compare_split(f32, one_gpu(p), "ragged split vs one GPU")


def test_scalar_scales_split():
    p = synth.make_problem(93, num_seqs=2, context_lens=[20000, 5000], q_lens=[1, 1],
                           scale_mode="scalar")
    bf, f32, lse = split_decode(p, 2)
    ref, ref_lse = O.decode(p)
    compare(bf, ref, "scalar split")
    compare_lse(lse, ref_lse, "scalar split")


def test_merge_against_oracle_merge_on_given_partials():
    """pa_lse_merge alone against the oracle's merge, on partials with -inf parts, large
    lse values (1e3, so exp needs the maximum taken out) and 7 parts (the unrolled loop's
    tail)."""
    rng = np.random.default_rng(5)
    P, R, H, D = 7, 5, 16, 128
    po = rng.standard_normal((P, R, H, D)).astype(np.float32)
    pl = (rng.standard_normal((P, R, H)) * 4 + 1000).astype(np.float32)
    pl[rng.random((P, R, H)) < 0.3] = -np.inf
    pl[:, 0, 0] = -np.inf                                   # no finite part at all
    po[np.isinf(pl)] = np.nan                               # an empty part's output is never read
    mo, ml = O.lse_merge(po.astype(np.float64), pl.astype(np.float64))
    tpo, tpl = torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda()
    out = torch.empty((R, H, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((R, H), dtype=torch.float32, device="cuda")
    B.lse_merge(tpo, tpl, out, lse)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    assert np.abs(got - mo).max() <= 1e-5
    compare_lse(lse.cpu().numpy(), ml, "merge lse", tol=1e-4)
    assert np.all(got[0, 0] == 0)
