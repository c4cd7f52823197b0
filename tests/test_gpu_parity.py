"""CUDA path against the fp64 oracle, through the C ABI (needs a GPU).

Bars: bf16 outputs within max-abs 1e-2 of the oracle and cosine >= 0.9999 for every
(row, head) vector, every row of every workload compared (the full-size ones included);
the row map and the page gather bit-exact; split-K against single pass within 1e-3
relative, element by element, in fp32 (the tolerances of the hot path's spec).
"""
import numpy as np
import pytest
import torch

from gpu_util import compare, compare_lse, compare_split, rows_of, subset
from oracle import oracle as O
from paged_fp8_kv_04_gb300 import device as dv
from paged_fp8_kv_04_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def gpu_run(p, out_dtype="bf16", partition_tokens=0, plan=None, tcgen05=False, **kw):
    d = dv.to_device(p)
    plan = plan or dv.plan_for(p, out_dtype=out_dtype, partition_tokens=partition_tokens,
                               tcgen05=tcgen05)
    out, lse = dv.run(plan, p, d, lse=True, **kw)
    torch.cuda.synchronize()
    flags = plan.device_status()
    return out.float().cpu().numpy(), lse.cpu().numpy(), flags


def check_against_oracle(p, what="", rel_rows=False, **kw):
    """Every row of p on the GPU against the oracle."""
    out, lse, flags = gpu_run(p, **kw)
    assert flags == 0, f"{what}: device flags {flags:#x}"
    ref, ref_lse = O.decode(p)
    compare(out, ref, what, rel_rows=rel_rows)
    compare_lse(lse, ref_lse, what, rel=1e-5 if rel_rows else 0.0)
    return out, lse


# ------------------------------------------------------------------------ the workloads

# FP8 plans with one query token may run the tcgen05 kernel (tcgen05=True) instead of
# the default mma.sync kernel; both stay covered.
@pytest.mark.parametrize("tc", [False, True])
def test_tiny_dense_decode(tc):
    check_against_oracle(synth.tiny_dense(0), what=f"tiny dense tcgen05={tc}", tcgen05=tc)


@pytest.mark.parametrize("tc", [False, True])
def test_dense_8k_full_size(tc):
    check_against_oracle(synth.dense_8k(1), what=f"dense 8K tcgen05={tc}", tcgen05=tc)


def test_dense_8k_bf16_control():
    check_against_oracle(synth.dense_8k(1, kv_dtype="bf16"), what="bf16 control")


@pytest.mark.parametrize("mode,tc", [("scalar", False), ("per_token", False), ("scalar", True),
                                     ("per_token", True)])
def test_long_128k_full_size(mode, tc):
    check_against_oracle(synth.long_128k(2, scale_mode=mode), what=f"128K {mode} tcgen05={tc}",
                         tcgen05=tc)


@pytest.mark.parametrize("kv_dtype,tc,q_len", [("fp8", False, 1), ("fp8", True, 1),
                                               ("fp8", False, 2), ("bf16", False, 1)])
def test_nan_codes_in_unattended_slots_stay_unread(kv_dtype, tc, q_len):
    """Slots past the context length in a request's last page hold NaN codes (bytes a
    cache may leave behind); they are masked, so the output must equal the oracle's,
    which never reads them."""
    p = synth.make_problem(11, num_seqs=3, context_lens=[200, 77, 130], q_lens=[q_len] * 3,
                           page_size=64, kv_dtype=kv_dtype)
    nan = 0x7F if kv_dtype == "fp8" else 0x7FC0
    for r in range(p.num_seqs):
        L = int(p.context_lens[r])
        last = int(p.block_table[r, (L - 1) // p.page_size])
        for o in range(L % p.page_size or p.page_size, p.page_size):
            p.v_cache[last, :, o, :] = nan
            p.k_cache[last, :, o, :] = nan
    out, _ = check_against_oracle(p, what=f"NaN slots {kv_dtype} tcgen05={tc} q_len={q_len}",
                                  tcgen05=tc)
    assert np.isfinite(out).all()


@pytest.mark.parametrize("batch", ["A", "B"])
def test_ragged_speculative_decode(batch):
    p = synth.ragged_spec(3, batch)
    if batch == "A":
        assert p.num_rows == 121 and sorted(set(p.q_lens.tolist())) == [1, 4]
    else:
        assert list(p.q_lens) == [4, 4, 6, 2]
    check_against_oracle(p, what=f"ragged {batch}")


def test_sparse_selected_pages_full_size():
    check_against_oracle(synth.sparse_selected(4), what="sparse")


# ------------------------------------------------- per-token scales over a wide range

@pytest.mark.parametrize("tc", [False, True])
def test_per_token_scales_spanning_2e20(tc):
    """Per-token K and V magnitudes of 2^-20 .. 2^20 within every request (each token row
    its own 2^u): the per-token V scale folded into P must neither overflow the P operand
    nor flush it, and the per-token K scale must carry scores of very different size.
    Every output finite, within 1e-2 of the oracle relative to its (row, head)'s scale,
    cosine >= 0.9999 per (row, head)."""
    p = synth.make_problem(70, num_seqs=6, context_lens=[8192, 3000, 129, 1, 5000, 640],
                           q_lens=[1] * 6, kv_mag_log2=20.0)
    assert p.v_scale.max() > 2.0 ** 12 and p.v_scale[p.v_scale > 0].min() < 2.0 ** -26
    check_against_oracle(p, what=f"per-token scales 2^+-20 tcgen05={tc}", rel_rows=True,
                         tcgen05=tc)


def test_per_token_scales_spanning_2e20_ragged_and_split():
    """The same magnitudes with ragged q_len (up to 6) and long requests split across CTAs,
    in fp32 out: the per-warp power of two of P meets the slice and split-K merges."""
    p = synth.make_problem(71, num_seqs=5, context_lens=[40000, 777, 20000, 9, 13000],
                           q_lens=[4, 1, 6, 2, 3], kv_mag_log2=20.0)
    check_against_oracle(p, what="per-token scales 2^+-20 ragged", rel_rows=True,
                         out_dtype="f32")


def test_small_per_token_scales_keep_precision():
    """Every token row at 2^-12 .. 2^-10 of N(0, 1): P must not sink into f16 subnormals
    (a fixed scale of P would flush most of it)."""
    import dataclasses
    p = synth.make_problem(72, num_seqs=4, context_lens=[4096, 200, 9000, 33], q_lens=[1] * 4)
    f = np.float32(2.0 ** -11)
    p = dataclasses.replace(p, k_scale=p.k_scale * f, v_scale=p.v_scale * f)
    check_against_oracle(p, what="small per-token scales", rel_rows=True)


@pytest.mark.parametrize("tc", [False, True])
def test_query_elements_spanning_2e16(tc):
    """Query elements of magnitude 2^-8 .. 2^8 (each its own 2^u) inside every head group."""
    p = synth.make_problem(73, num_seqs=4, context_lens=[3000, 130, 8192, 700], q_lens=[1] * 4,
                           q_mag_log2=8.0)
    check_against_oracle(p, what=f"wide-range q tcgen05={tc}", rel_rows=True, tcgen05=tc)


# --------------------------------------------------------------------------- invariants

def test_sparse_all_pages_equals_dense_on_a_slice():
    """A slice of the sparse workload (2 requests, a real partial last page): selecting
    every page equals the dense run; both equal the oracle."""
    p = synth.make_problem(40, num_seqs=2, context_lens=[130000, 5000], q_lens=[1, 4],
                           page_size=128)
    npg = (p.context_lens + 127) // 128
    sel = np.full((2, int(npg.max())), -1, dtype=np.int32)
    rng = np.random.default_rng(1)
    for r in range(2):
        sel[r, :npg[r]] = rng.permutation(npg[r])
    import dataclasses
    ps = dataclasses.replace(p, selected=sel, num_selected=npg.astype(np.int32))
    dense, _, f1 = gpu_run(p, out_dtype="f32")
    sparse, _, f2 = gpu_run(ps, out_dtype="f32")
    assert f1 == 0 and f2 == 0
    compare_split(sparse, dense, "sparse over every page vs dense")
    ref, _ = O.decode(p)
    compare(dense, ref, "dense slice")


def test_split_k_matches_single_pass_fp32():
    p = synth.long_128k(2, scale_mode="per_token", num_seqs=4)
    single, _, f0 = gpu_run(p, out_dtype="f32", partition_tokens=1 << 20)
    assert f0 == 0
    for part in (0, 512, 2048, 8192):
        split, _, f = gpu_run(p, out_dtype="f32", partition_tokens=part)
        assert f == 0
        compare_split(split, single, f"partition {part} vs one pass")


def test_scalar_mode_equals_uniform_per_token_scales():
    import dataclasses
    p = synth.make_problem(41, num_seqs=3, context_lens=[3000, 777, 129], q_lens=[1, 1, 1],
                           scale_mode="scalar")
    ks = np.full((p.num_pages, 1, p.page_size), np.float32(p.k_scale_scalar), np.float32)
    vs = np.full((p.num_pages, 1, p.page_size), np.float32(p.v_scale_scalar), np.float32)
    pt = dataclasses.replace(p, scale_mode="per_token", k_scale=ks, v_scale=vs)
    a, _, _ = gpu_run(p, out_dtype="f32")
    b, _, _ = gpu_run(pt, out_dtype="f32")
    compare_split(a, b, "scalar vs uniform per-token")


def test_ragged_equals_uniform_row_by_row():
    p = synth.make_problem(42, num_seqs=4, context_lens=[900, 4000, 300, 2500],
                           q_lens=[4, 4, 6, 2])
    rag, _, _ = gpu_run(p, out_dtype="f32")
    for r in range(4):
        one = subset(p, [r])
        o1, _, _ = gpu_run(one, out_dtype="f32")
        compare_split(rag[rows_of(p, [r])], o1, f"ragged batch vs request {r} alone")


# ------------------------------------------------------------------------ other shapes

@pytest.mark.parametrize("ps", [16, 32, 64])
def test_page_sizes(ps):
    p = synth.make_problem(43 + ps, num_seqs=3, context_lens=[1000, 37, 400], q_lens=[1, 1, 1],
                           page_size=ps)
    check_against_oracle(p, what=f"page {ps}")


def test_two_kv_heads_ragged():
    p = synth.make_problem(44, num_seqs=3, context_lens=[700, 260, 1500], q_lens=[2, 1, 3],
                           num_kv_heads=2)
    check_against_oracle(p, what="Hkv 2")


def test_q_len_eight():
    p = synth.make_problem(45, num_seqs=3, context_lens=[600, 128, 2049], q_lens=[8, 5, 7])
    check_against_oracle(p, what="q_len 8")


def test_sparse_page16_with_padding():
    import dataclasses
    p = synth.make_problem(46, num_seqs=3, context_lens=[1000, 300, 77], q_lens=[1, 3, 2],
                           page_size=16, selected_pages=12)
    sel = p.selected.copy()
    sel[0, 3] = -1
    p = dataclasses.replace(p, selected=sel)
    check_against_oracle(p, what="sparse page 16")


# ------------------------------------------------------------------------- exactness

def test_row_map_bit_exact():
    for p in (synth.ragged_spec(3, "A"), synth.ragged_spec(3, "B"), synth.tiny_dense(0)):
        d = dv.to_device(p)
        plan = dv.plan_for(p)
        rm = plan.row_map(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["context_lens"],
                          **dv.call_kwargs(p, d))
        torch.cuda.synchronize()
        assert np.array_equal(rm.cpu().numpy(), O.row_map(p.cu_seqlens_q, p.context_lens))


def expected_tiles(p):
    """Independent host listing of every KV tile: (r, h, tile, [(slot, lp, phys)])."""
    ppt = 128 // p.page_size
    tiles = []
    for r in range(p.num_seqs):
        L = int(p.context_lens[r])
        npg = (L + p.page_size - 1) // p.page_size
        if p.selected is None:
            nt = (L + 127) // 128
            lps = lambda t: [t * ppt + k if t * ppt + k < npg else -1 for k in range(ppt)]
        else:
            ns = int(p.num_selected[r])
            nt = (ns + ppt - 1) // ppt
            def lps(t, r=r, ns=ns, npg=npg):
                out = []
                for k in range(ppt):
                    i = t * ppt + k
                    e = int(p.selected[r, i]) if i < ns else -1
                    out.append(e if 0 <= e < npg else -1)
                return out
        if p.q_lens[r] == 0:
            nt = 0
        for h in range(p.num_kv_heads):
            for t in range(nt):
                tiles.append((r, h, t, [(k, lp, int(p.block_table[r, lp]) if lp >= 0 else -1)
                                        for k, lp in enumerate(lps(t))]))
    return tiles


@pytest.mark.parametrize("case", ["tiny", "sparse16", "ragged", "bf16", "two_heads"])
def test_gather_bit_exact(case):
    if case == "tiny":
        p = synth.tiny_dense(0)
    elif case == "sparse16":
        p = synth.make_problem(47, num_seqs=3, context_lens=[1000, 300, 77], q_lens=[1, 3, 2],
                               page_size=16, selected_pages=12)
    elif case == "ragged":
        p = synth.ragged_spec(3, "B")
    elif case == "bf16":
        p = synth.make_problem(48, num_seqs=2, context_lens=[300, 129], q_lens=[1, 1],
                               kv_dtype="bf16", scale_mode="none")
    else:
        p = synth.make_problem(49, num_seqs=2, context_lens=[300, 129], q_lens=[1, 2],
                               num_kv_heads=2, page_size=32)
    tiles = expected_tiles(p)
    d = dv.to_device(p)
    plan = dv.plan_for(p)
    dump, tb = plan.gather(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                           d["context_lens"], len(tiles), **dv.call_kwargs(p, d))
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    dump = dump.cpu().numpy()
    fp8 = p.kv_dtype == "fp8"
    rowb = 128 if fp8 else 256
    ps = p.page_size
    for gt, (r, h, t, slots) in enumerate(tiles):
        blk = dump[gt * tb:(gt + 1) * tb]
        hdr = blk[:128].view(np.int32)
        assert (hdr[0], hdr[1], hdr[2]) == (r, h, t), (gt, hdr[:8])
        kt = blk[128:128 + 128 * rowb].reshape(128, rowb)
        vt = blk[128 + 128 * rowb:128 + 256 * rowb].reshape(128, rowb)
        for k, lp, phys in slots:
            assert hdr[16 + k] == phys and hdr[8 + k] == (lp * ps if lp >= 0 else -1)
            if lp < 0:
                continue
            want_k = p.k_cache[phys, h].view(np.uint8).reshape(ps, rowb)
            want_v = p.v_cache[phys, h].view(np.uint8).reshape(ps, rowb)
            assert np.array_equal(kt[k * ps:(k + 1) * ps], want_k), (gt, k)
            assert np.array_equal(vt[k * ps:(k + 1) * ps], want_v), (gt, k)
            if fp8 and p.scale_mode == "per_token":
                sc = blk[128 + 256 * rowb:].view(np.float32)
                assert np.array_equal(sc[k * ps:(k + 1) * ps], p.k_scale[phys, h])
                assert np.array_equal(sc[128 + k * ps:128 + (k + 1) * ps], p.v_scale[phys, h])
    # the gathered positions below each request's context are, in order, the oracle's
    # key set of the request's last row (whose cutoff is the context length)
    for r in range(p.num_seqs):
        if p.q_lens[r] == 0:
            continue
        got = []
        for (rr, h, t, slots) in tiles:
            if rr == r and h == 0:
                for k, lp, phys in slots:
                    if lp >= 0:
                        got.extend(x for x in range(lp * ps, lp * ps + ps) if x < p.context_lens[r])
        want = O.key_positions(p, r, int(p.q_lens[r]) - 1)
        assert np.array_equal(np.array(got, dtype=np.int64), want), r


# ------------------------------------------------------------------- robustness (no faults)

def test_bad_page_id_is_flagged_not_read():
    p = synth.make_problem(50, num_seqs=3, context_lens=[500, 400, 300], q_lens=[1, 1, 1])
    bt = p.block_table.copy()
    bt[1, 2] = p.num_pages + 5
    import dataclasses
    bad = dataclasses.replace(p, block_table=bt)
    out, lse, flags = gpu_run(bad)
    assert flags & 0x01, f"flags {flags:#x}"
    ref, _ = O.decode(subset(p, [0, 2]))
    compare(out[rows_of(p, [0, 2])], ref, "untouched requests")


def test_uniform_plan_flags_ragged_device_cu():
    """Without the host mirror, a uniform plan given the [4, 4, 6, 2] segment on the
    device raises PA_DEV_NOT_UNIFORM instead of mis-mapping rows silently."""
    p = synth.make_problem(51, num_seqs=4, context_lens=[300, 300, 300, 300], q_lens=[4, 4, 6, 2])
    d = dv.to_device(p)
    plan = dv.plan_for(p, ragged=False, q_len=4, max_context_len=300)
    kw = dv.call_kwargs(p, d, host_mirror=False)
    plan.decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["context_lens"], **kw)
    assert plan.device_status() & 0x08


def test_empty_key_sets_give_zeros():
    p = synth.make_problem(52, num_seqs=3, context_lens=[0, 200, 0], q_lens=[1, 1, 1])
    out, lse, flags = gpu_run(p)
    assert flags & 0x04  # context_len < q_len
    assert np.all(out[[0, 2]] == 0) and np.all(np.isneginf(lse[[0, 2]]))
    ref, _ = O.decode(subset(p, [1]))
    compare(out[[1]], ref, "non-empty request")


def test_repeated_calls_bit_identical():
    """Split-K counters reset themselves: back-to-back calls agree bit for bit."""
    p = synth.long_128k(2, scale_mode="per_token", num_seqs=2, context=20000)
    d = dv.to_device(p)
    plan = dv.plan_for(p)
    a, _ = dv.run(plan, p, d)
    b, _ = dv.run(plan, p, d)
    c, _ = dv.run(plan, p, d)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(b, c)
    assert plan.device_status() == 0


def test_cuda_graph_capture_and_replay():
    p = synth.make_problem(53, num_seqs=4, context_lens=[5000, 3000, 7000, 100], q_lens=[1] * 4)
    d = dv.to_device(p)
    plan = dv.plan_for(p)
    ref, _ = dv.run(plan, p, d)
    out = torch.empty_like(ref)
    kw = dv.call_kwargs(p, d)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["context_lens"],
                    out=out, **kw)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


# ------------------------------------------------- many rows: per-token-as-decode prefill

def test_prefill_as_decode_dense():
    """A 300-token prefill chunk after 100 prompt tokens, one request per token sharing the
    sequence's pages: every row against the oracle (each attends its causal prefix)."""
    check_against_oracle(synth.prefill_as_decode(6, 300, 100, page_size=16),
                         what="prefill as decode")


def test_prefill_as_decode_sparse():
    """The sparse prefill: each token's request attends 8 of its prefix's pages."""
    check_against_oracle(synth.prefill_as_decode(7, 200, 2000, page_size=16, selected_pages=8),
                         what="sparse prefill as decode")


def test_prefill_as_decode_full_size():
    """The bench's prefill workload (2048 tokens after 6144), every row."""
    check_against_oracle(synth.prefill_as_decode(6, 2048, 6144), what="prefill 2K after 6K")


@pytest.mark.parametrize("tc", [False, True])
def test_empty_page_slots_after_nan_in_shared_memory(tc):
    """Sparse decode whose tiles have empty page slots (3 selected pages of 16 tokens in a
    128-token tile), launched right after a kernel that stages NaN through shared memory:
    the empty slots' stale per-token scales must not reach the output."""
    p = synth.make_problem(48, num_seqs=6, context_lens=[300, 77, 1000, 16, 129, 500],
                           q_lens=[1] * 6, page_size=16, selected_pages=3)
    d = dv.to_device(p)
    plan = dv.plan_for(p, tcgen05=tc)
    x = torch.full((2048, 2048), float("nan"), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        y = x @ x
    out, lse = dv.run(plan, p, d, lse=True)
    torch.cuda.synchronize()
    del y
    assert plan.device_status() == 0
    ref, ref_lse = O.decode(p)
    compare(out.float().cpu().numpy(), ref, f"empty slots after NaN smem tcgen05={tc}")
    compare_lse(lse.cpu().numpy(), ref_lse, "lse")
