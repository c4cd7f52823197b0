"""The KV quantise-and-write kernel against the oracle, through the C ABI (needs a GPU).

Codes and scales are integer / bit results (the fp32 scale amax / 448, and each code the
e4m3 rounding of the exact quotient x / scale on both sides), so the bar is bit-exact:
every byte of both caches and every scale bit, including the rows the call must leave
alone.  Then the producer-to-consumer round trip: pa_decode over a cache that
pa_kv_quantize_write filled equals the oracle's attention over the oracle's cache.
"""
import numpy as np
import pytest
import torch

from gpu_util import compare, compare_lse
from oracle import oracle as O
from paged_fp8_kv_04_gb300 import binding as B
from paged_fp8_kv_04_gb300 import device as dv
from paged_fp8_kv_04_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _dev(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16)
    return t.cuda()


def run_gpu(c: synth.KvWriteCase):
    """The case through pa_kv_quantize_write; returns the four arrays and the status word."""
    d = [_dev(x) for x in (c.k_new, c.v_new, c.slot_mapping, c.k_cache, c.v_cache,
                           c.k_scale, c.v_scale)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.kv_quantize_write(*d, status=status)
    torch.cuda.synchronize()
    kc, vc, ks, vs = (x.cpu().numpy() for x in d[3:])
    return kc, vc, ks, vs, int(status.item())


def run_oracle(c: synth.KvWriteCase):
    kc, vc, ks, vs = c.k_cache.copy(), c.v_cache.copy(), c.k_scale.copy(), c.v_scale.copy()
    bad = O.kv_quantize_write(c.k_new, c.v_new, c.slot_mapping, kc, vc, ks, vs)
    return kc, vc, ks, vs, bad


def assert_bit_exact(c):
    gk, gv, gks, gvs, status = run_gpu(c)
    ok, ov, oks, ovs, bad = run_oracle(c)
    for what, g, o in (("k codes", gk, ok), ("v codes", gv, ov)):
        diff = np.argwhere(g != o)
        assert diff.size == 0, f"{c.name}: {what} differ at {diff[:5].tolist()} ({len(diff)} bytes)"
    for what, g, o in (("k scales", gks, oks), ("v scales", gvs, ovs)):
        assert np.array_equal(g.view(np.uint32), o.view(np.uint32)), f"{c.name}: {what} differ"
    assert (status & B.DEV_BAD_SLOT != 0) == (bad > 0), f"{c.name}: status {status:#x}, bad {bad}"


@pytest.mark.parametrize("T,Hkv,ps,P,skip,past", [
    (37, 2, 16, 10, 3, 1),      # several heads, small pages, skipped and bad slots
    (200, 1, 128, 4, 5, 0),     # one head, 128-token pages
    (1, 1, 32, 1, 0, 0),        # a single token
    (130, 3, 64, 8, 0, 2),      # an odd head count, a tail group of units
])
def test_kv_quantize_write_bit_exact(T, Hkv, ps, P, skip, past):
    c = synth.kv_write_case(100 + T, T, Hkv, ps, P, skip=skip, past_end=past,
                            name=f"T{T} Hkv{Hkv} ps{ps}")
    assert_bit_exact(c)


def test_kv_quantize_write_full_size():
    """The bench's workload (the dense-8K batch written at once), every byte compared."""
    assert_bit_exact(synth.kv_write_prefill_8k(5))


def test_kv_quantize_write_near_ties_bit_exact():
    """Rows whose quotients x / scale sit a hair off an e4m3 rounding midpoint (where an
    fp32 product with 448 / amax, or an fp32 quotient, would pick the other code): every
    code as the oracle's exact quotient decides it."""
    import oracle_pins
    rows = {}
    for amax, x in oracle_pins._near_tie_rows():
        rows.setdefault(amax, []).append(x)
    xs = np.zeros((len(rows), 2, 128), np.float32)
    for t, (amax, items) in enumerate(sorted(rows.items())):
        for d, x in enumerate(items[:127]):
            xs[t, 0, d] = float(x) * (-1.0 if d % 3 == 1 else 1.0)
            xs[t, 1, 127 - d] = float(x) * 2.0 ** (-60 + 10 * (t % 13))  # other binades
        xs[t, 0, 127] = float(amax)
        xs[t, 1, 0] = float(amax) * 2.0 ** (-60 + 10 * (t % 13))
    k = synth.bf16_bits(xs)
    v = synth.bf16_bits(xs[::-1].copy())
    T, P, ps = xs.shape[0], (xs.shape[0] + 15) // 16, 16
    c = synth.KvWriteCase(k, v, np.arange(T, dtype=np.int64),
                          np.full((P, 2, ps, 128), 0x11, np.uint8), np.full((P, 2, ps, 128), 0x22, np.uint8),
                          np.zeros((P, 2, ps), np.float32), np.zeros((P, 2, ps), np.float32),
                          name="near ties")
    assert_bit_exact(c)


def test_decode_of_the_written_full_size_cache():
    """The producer-to-consumer test at full size: the 262144-token batch (per-token
    magnitudes 2^-20 .. 2^20, zero rows, single-value rows) written by
    pa_kv_quantize_write, then decoded as the dense-8K batch by pa_decode; every row
    against the oracle's attention over the oracle's own cache."""
    import dataclasses
    c = synth.kv_write_prefill_8k(5)
    gk, gv, gks, gvs, status = run_gpu(c)
    ok, ov, oks, ovs, bad = run_oracle(c)
    assert status == 0 and bad == 0
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)
    base = synth.dense_8k(1)
    p_gpu = dataclasses.replace(base, k_cache=gk, v_cache=gv, k_scale=gks, v_scale=gvs,
                                block_table=c.block_table, context_lens=c.context_lens)
    p_ora = dataclasses.replace(p_gpu, k_cache=ok, v_cache=ov, k_scale=oks, v_scale=ovs)
    d = dv.to_device(p_gpu)
    plan = dv.plan_for(p_gpu)
    out, lse = dv.run(plan, p_gpu, d, lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ref, ref_lse = O.decode(p_ora)
    compare(out.float().cpu().numpy(), ref, "decode of the written cache", rel_rows=True)
    # scores reach ~1e6 with keys of 2^20: lse to fp32's relative precision
    compare_lse(lse.cpu().numpy(), ref_lse, "decode of the written cache", rel=1e-5)


def test_zero_tokens_is_a_no_op():
    c = synth.kv_write_case(7, 4, 1, 16, 2)
    d = [_dev(x) for x in (c.k_new, c.v_new, c.slot_mapping, c.k_cache, c.v_cache,
                           c.k_scale, c.v_scale)]
    a = B.kv_write_args(*d, num_tokens=0)
    B.kv_quantize_write(None, None, None, d[3], None, None, None, args=a)
    torch.cuda.synchronize()
    assert np.array_equal(d[3].cpu().numpy(), c.k_cache)


@pytest.mark.parametrize("base", ["tiny", "ragged_b"])
def test_producer_to_consumer_round_trip(base):
    """pa_decode over a cache written by pa_kv_quantize_write equals the oracle's attention
    over the cache the oracle's quantiser writes (the two caches are also compared)."""
    p = synth.tiny_dense(3) if base == "tiny" else synth.ragged_spec(4, "B")
    ps, Hkv = p.page_size, p.num_kv_heads
    slots = []
    for r in range(p.num_seqs):
        for pos in range(int(p.context_lens[r])):
            slots.append(int(p.block_table[r, pos // ps]) * ps + pos % ps)
    T = len(slots)
    rng = np.random.default_rng(9)
    k_new = synth.bf16_bits(rng.standard_normal((T, Hkv, 128)).astype(np.float32) * 2)
    v_new = synth.bf16_bits(rng.standard_normal((T, Hkv, 128)).astype(np.float32))
    P = p.k_cache.shape[0]
    c = synth.KvWriteCase(k_new, v_new, np.array(slots, dtype=np.int64),
                          np.zeros((P, Hkv, ps, 128), np.uint8), np.zeros((P, Hkv, ps, 128), np.uint8),
                          np.zeros((P, Hkv, ps), np.float32), np.zeros((P, Hkv, ps), np.float32),
                          name=f"round trip {base}")
    gk, gv, gks, gvs, status = run_gpu(c)
    ok, ov, oks, ovs, bad = run_oracle(c)
    assert status == 0 and bad == 0
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)
    assert np.array_equal(gks.view(np.uint32), oks.view(np.uint32))
    assert np.array_equal(gvs.view(np.uint32), ovs.view(np.uint32))
    import dataclasses
    q_gpu = dataclasses.replace(p, k_cache=gk, v_cache=gv, k_scale=gks, v_scale=gvs)
    q_ora = dataclasses.replace(p, k_cache=ok, v_cache=ov, k_scale=oks, v_scale=ovs)
    d = dv.to_device(q_gpu)
    plan = dv.plan_for(q_gpu)
    out, lse = dv.run(plan, q_gpu, d, lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ref, ref_lse = O.decode(q_ora)
    compare(out.float().cpu().numpy(), ref, f"round trip {base}")
    compare_lse(lse.cpu().numpy(), ref_lse, f"round trip {base}")


def test_every_token_skipped_changes_nothing():
    c = synth.kv_write_case(8, 50, 2, 16, 8, skip=50)
    gk, gv, gks, gvs, status = run_gpu(c)
    assert status == 0
    assert np.array_equal(gk, c.k_cache) and np.array_equal(gv, c.v_cache)
    assert np.array_equal(gks.view(np.uint32), c.k_scale.view(np.uint32))
    assert np.array_equal(gvs.view(np.uint32), c.v_scale.view(np.uint32))
