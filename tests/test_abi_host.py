"""Host-side checks of the C ABI: the library builds and exports every symbol pa.h
declares, and plans and calls are refused at set-up exactly as documented.  Nothing
here launches a kernel: calls are checked with pa_decode_check on check-only plans,
whose fake device pointers are never dereferenced."""
import ctypes

import numpy as np
import pytest

from paged_fp8_kv_04_gb300 import binding as B
from paged_fp8_kv_04_gb300 import build as libbuild

OK, INVALID, UNSUP, CAP, RAGGED, ALIGN, CUDA, DEVDATA, WS = range(9)


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return B.lib()


def test_exports_every_header_symbol(lib):
    names = B.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pa.h but not exported"


def test_status_strings(lib):
    for code, name in B.STATUS.items():
        assert lib.pa_status_string(code).decode() == name


def desc(**kw):
    base = dict(max_batch=32, max_context_len=8192, num_sms=152)
    base.update(kw)
    return B.make_desc(**base)


@pytest.mark.parametrize("kw,want", [
    (dict(), OK),
    (dict(group_size=8), UNSUP),
    (dict(head_dim=64), UNSUP),
    (dict(page_size=256), UNSUP),
    (dict(page_size=16), OK),
    (dict(scale_mode="none"), UNSUP),
    (dict(kv_dtype="bf16"), UNSUP),
    (dict(kv_dtype="bf16", scale_mode="none"), OK),
    (dict(scale_mode="scalar"), OK),
    (dict(q_len=0), INVALID),
    (dict(q_len=9), UNSUP),
    (dict(q_len=8, q_mode="ragged"), OK),
    (dict(max_batch=4097), UNSUP),
    (dict(max_batch=0), INVALID),
    (dict(partition_tokens=100), UNSUP),
    (dict(partition_tokens=512), OK),
    (dict(out_dtype="f32"), OK),
    (dict(num_kv_heads=0), UNSUP),
])
def test_plan_validation(lib, kw, want):
    d = desc(**kw)
    assert lib.pa_plan_validate(ctypes.byref(d)) == want
    size = lib.pa_plan_workspace_size(ctypes.byref(d))
    assert (size > 0) == (want == OK)


def test_reserved_fields_must_be_zero(lib):
    d = desc()
    d.reserved[1] = 3
    assert lib.pa_plan_validate(ctypes.byref(d)) == INVALID
    d = desc()
    d.flags = 0x4
    assert lib.pa_plan_validate(ctypes.byref(d)) == INVALID
    assert lib.pa_plan_validate(ctypes.byref(desc(pdl=False))) == OK


def test_workspace_size_is_bounded_and_deterministic(lib):
    d = desc()
    a = lib.pa_plan_workspace_size(ctypes.byref(d))
    assert a == lib.pa_plan_workspace_size(ctypes.byref(desc())) and a % 256 == 0
    # balanced schedule: partial slots scale with the SM count, not with the batch
    big = lib.pa_plan_workspace_size(ctypes.byref(desc(max_batch=4096)))
    assert big - a == (4096 - 32) * 4 // 256 * 256 or big > a
    assert lib.pa_plan_workspace_size(ctypes.byref(desc(q_len=4, q_mode="ragged"))) > a
    # fixed partitions: one slot pair per (request, head, partition)
    part = lib.pa_plan_workspace_size(ctypes.byref(desc(partition_tokens=512)))
    slots = 2 * 32 * 16
    assert part >= slots * 16 * 128 * 4


def _info(lib, d):
    plan = ctypes.c_void_p()
    assert lib.pa_plan_create(ctypes.byref(d), None, 0, ctypes.byref(plan)) == OK
    inf = B.PlanInfo()
    assert lib.pa_plan_get_info(plan, ctypes.byref(inf)) == OK
    lib.pa_plan_destroy(plan)
    return inf


def test_shared_memory_budget_pinned(lib):
    """The stage count and shared-memory carve are computed in one place (the plan) and
    pinned here (ROCm/ATOM PR 2710 review, "Smaller": an unpinned mirrored LDS budget)."""
    inf = _info(lib, desc())
    assert inf.threads_per_cta == 384 and inf.tile_tokens == 128
    # one query token: a 2-slot exchange buffer (the CTA's last merge runs in stage
    # memory) leaves room for 6 FP8 stages of 33 KB, 3 BF16 stages of 64 KB
    assert inf.stages == 6 and inf.smem_bytes <= 232448
    assert inf.grid_ctas == 152 and inf.partial_slots == 304
    bf = _info(lib, desc(kv_dtype="bf16", scale_mode="none"))
    assert bf.stages == 3 and bf.smem_bytes <= 232448
    q4 = _info(lib, desc(q_len=4, q_mode="ragged", max_batch=64))
    assert q4.stages == 4 and q4.smem_bytes <= 232448
    q8 = _info(lib, desc(q_len=8, q_mode="ragged", max_batch=4096))
    assert q8.stages >= 2 and q8.smem_bytes <= 232448


def test_create_refuses_bad_workspace(lib):
    d = desc()
    plan = ctypes.c_void_p()
    assert lib.pa_plan_create(ctypes.byref(d), None, 1024, ctypes.byref(plan)) == WS
    assert not plan.value
    bad = desc(head_dim=96)
    assert lib.pa_plan_create(ctypes.byref(bad), None, 0, ctypes.byref(plan)) == UNSUP


class FakeCall:
    """Aligned fake device addresses (never dereferenced: only pa_decode_check sees them)."""

    def __init__(self, B_, rows, **over):
        self.a = B.DecodeArgs()
        addr = iter(range(0x100000, 0x10000000, 0x10000))
        for f in ("q", "k_cache", "v_cache", "k_scale", "v_scale", "block_table", "context_lens",
                  "out"):
            setattr(self.a, f, next(addr))
        self.a.num_pages = 4096
        self.a.block_table_stride = 64
        self.a.num_seqs = B_
        self.a.num_rows = rows
        self.a.sm_scale = 1.0 / np.sqrt(128.0)
        self.keep = []
        for k, v in over.items():
            if isinstance(v, np.ndarray):
                v = np.ascontiguousarray(v, dtype=np.int32)
                self.keep.append(v)
                v = v.ctypes.data
            setattr(self.a, k, v)


def _plan(lib, **kw):
    d = desc(**kw)
    plan = ctypes.c_void_p()
    assert lib.pa_plan_create(ctypes.byref(d), None, 0, ctypes.byref(plan)) == OK
    return plan


def check(lib, plan, call):
    return lib.pa_decode_check(plan, ctypes.byref(call.a))


def test_uniform_plan_accepts_uniform_segment(lib):
    plan = _plan(lib, q_len=4, max_batch=32, max_rows=128)
    cu = np.arange(0, 4 * 31 + 1, 4)
    assert check(lib, plan, FakeCall(31, 124, cu_seqlens_q_host=cu)) == OK
    assert check(lib, plan, FakeCall(31, 124)) == OK


def test_uniform_plan_refuses_121_rows(lib):
    """30 requests with q_len 4 and one with q_len 1 give 121 rows, which a uniform
    q_len-4 plan cannot hold (ROCm/ATOM PR 2122, section 2)."""
    plan = _plan(lib, q_len=4, max_batch=32, max_rows=128)
    assert check(lib, plan, FakeCall(31, 121)) == RAGGED


def test_uniform_plan_refuses_4_4_6_2_with_host_mirror(lib):
    """[4, 4, 6, 2] sums to 16 and divides by 4, yet is ragged: caught from the host
    mirror of cu_seqlens_q (ROCm/ATOM PR 2122, section 2)."""
    plan = _plan(lib, q_len=4, max_batch=32, max_rows=128)
    cu = np.array([0, 4, 8, 14, 16])
    assert check(lib, plan, FakeCall(4, 16, cu_seqlens_q_host=cu)) == RAGGED
    assert check(lib, plan, FakeCall(4, 16, cu_seqlens_q_host=np.array([0, 4, 8, 12, 16]))) == OK


def test_ragged_plan(lib):
    plan = _plan(lib, q_len=8, q_mode="ragged", max_batch=32, max_rows=256)
    cu = np.array([0, 4, 8, 14, 16])
    assert check(lib, plan, FakeCall(4, 16)) == INVALID          # cu_seqlens_q is required
    assert check(lib, plan, FakeCall(4, 16, cu_seqlens_q=0x9000000, cu_seqlens_q_host=cu)) == OK
    big = np.array([0, 4, 13, 14, 16])                           # one request with 9 rows
    assert check(lib, plan, FakeCall(4, 16, cu_seqlens_q=0x9000000, cu_seqlens_q_host=big)) == CAP
    bad = np.array([0, 4, 3, 14, 16])
    assert check(lib, plan, FakeCall(4, 16, cu_seqlens_q=0x9000000, cu_seqlens_q_host=bad)) == INVALID
    wrong_total = np.array([0, 4, 8, 14, 15])
    assert check(lib, plan, FakeCall(4, 16, cu_seqlens_q=0x9000000,
                                      cu_seqlens_q_host=wrong_total)) == INVALID


def test_capacity_refusals(lib):
    plan = _plan(lib, max_batch=32, max_context_len=8192)
    assert check(lib, plan, FakeCall(33, 33)) == CAP
    assert check(lib, plan, FakeCall(32, 32)) == OK
    assert check(lib, plan, FakeCall(32, 32, num_pages=1 << 30)) == CAP
    assert check(lib, plan, FakeCall(0, 0)) == OK


def test_pointer_and_alignment_refusals(lib):
    plan = _plan(lib)
    assert check(lib, plan, FakeCall(2, 2, k_scale=None)) == INVALID
    assert check(lib, plan, FakeCall(2, 2, out=None)) == INVALID
    assert check(lib, plan, FakeCall(2, 2, q=0x100008)) == ALIGN
    assert check(lib, plan, FakeCall(2, 2, k_cache=0x200004)) == ALIGN
    assert check(lib, plan, FakeCall(2, 2, sm_scale=0.0)) == INVALID
    assert check(lib, plan, FakeCall(2, 2, sm_scale=float("nan"))) == INVALID
    assert check(lib, plan, FakeCall(2, 2, block_table_stride=0)) == INVALID
    assert check(lib, plan, FakeCall(2, 2, reserved0=1)) == INVALID


def test_scalar_mode_scales(lib):
    plan = _plan(lib, scale_mode="scalar")
    assert check(lib, plan, FakeCall(2, 2, k_scale=None, v_scale=None, k_scale_scalar=0.01,
                                     v_scale_scalar=0.02)) == OK
    assert check(lib, plan, FakeCall(2, 2, k_scale_scalar=float("inf"))) == INVALID
    assert check(lib, plan, FakeCall(2, 2, v_scale_scalar=-1.0)) == INVALID


def test_sparse_refusals(lib):
    dense = _plan(lib)
    sel = dict(selected_pages=0xA000000, num_selected=0xA100000, selected_stride=64)
    assert check(lib, dense, FakeCall(2, 2, **sel)) == UNSUP
    sparse = _plan(lib, max_selected_pages=64)
    assert check(lib, sparse, FakeCall(2, 2, **sel)) == OK
    assert check(lib, sparse, FakeCall(2, 2, selected_pages=0xA000000, num_selected=0xA100000,
                                       selected_stride=65)) == CAP
    assert check(lib, sparse, FakeCall(2, 2, selected_pages=0xA000000, selected_stride=8)) == INVALID


def test_decode_on_check_only_plan_launches_nothing(lib):
    plan = _plan(lib)
    call = FakeCall(2, 2)
    assert lib.pa_decode(plan, ctypes.byref(call.a), None) == WS
    rm = ctypes.c_void_p(0x7000000)
    assert lib.pa_debug_row_map(plan, ctypes.byref(call.a), rm, None) == WS
    assert lib.pa_debug_gather(plan, ctypes.byref(call.a), ctypes.c_void_p(0x7000000), 1 << 20,
                               None) == WS


def test_noalloc_refuses_a_plan_larger_than_its_scratch(lib):
    """pa_decode_noalloc refuses, before touching a GPU, a descriptor whose workspace
    exceeds its fixed scratch (q_len 8 on 152 SMs needs about 20 MB)."""
    big = desc(q_len=8, q_mode="ragged")
    assert lib.pa_plan_workspace_size(ctypes.byref(big)) > (8 << 20)
    call = FakeCall(2, 2, cu_seqlens_q=0x9000000)
    assert lib.pa_decode_noalloc(ctypes.byref(big), ctypes.byref(call.a), None) == CAP
    assert lib.pa_decode_noalloc(None, ctypes.byref(call.a), None) == INVALID


def _kv_args(**over):
    a = B.KvWriteArgs()
    vals = dict(k_new=0x100000, v_new=0x200000, slot_mapping=0x300000, k_cache=0x400000,
                v_cache=0x500000, k_scale=0x600000, v_scale=0x700000, status=None,
                num_tokens=0, num_pages=8, num_kv_heads=1, head_dim=128, page_size=128,
                reserved=0)
    vals.update(over)
    for k, v in vals.items():
        setattr(a, k, v)
    return a


def test_kv_quantize_write_refusals(lib):
    """pa_kv_quantize_write checks its arguments before touching a device; with no
    tokens a valid call enqueues nothing and succeeds."""
    call = lambda **kw: lib.pa_kv_quantize_write(ctypes.byref(_kv_args(**kw)), None)
    assert lib.pa_kv_quantize_write(None, None) == INVALID
    assert call() == OK
    assert call(head_dim=64) == UNSUP
    assert call(page_size=48) == UNSUP
    assert call(page_size=256) == UNSUP
    assert call(num_tokens=-1) == INVALID
    assert call(num_kv_heads=0) == INVALID
    assert call(num_pages=0) == INVALID
    assert call(reserved=3) == INVALID
    assert call(num_tokens=1 << 30, num_kv_heads=4) == INVALID
    assert call(k_new=None) == INVALID
    assert call(v_scale=None) == INVALID
    assert call(k_new=0x100008) == ALIGN
    assert call(v_cache=0x500004) == ALIGN
    assert call(k_scale=0x600002) == ALIGN
    assert call(slot_mapping=0x300004) == ALIGN
    assert call(status=0x800002) == ALIGN


def _ix_args(**over):
    a = B.IndexArgs()
    vals = dict(q=0x100000, k_cache=0x200000, k_scale=0x300000, block_table=0x400000,
                context_lens=0x500000, cu_seqlens_q=0x600000, selected=0x700000,
                num_selected=0x800000, scores=0x900000, status=None, num_pages=64,
                num_seqs=2, num_rows=0, index_heads=1, head_dim=128, page_size=128, topk=8,
                block_table_stride=16, max_q_len=1, sm_scale=0.088, reserved=0)
    vals.update(over)
    for k, v in vals.items():
        setattr(a, k, v)
    return a


def test_index_topk_refusals(lib):
    """pa_index_topk checks its arguments before touching a device; with no rows a valid
    call enqueues nothing and succeeds."""
    call = lambda **kw: lib.pa_index_topk(ctypes.byref(_ix_args(**kw)), None)
    assert lib.pa_index_topk(None, None) == INVALID
    assert call() == OK
    assert call(head_dim=64) == UNSUP
    assert call(page_size=8) == UNSUP
    assert call(max_q_len=5, index_heads=4) == UNSUP
    assert call(max_q_len=4, index_heads=4) == OK
    assert call(topk=0) == INVALID
    assert call(topk=2048) == INVALID
    assert call(block_table_stride=0) == INVALID
    assert call(block_table_stride=20000) == INVALID
    assert call(sm_scale=0.0) == INVALID
    assert call(sm_scale=float("inf")) == INVALID
    assert call(num_seqs=0) == INVALID
    assert call(reserved=1) == INVALID
    assert call(scores=None) == INVALID
    assert call(k_scale=None) == OK
    assert call(k_cache=0x200008) == ALIGN
    assert call(scores=0x900004) == ALIGN
    assert call(selected=0x700002) == ALIGN


def test_missing_library_fails_loudly(tmp_path):
    """Without the built CUDA library the binding raises; there is no CPU fallback."""
    with pytest.raises(ImportError):
        B.lib(str(tmp_path / "libpagedfp8.so"))


def test_product_modules_do_not_import_the_oracle():
    """The package (binding, device helpers, input generators, build) never imports the
    oracle: only tests, the smoke check and the benchmark's baseline legs may."""
    import pathlib
    import re
    pkg = pathlib.Path(B.__file__).parent
    for f in pkg.glob("*.py"):
        text = f.read_text()
        assert not re.search(r"^\s*(from|import)\s+oracle\b", text, re.M), f"{f.name} imports the oracle"


def test_oracle_and_cuda_sources_share_nothing():
    """The C oracle includes no project header and the CUDA sources include nothing from
    the oracle: the two sides are written independently."""
    import pathlib
    import re
    root = pathlib.Path(B.__file__).parent.parent
    oracle_src = (root / "oracle" / "pa_oracle.c").read_text()
    incs = re.findall(r'#include\s+[<"]([^>"]+)[>"]', oracle_src)
    assert all(i in ("math.h", "pthread.h", "stdint.h", "stdlib.h", "string.h") for i in incs), incs
    for f in (root / "paged_fp8_kv_04_gb300" / "csrc").iterdir():
        text = f.read_text()
        assert "oracle" not in " ".join(re.findall(r'#include\s+[<"]([^>"]+)[>"]', text)), f.name


def test_trace_only_in_the_traced_build(lib):
    # the default build carries no trace code: pa_debug_trace refuses without a GPU call
    buf = (ctypes.c_uint64 * 16)()
    assert lib.pa_debug_trace(ctypes.cast(buf, ctypes.c_void_p), ctypes.sizeof(buf)) == 2  # unsupported
