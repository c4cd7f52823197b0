"""The decode kernel's launch trace (the traced build of the library; needs a GPU).

pa_debug_trace is a diagnostic: the library built with tracing records the global timer
at fixed points of every CTA's run.  The trace must be consistent with the run it
describes: every CTA's marks of one launch in the order the kernel passes them, its tile
range the schedule's, and the launch count advancing by one per call.  The traced
library must also decode like the default one.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_fp8_kv_04_gb300 import binding as B
from paged_fp8_kv_04_gb300 import build as libbuild
from paged_fp8_kv_04_gb300 import device as dv
from paged_fp8_kv_04_gb300 import synth

pytestmark = pytest.mark.gpu

ENTRY, PROLOGUE, PRODUCER, CONSUMER, FIRST, LAST, EXIT, CALL, A, Bm = 0, 1, 2, 3, 4, 5, 10, 11, 12, 13


@pytest.fixture(scope="module")
def traced():
    import __graft_entry__
    __graft_entry__.build()
    default = B.lib()
    traced_lib = B.lib(libbuild.build(trace=True))
    yield default, traced_lib
    B._lib = default


def _run(lib, p, calls):
    saved = B._lib
    B._lib = lib
    try:
        d = dv.to_device(p, "cuda")
        plan = dv.plan_for(p, device="cuda")
        out = None
        for _ in range(calls):
            out = plan.decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                              d["context_lens"], **dv.call_kwargs(p, d))
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        return plan, out
    finally:
        B._lib = saved


def test_trace_marks_are_ordered(traced):
    default, traced_lib = traced
    # contexts of 1..5 K tokens: sequences split over several CTAs and whole ones
    p = synth.make_problem(21, num_seqs=12, context_lens=[1024 * (1 + i % 5) + 7 * i for i in range(12)],
                           q_lens=[1] * 12)
    calls = 20
    plan, out = _run(traced_lib, p, calls)
    _, ref = _run(default, p, 1)
    assert torch.equal(out, ref), "the traced library must decode like the default one"
    buf = np.zeros((16, 1024, 16), dtype=np.uint64)
    assert traced_lib.pa_debug_trace(ctypes.c_void_p(buf.ctypes.data), buf.nbytes) == 0
    grid = plan.info()["grid_ctas"]
    t = buf[:, :grid, :].astype(np.int64)
    order = np.argsort(t[:, 0, CALL])
    t = t[order]
    # 16 slots hold consecutive launches, the same count in every CTA of a launch
    counts = t[:, :, CALL]
    assert np.all(counts == counts[:, :1])
    assert np.array_equal(np.diff(counts[:, 0]), np.ones(15, dtype=np.int64))
    last = t[-1]
    busy = last[:, Bm] > last[:, A]
    assert busy.any()
    # the tile ranges of the busy CTAs tile the work without overlap
    rng = sorted((int(a), int(b)) for a, b in zip(last[busy, A], last[busy, Bm]))
    for (a0, b0), (a1, b1) in zip(rng, rng[1:]):
        assert b0 <= a1
    for k0, k1 in ((ENTRY, PROLOGUE), (PROLOGUE, CONSUMER), (CONSUMER, FIRST), (FIRST, LAST),
                   (LAST, EXIT), (PROLOGUE, PRODUCER)):
        assert np.all(last[busy, k1] >= last[busy, k0]), (k0, k1)
    # launches follow one another: each begins after the previous one's first entry
    assert np.all(np.diff(t[:, :, ENTRY].min(axis=1)) > 0)
