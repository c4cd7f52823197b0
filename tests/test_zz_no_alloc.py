"""pa_decode_noalloc against pa_decode (needs a GPU).

Some callers cannot allocate device memory when they set up or run a decode -- an
engine plugin whose enqueue step must not allocate, or a runtime whose device memory
pool is fixed before the first request -- so they cannot give pa_plan_create the
workspace that pa_decode uses.  pa_decode_noalloc serves them from a fixed scratch
array inside the library.  This file is collected last, so that a run which stops at
the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from gpu_util import compare
from paged_fp8_kv_04_gb300 import binding as B
from paged_fp8_kv_04_gb300 import device as dv
from paged_fp8_kv_04_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_noalloc_matches_pa_decode_on_two_calls_in_a_row():
    # mixed context lengths: several requests are split across CTAs, so the split-K
    # partials and arrival counters live in the fixed scratch
    p = synth.make_problem(60, num_seqs=8, context_lens=[3000, 5000, 1, 700, 8192, 4096, 129, 2500],
                           q_lens=[1] * 8)
    d = dv.to_device(p)
    plan = dv.plan_for(p)
    ref, _ = dv.run(plan, p, d)
    torch.cuda.synchronize()
    ref = ref.float().cpu().numpy()
    lib = B.lib()
    kw = dv.call_kwargs(p, d)
    for call in range(2):
        out = torch.full(d["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        keep = []
        a = plan.args(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["context_lens"],
                      out=out, keep=keep, **kw)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        st = lib.pa_decode_noalloc(ctypes.byref(plan.desc), ctypes.byref(a), stream)
        assert st == 0, B.STATUS.get(st, st)
        torch.cuda.synchronize()
        compare(out.float().cpu().numpy(), ref, f"pa_decode_noalloc call {call}")
