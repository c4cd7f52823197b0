"""pa_decode_noalloc against pa_decode and the oracle (needs a GPU).

Some callers cannot allocate device memory when they set up or run a decode -- an
engine plugin whose enqueue step must not allocate, or a runtime whose device memory
pool is fixed before the first request -- so they cannot give pa_plan_create the
workspace that pa_decode uses.  pa_decode_noalloc serves them from a fixed scratch
array inside the library.  It runs the same kernel and schedule as pa_decode, so its
output must equal pa_decode's bit for bit, and both must match the oracle.  This file
is collected last, so that a run which stops at the first failure has already run every
other test.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from gpu_util import compare
from oracle import oracle as O
from paged_fp8_kv_04_gb300 import binding as B
from paged_fp8_kv_04_gb300 import device as dv
from paged_fp8_kv_04_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _problem():
    # mixed context lengths: several requests are split across CTAs, so the split-K
    # partials and arrival counters live in the fixed scratch
    return synth.make_problem(60, num_seqs=8,
                              context_lens=[3000, 5000, 1, 700, 8192, 4096, 129, 2500],
                              q_lens=[1] * 8)


def _noalloc_calls(p, d, plan, calls=2):
    """pa_decode_noalloc with the plan's descriptor, `calls` times in a row."""
    lib = B.lib()
    kw = dv.call_kwargs(p, d)
    outs = []
    for _ in range(calls):
        out = torch.full(d["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        keep = []
        a = plan.args(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["context_lens"],
                      out=out, keep=keep, **kw)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        st = lib.pa_decode_noalloc(ctypes.byref(plan.desc), ctypes.byref(a), stream)
        assert st == 0, B.STATUS.get(st, st)
        torch.cuda.synchronize()
        outs.append(out)
    return outs


@pytest.mark.parametrize("tc", [False, True])
def test_noalloc_matches_pa_decode_on_two_calls_in_a_row(tc):
    p = _problem()
    d = dv.to_device(p)
    plan = dv.plan_for(p, tcgen05=tc)
    ref, _ = dv.run(plan, p, d)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    for k, out in enumerate(_noalloc_calls(p, d, plan)):
        assert torch.equal(out, ref), f"call {k}: differs from pa_decode (tcgen05={tc})"
    oracle_out, _ = O.decode(p)
    compare(ref.float().cpu().numpy(), oracle_out, f"pa_decode_noalloc vs oracle (tcgen05={tc})")


_FRESH = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import torch
from test_zz_no_alloc import _problem, _noalloc_calls
from paged_fp8_kv_04_gb300 import device as dv
p = _problem()
d = dv.to_device(p)
# the descriptor of a tcgen05 plan, but no pa_plan_create before the no-alloc call: the
# call's own set-up must raise the kernel's shared-memory limit on this device
plan = dv.plan_for(p, tcgen05=True, check_only=True)
outs = _noalloc_calls(p, d, plan)
full = dv.plan_for(p, tcgen05=True)
ref, _ = dv.run(full, p, d)
torch.cuda.synchronize()
assert full.info()["kernel"] == 1
for k, o in enumerate(outs):
    assert torch.equal(o, ref), k
print("fresh-process no-alloc ok")
"""


def test_noalloc_tcgen05_first_call_in_a_fresh_process():
    """In a new process, pa_decode_noalloc with a tcgen05 descriptor runs before any plan
    of the library has been created, and still equals pa_decode."""
    code = _FRESH.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "fresh-process no-alloc ok" in r.stdout
