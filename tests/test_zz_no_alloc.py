"""fdec_run_static_workspace: a run for callers that cannot allocate device memory.

Such callers (a plug-in inside a program whose memory pool owns the device, or
a loop that must never call cudaMalloc because it may synchronise the device)
pass only inputs and outputs; the library keeps its partials in an array built
into it.  Its results must match fdec_run's with a caller workspace, call after
call.  This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import LSE_TOL, OUT_TOL, lse_abs_err, row_rel_err


def _run_both(w, **plan_opts):
    dev = w.q.device
    table = torch.as_tensor(w.page_table, device=dev)
    lens = torch.as_tensor(w.seq_lens, device=dev)
    pd = fd.PagedDecode(w.seq_lens, w.q_len, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype,
                        w.causal, device=dev, **plan_opts)
    shape = (w.batch, w.q_len, w.num_qo_heads, w.head_dim)
    ref_o = torch.empty(shape, device=dev)
    ref_l = torch.empty(shape[:3], device=dev)
    pd.run(w.q, w.k, w.v, table, lens, ref_o, ref_l, scale=w.scale)
    got = []
    for _ in range(2):  # two calls in a row share the one built-in array
        o = torch.full(shape, float("nan"), device=dev)
        l = torch.full(shape[:3], float("nan"), device=dev)
        fd.fdec_run_static_workspace(pd.plan, w.q, w.k, w.v, table, lens, o, l, scale=w.scale)
        torch.cuda.synchronize()
        got.append((o.cpu().double().numpy(), l.cpu().double().numpy()))
    # the caller's own workspace still works after the built-in one was used
    o2 = torch.empty(shape, device=dev)
    l2 = torch.empty(shape[:3], device=dev)
    pd.run(w.q, w.k, w.v, table, lens, o2, l2, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o2, ref_o) and torch.equal(l2, ref_l)
    return ref_o.cpu().double().numpy(), ref_l.cpu().double().numpy(), got, pd


@pytest.mark.gpu
@pytest.mark.parametrize("make", [
    lambda: W.long_context(32768, device="cuda"),                       # split + one reduction pass
    lambda: W.tiny(device="cuda"),                                      # a single split, no reduction
    lambda: W.make(3, 2, 16, 4, 128, 16, [70, 900, 2500], dtype="f16", causal=True, device="cuda", seed=4),
])
def test_no_alloc_run_matches_fdec_run_on_two_calls(make):
    w = make()
    ref_o, ref_l, got, _ = _run_both(w)
    for o, l in got:
        assert np.isfinite(o).all()
        assert row_rel_err(o, ref_o) <= OUT_TOL
        assert lse_abs_err(l, ref_l) <= LSE_TOL


@pytest.mark.gpu
def test_no_alloc_run_with_two_reduction_passes():
    w = W.long_context(32768, device="cuda")
    ref_o, ref_l, got, pd = _run_both(w, blocks_per_split=1, reducer_fanin=16)
    assert pd.info["reduce_passes"] == 3
    for o, l in got:
        assert row_rel_err(o, ref_o) <= OUT_TOL and lse_abs_err(l, ref_l) <= LSE_TOL


def test_plans_larger_than_the_built_in_array_are_refused():
    # 64 sequences of 262144 tokens, one partial per 64-token block: ~hundreds of MB of partials
    plan = fd.fdec_plan([262144] * 64, 1, 64, 32, 4, 128, "bf16", blocks_per_split=1, num_sms=152)
    assert plan.workspace_bytes > (16 << 20)
    lib = fd._load()
    null_desc = fd.KVDesc(0, 1, 0, 0, 0)
    st = lib.fdec_run_static_workspace(plan.handle, None, 0, 0, null_desc, null_desc, None, 0, None,
                                       ctypes.c_float(1.0), None, None, None)
    assert fd.STATUS_NAMES[st] == "FDEC_ERR_WORKSPACE"
    assert "16777216" in fd.fdec_last_error()


_FRESH_PROCESS = r'''
import sys
sys.path.insert(0, sys.argv[1])
import numpy as np
import torch
import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import LSE_TOL, OUT_TOL, lse_abs_err, oracle_run, row_rel_err
w = W.make(2, 1, 32, 4, 128, 64, [5000, 70], dtype="bf16", device="cuda", seed=9)
plan = fd.fdec_plan(w.seq_lens, 1, w.page_size, 32, 4, 128, "bf16")  # never uploaded
table = torch.as_tensor(w.page_table, device="cuda")
lens = torch.as_tensor(w.seq_lens, device="cuda")
ref_o, ref_l = oracle_run(w.to("cpu"))
for call in range(2):
    o = torch.full((2, 1, 32, 128), float("nan"), device="cuda")
    l = torch.full((2, 1, 32), float("nan"), device="cuda")
    fd.fdec_run_static_workspace(plan, w.q, w.k, w.v, table, lens, o, l, scale=w.scale)
    torch.cuda.synchronize()
    e_o = row_rel_err(o.cpu().double().numpy(), ref_o)
    e_l = lse_abs_err(l.cpu().double().numpy(), ref_l)
    assert e_o <= OUT_TOL and e_l <= LSE_TOL, (call, e_o, e_l)
print("fresh-process no-alloc run ok")
'''


@pytest.mark.gpu
def test_first_call_in_a_fresh_process_on_a_plan_that_was_never_uploaded():
    # The intended use: a caller that cannot allocate makes a plan and calls the
    # no-alloc entry point first, before anything else in the process touched the
    # kernels (attributes, tensor maps) or the built-in array.
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH_PROCESS, root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "fresh-process no-alloc run ok" in r.stdout
