"""CUDA-graph capture: fdec_run makes only kernel launches, so the very first
call of a fresh process may be captured, and one captured decode step replays
correctly while the device lengths grow up to the planned capacity (the
FlashInfer PR's reduce-overhead warm-up case and the llama.cpp PR's cold-start
capture question, on this library)."""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import assert_parity, oracle_run

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_first_call_of_a_fresh_process_is_captured():
    code = textwrap.dedent("""
        import numpy as np, torch
        import paged_split_kv_gather_gb300 as fd
        from paged_split_kv_gather_gb300 import workloads as W
        w = W.long_context(3000, device="cuda")
        table = torch.as_tensor(w.page_table, device="cuda")
        lens = torch.as_tensor(w.seq_lens, device="cuda")
        out = torch.zeros(1, 1, 32, 128, device="cuda"); lse = torch.zeros(1, 1, 32, device="cuda")
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            pd = fd.PagedDecode(w.seq_lens, 1, 64, 32, 4, 128, "bf16", stream=s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale, stream=s)
        torch.cuda.synchronize()
        assert torch.all(out == 0)          # nothing ran during capture
        g.replay(); torch.cuda.synchronize()
        ref = torch.empty_like(out); rl = torch.empty_like(lse)
        pd.run(w.q, w.k, w.v, table, lens, ref, rl, scale=w.scale); torch.cuda.synchronize()
        assert torch.equal(out, ref) and torch.equal(lse, rl)
        print("CAPTURED_FIRST_CALL_OK")
    """)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert "CAPTURED_FIRST_CALL_OK" in r.stdout, r.stdout + r.stderr


def test_plan_upload_refuses_a_capturing_stream():
    w = W.tiny(device="cuda")
    plan = fd.fdec_plan(w.seq_lens, 1, 16, 4, 1, 64, "f16")
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(fd.FdecError) as ei:
        with torch.cuda.graph(g, stream=s):
            fd.fdec_plan_upload(plan, ws, stream=s)
    assert ei.value.status_name == "FDEC_ERR_CAPTURING"


def test_captured_decode_loop_with_growing_lengths_equals_eager():
    cap = 3000
    w = W.make(2, 1, 32, 8, 128, 16, [cap, cap], dtype="bf16", device="cuda", seed=3)
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.tensor([1900, 1000], dtype=torch.int32, device="cuda")
    out = torch.zeros(2, 1, 32, 128, device="cuda")
    lse = torch.zeros(2, 1, 32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pd = fd.PagedDecode([cap, cap], 1, 16, 32, 8, 128, "bf16", stream=s)
        pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale, stream=s)  # warm
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale, stream=s)
    torch.cuda.synchronize()
    w_cpu = w.to("cpu")
    for step in range(64):
        cur = np.array([1900 + 17 * step, 1000 + 31 * step], dtype=np.int32)
        lens.copy_(torch.as_tensor(cur))
        g.replay()
        torch.cuda.synchronize()
        ref_o = torch.empty_like(out)
        ref_l = torch.empty_like(lse)
        pd.run(w.q, w.k, w.v, table, lens, ref_o, ref_l, scale=w.scale)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l), step
        if step in (0, 37, 63):
            ro, rl = oracle_run(w_cpu, seq_lens=cur)
            assert_parity(out.cpu(), lse.cpu(), ro, rl, f"graph step {step}")
    assert pd.device_errors() == 0


def test_first_call_with_an_e4m3_cache_and_scales_is_captured():
    """The pages' capture failure came from a lazily allocated unit-scale tensor for
    fp8 caches; here the scales are launch arguments, so the very first scaled call
    over an E4M3 cache captures and replays exactly."""
    code = textwrap.dedent("""
        import torch
        import paged_split_kv_gather_gb300 as fd
        from paged_split_kv_gather_gb300 import workloads as W
        w = W.long_context(3000, device="cuda", kv_dtype="fp8")
        table = torch.as_tensor(w.page_table, device="cuda")
        lens = torch.as_tensor(w.seq_lens, device="cuda")
        out = torch.zeros(1, 1, 32, 128, device="cuda"); lse = torch.zeros(1, 1, 32, device="cuda")
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            pd = fd.PagedDecode(w.seq_lens, 1, 64, 32, 4, 128, "bf16", stream=s, kv_dtype="fp8")
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale, stream=s, k_scale=0.5, v_scale=3.0)
        torch.cuda.synchronize()
        assert torch.all(out == 0)
        g.replay(); torch.cuda.synchronize()
        ref = torch.empty_like(out); rl = torch.empty_like(lse)
        pd.run(w.q, w.k, w.v, table, lens, ref, rl, scale=w.scale, k_scale=0.5, v_scale=3.0)
        torch.cuda.synchronize()
        assert torch.equal(out, ref) and torch.equal(lse, rl)
        print("CAPTURED_E4M3_OK")
    """)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert "CAPTURED_E4M3_OK" in r.stdout, r.stdout + r.stderr
