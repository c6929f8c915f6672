"""Benchmark: paged split-KV decode, µs/call and achieved HBM GB/s against the measured peak.

One step = one fdec_run over the workload (split kernel over the gathered
pages + the log-sum-exp reduction), with every input resident in HBM.  The
headline workload is the long-context decode at 262144 tokens (batch 1,
32 query / 4 KV heads, head_dim 128, bf16, page 64, 537 MB of K/V per call,
more than the 129 MB L2, so consecutive steps do not hit in L2).  The same line
carries the whole long-context sweep (1900 ... 262144 tokens), each point
timed per call with an L2 flush before it (eagerly between CUDA events, and
replayed from a CUDA graph of (flush, call) pairs minus the flushes), and back
to back in a CUDA graph whose calls rotate over copies of the K/V pools (each
call's pages out of L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fdec|reference]

--impl reference times the float64 CPU oracle on the same workload (a bounded
sample per step) on this host's cores.  With --gpus N > 1 (torchrun), every
rank runs its own replica of the workload: the path has no exchange step, so
there is no collective on the data path (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged split-KV decode: µs/call and achieved HBM GB/s vs GB300 peak, per KV length"
HEADLINE_LENGTH = 262144
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _bf16_peak():
    """Dense bf16 TFLOP/s: the burst figure (a kernel timed alone, per call)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def _attention_flops(w) -> float:
    """Algorithmic FLOPs of one call: 2 D per visible (query row, token) pair for
    q.K and 2 D for p.V (bottom-right causal visibility)."""
    total = 0
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        for i in range(w.q_len):
            n = min(L, L - w.q_len + i + 1) if w.causal else L
            total += max(n, 0)
    return 4.0 * w.head_dim * w.num_qo_heads * total


def _dense_query(dev, calls, hbm_peak, q_lens=(4, 8, 2048)):
    """Multi-token queries over the paged cache (batch 4, 32/8 heads, D 128, bf16,
    page 16, prefix 8192 + q_len, causal): q_len 4 and 8 (speculative decode) and
    2048 (a prefill chunk).  q_len x group > 16 takes the tcgen05 path (> 32 at head_dim 256), also
    timed on the 16-row warp-level kernel for comparison."""
    import torch

    import paged_split_kv_gather_gb300 as fd
    from paged_split_kv_gather_gb300 import workloads as W

    tflops_peak, tflops_kind = _bf16_peak()
    names = {fd.FDEC_PATH_SIMT: "simt", fd.FDEC_PATH_MMA: "mma", fd.FDEC_PATH_TC: "tcgen05"}
    flush = L2Flush(torch, dev)
    res = []
    for q_len in q_lens:
        w = W.multi_token(q_len, device=dev)
        table = torch.as_tensor(w.page_table, device=dev)
        lens = torch.as_tensor(w.seq_lens, device=dev)
        out = torch.empty((w.batch, q_len, w.num_qo_heads, w.head_dim), device=dev)
        lse = torch.empty((w.batch, q_len, w.num_qo_heads), device=dev)
        flops = _attention_flops(w)
        # the warp-level tensor-core kernel beside the tcgen05 one wherever the plan picks the latter
        paths = [fd.FDEC_PATH_AUTO] + ([fd.FDEC_PATH_MMA] if q_len * (w.num_qo_heads // w.num_kv_heads) > 16 else [])
        for path in paths:
            pd = fd.PagedDecode(w.seq_lens, q_len, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim,
                                w.dtype, w.causal, device=dev, path=path)
            for _ in range(3):
                pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale)
            n = calls if q_len < 64 else max(5, calls // 5)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            torch.cuda._sleep(int(n * 2e5))  # the host runs ahead: no host gap between a call's events
            for a, b in evs:
                flush()
                a.record()
                pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale)
                b.record()
            torch.cuda.synchronize()
            assert pd.device_errors() == 0
            us = float(np.median([a.elapsed_time(b) * 1e3 for a, b in evs]))
            tf = flops / (us * 1e-6) / 1e12
            gbs = w.kv_bytes / (us * 1e-6) / 1e9
            res.append({"q_len": q_len, "path": names[pd.info["path"]], "us_per_call": round(us, 2),
                        "TFLOP_per_s": round(tf, 1), "frac_of_bf16_peak": round(tf / tflops_peak, 4),
                        "GB_per_s": round(gbs, 1), "frac_of_hbm_peak": round(gbs / hbm_peak, 4),
                        "launches": int(pd.info["launches"]), "split_ctas": int(pd.info["num_split_ctas"])})
            if q_len < 64:  # speculative decode: also back to back, each call's pages out of L2
                b2b, ncp = _back_to_back_us(
                    torch, w, lambda k, v, pd=pd: pd.run(w.q, k, v, table, lens, out, lse, scale=w.scale))
                g_b = w.kv_bytes / (b2b * 1e-6) / 1e9
                res[-1].update({"back_to_back_us_per_call": round(b2b, 2), "back_to_back_GB_per_s": round(g_b, 1),
                                "back_to_back_frac_of_hbm_peak": round(g_b / hbm_peak, 4),
                                "back_to_back_pool_copies": ncp})
            del pd
        del w, table, lens, out, lse
    del flush
    return {"workload": "multi_token: batch 4, 32/8 heads, head_dim 128, bf16, page 16, KV 8192 + q_len, causal",
            "bf16_peak_tflops": tflops_peak, "bf16_peak_kind": tflops_kind,
            "flops": "4 x head_dim per visible (query head, query token, key token)", "points": res}


def _crossover(dev, calls):
    """16-row warp-level kernel against the tcgen05 kernel per head_dim and row count
    (rows = q_len x group): batch 4, 32/8 heads, KV 8192 + q_len, causal, bf16, page 16.
    The planner's AUTO rule takes tcgen05 above 16 rows for head_dim 64-192 and above 32 at 256."""
    import torch

    import paged_split_kv_gather_gb300 as fd
    from paged_split_kv_gather_gb300 import workloads as W

    flush = L2Flush(torch, dev)
    table_out = {}
    for d in (64, 128, 192, 256, 512):
        for q_len in (4, 8, 16):
            rows = q_len * 4
            w = W.make(4, q_len, 32, 8, d, 16, [8192 + q_len] * 4, dtype="bf16", causal=True, device=dev, seed=3)
            tb = torch.as_tensor(w.page_table, device=dev)
            ln = torch.as_tensor(w.seq_lens, device=dev)
            out = torch.empty((4, q_len, 32, d), device=dev)
            lse = torch.empty((4, q_len, 32), device=dev)
            entry = {}
            for name, path in (("mma", fd.FDEC_PATH_MMA), ("tcgen05", fd.FDEC_PATH_TC), ("auto", fd.FDEC_PATH_AUTO)):
                if path == fd.FDEC_PATH_TC and d == 512:
                    continue
                pd = fd.PagedDecode(w.seq_lens, q_len, 16, 32, 8, d, "bf16", True, device=dev, path=path)

                def run(pd=pd, w=w, tb=tb, ln=ln, out=out, lse=lse):
                    pd.run(w.q, w.k, w.v, tb, ln, out, lse, scale=w.scale)

                for _ in range(3):
                    run()
                med, _ = _time_calls(torch, run, calls, flush)
                entry[name] = round(med, 2) if name != "auto" else ("tcgen05" if pd.info["path"] == fd.FDEC_PATH_TC
                                                                   else "mma")
                del pd
            table_out[f"D{d}_rows{rows}"] = entry
            del w, tb, ln, out, lse
        torch.cuda.empty_cache()
    del flush
    return {"workload": "batch 4, 32/8 heads, KV 8192 + q_len, causal, bf16, page 16; us per flushed call",
            "points": table_out}


class L2Flush:
    """Evict the L2 between timed calls: write one buffer larger than the L2, then
    read another, so that the write-back of the dirty lines happens here, outside
    the timed call, and the L2 is left holding clean lines of an unrelated buffer."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.fill_(0.0)
        self.torch.sum(self.r)


def _time_calls(torch, run, calls, flush):
    """Median and min µs of `calls` calls of run(), each after an L2-evicting read,
    all enqueued behind a device-side delay (no host gap inside a call's events)."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
    torch.cuda._sleep(int(calls * 2e5))
    for a, b in evs:
        flush()
        a.record()
        run()
        b.record()
    torch.cuda.synchronize()
    t = [a.elapsed_time(b) * 1e3 for a, b in evs]
    return float(np.median(t)), float(min(t))


def _time_graph(torch, run, reps, flush, flush_us=None):
    """µs per call replayed from a CUDA graph: a graph of `reps` (L2 eviction, call)
    pairs against a graph of the evictions alone (or the given per-eviction µs)."""
    def capture(with_call):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for _ in range(reps):
                    flush()
                    if with_call:
                        run()
        torch.cuda.current_stream().wait_stream(side)
        return g

    res = []
    for with_call in ((True, False) if flush_us is None else (True,)):
        g = capture(with_call)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = 1e30
        for _ in range(5):
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b) * 1e3)
        res.append(best)
        del g
    base = res[1] if flush_us is None else flush_us * reps
    return max(0.0, (res[0] - base) / reps)


def _time_graph_once(torch, run_all):
    """µs of one replay of a CUDA graph of run_all() (best of 5)."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            run_all()
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 1e30
    for _ in range(5):
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b) * 1e3)
    del g
    return best


def _back_to_back_us(torch, w, run_kv, reps_min=20):
    """µs per call back to back: a CUDA graph of calls rotating over n copies of the
    K/V pools (and of q8_0 scale pools; n such that ~256 MB, twice the L2, are
    streamed between two reads of one copy), best of 5 replays / calls.
    run_kv(k, v, *scale_pools) runs one call on given pools."""
    n = 1 + -(-(256 << 20) // int(w.kv_bytes))
    pools = [w.k, w.v] + ([w.k_scales, w.v_scales] if w.kv_dtype == "q8_0" else [])
    copies = [[t] + [t.clone() for _ in range(n - 1)] for t in pools]
    reps = n * max(1, -(-reps_min // n))

    def run_all():
        for c in range(reps):
            run_kv(*(cp[c % n] for cp in copies))

    run_all()
    torch.cuda.synchronize()
    us = _time_graph_once(torch, run_all) / reps
    del copies
    return us, n


def _e4m3_point(dev, calls, hbm_peak, flush):
    """Quantised cache: the long-context shape (262144 tokens, 32/4 heads, D 128, page 64)
    over E4M3 codes with a k_scale and a v_scale; kv_bytes counts the 1-byte codes."""
    import torch

    import paged_split_kv_gather_gb300 as fd
    from paged_split_kv_gather_gb300 import workloads as W

    w = W.long_context(262144, device=dev, kv_dtype="fp8")
    pd = fd.PagedDecode(w.seq_lens, 1, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype,
                        device=dev, kv_dtype="fp8")
    table = torch.as_tensor(w.page_table, device=dev)
    lens = torch.as_tensor(w.seq_lens, device=dev)
    out = torch.empty((1, 1, w.num_qo_heads, w.head_dim), device=dev)
    lse = torch.empty((1, 1, w.num_qo_heads), device=dev)

    def run():
        pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale, k_scale=0.5, v_scale=2.0)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    med, mn = _time_calls(torch, run, calls, flush)
    gbs = w.kv_bytes / (med * 1e-6) / 1e9
    b2b, n = _back_to_back_us(torch, w, lambda k, v: pd.run(w.q, k, v, table, lens, out, lse, scale=w.scale,
                                                            k_scale=0.5, v_scale=2.0))
    g_b = w.kv_bytes / (b2b * 1e-6) / 1e9
    gf = _time_graph(torch, run, 20, flush)
    return {"us_per_call": round(med, 2), "us_min": round(mn, 2), "kv_bytes": int(w.kv_bytes),
            "GB_per_s": round(gbs, 1), "frac_of_peak": round(gbs / hbm_peak, 4),
            "graph_flushed_us_per_call": round(gf, 2),
            "graph_flushed_frac_of_peak": round(w.kv_bytes / (gf * 1e-6) / 1e9 / hbm_peak, 4),
            "back_to_back_us_per_call": round(b2b, 2), "back_to_back_GB_per_s": round(g_b, 1),
            "back_to_back_frac_of_peak": round(g_b / hbm_peak, 4), "back_to_back_pool_copies": n,
            "path": int(pd.info["path"]), "launches": int(pd.info["launches"]),
            "max_splits": int(pd.info["max_splits"]), "scales": {"k_scale": 0.5, "v_scale": 2.0}}


def _q8_point(dev, calls, hbm_peak, flush):
    """q8_0 cache: the long-context shape (262144 tokens, 32/4 heads, D 128, page 64,
    bf16 queries) over int8 codes with binary16 block scales (no spikes: the keys are
    drawn as codes); kv_bytes counts the codes and the scales."""
    import torch

    import paged_split_kv_gather_gb300 as fd
    from paged_split_kv_gather_gb300 import workloads as W

    w = W.make(1, 1, 32, 4, 128, 64, [262144], dtype="bf16", seed=0, device=dev, kv_dtype="q8_0",
               name="long_context_q8_0_L262144")
    pd = fd.PagedDecode(w.seq_lens, 1, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype,
                        device=dev, kv_dtype="q8_0")
    table = torch.as_tensor(w.page_table, device=dev)
    lens = torch.as_tensor(w.seq_lens, device=dev)
    out = torch.empty((1, 1, w.num_qo_heads, w.head_dim), device=dev)
    lse = torch.empty((1, 1, w.num_qo_heads), device=dev)

    def run():
        pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale, k_scales=w.k_scales, v_scales=w.v_scales)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    med, mn = _time_calls(torch, run, calls, flush)
    assert pd.device_errors() == 0
    gbs = w.kv_bytes / (med * 1e-6) / 1e9
    b2b, n = _back_to_back_us(torch, w, lambda k, v, ks, vs: pd.run(w.q, k, v, table, lens, out, lse, scale=w.scale,
                                                                    k_scales=ks, v_scales=vs))
    g_b = w.kv_bytes / (b2b * 1e-6) / 1e9
    gf = _time_graph(torch, run, 20, flush)
    return {"us_per_call": round(med, 2), "us_min": round(mn, 2), "kv_bytes": int(w.kv_bytes),
            "GB_per_s": round(gbs, 1), "frac_of_peak": round(gbs / hbm_peak, 4),
            "graph_flushed_us_per_call": round(gf, 2),
            "graph_flushed_frac_of_peak": round(w.kv_bytes / (gf * 1e-6) / 1e9 / hbm_peak, 4),
            "back_to_back_us_per_call": round(b2b, 2), "back_to_back_GB_per_s": round(g_b, 1),
            "back_to_back_frac_of_peak": round(g_b / hbm_peak, 4), "back_to_back_pool_copies": n,
            "path": int(pd.info["path"]), "launches": int(pd.info["launches"]),
            "max_splits": int(pd.info["max_splits"])}


def _config_points(dev, calls, hbm_peak):
    """The other workloads' µs/call and GB/s (tiny decode, batched GQA decode, the
    ragged serving batch at head_dim 192/256/512), a no-cliff sweep of the long-context
    shape over L = 1024 ... 8192 step 64, and CUDA-graph-replayed µs/call where launch
    latency matters (tiny decode, long-context L <= 4800)."""
    import torch

    import paged_split_kv_gather_gb300 as fd
    from paged_split_kv_gather_gb300 import workloads as W

    flush = L2Flush(torch, dev)

    def runner(w, capacities=None, **plan_opts):
        caps = w.seq_lens if capacities is None else capacities
        if w.kv_dtype:
            plan_opts.setdefault("kv_dtype", w.kv_dtype)
        pd = fd.PagedDecode(caps, w.q_len, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype,
                            w.causal, device=dev, **plan_opts)
        table = torch.as_tensor(w.page_table, device=dev)
        lens = torch.as_tensor(np.asarray(caps, dtype=np.int32), device=dev)
        out = torch.empty((w.batch, w.q_len, w.num_qo_heads, w.head_dim), device=dev)
        lse = torch.empty((w.batch, w.q_len, w.num_qo_heads), device=dev)

        def run():
            pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale)

        for _ in range(3):
            run()
        torch.cuda.synchronize()
        return pd, run

    points = {}
    for name, make in (("tiny_decode", lambda: W.tiny(device=dev)),
                       ("batched_gqa_decode", lambda: W.batched_gqa(device=dev)),
                       *[(f"ragged_serving_D{d}", (lambda d=d: W.ragged(d, device=dev))) for d in W.RAGGED_HEAD_DIMS]):
        w = make()
        pd, run = runner(w)
        med, mn = _time_calls(torch, run, calls, flush)
        gbs = w.kv_bytes / (med * 1e-6) / 1e9
        pt = {"us_per_call": round(med, 2), "us_min": round(mn, 2), "kv_bytes": int(w.kv_bytes),
              "GB_per_s": round(gbs, 1), "frac_of_peak": round(gbs / hbm_peak, 4),
              "path": int(pd.info["path"]), "launches": int(pd.info["launches"])}
        if name == "tiny_decode":
            pt["graph_us_per_call"] = round(_time_graph(torch, run, 20, flush), 2)
        if name == "batched_gqa_decode":
            table = torch.as_tensor(w.page_table, device=dev)
            lens = torch.as_tensor(w.seq_lens, device=dev)
            o_b = torch.empty((w.batch, w.q_len, w.num_qo_heads, w.head_dim), device=dev)
            l_b = torch.empty((w.batch, w.q_len, w.num_qo_heads), device=dev)
            b2b, n = _back_to_back_us(torch, w, lambda k, v: pd.run(w.q, k, v, table, lens, o_b, l_b, scale=w.scale))
            g_b = w.kv_bytes / (b2b * 1e-6) / 1e9
            gf = _time_graph(torch, run, 20, flush)
            pt.update({"back_to_back_us_per_call": round(b2b, 2), "back_to_back_GB_per_s": round(g_b, 1),
                       "back_to_back_frac_of_peak": round(g_b / hbm_peak, 4), "back_to_back_pool_copies": n,
                       "graph_flushed_us_per_call": round(gf, 2),
                       "graph_flushed_frac_of_peak": round(w.kv_bytes / (gf * 1e-6) / 1e9 / hbm_peak, 4)})
        points[name] = pt
        del pd, run, w
        torch.cuda.empty_cache()

    # Paged append (the cache's write side): one new token per sequence (a decode
    # step) and a 512-token chunk per sequence (a prefill chunk), 64 sequences of
    # 4096-token capacity, 8 KV heads, D 128.  Bytes = new K and V rows read + written.
    wa = W.make(64, 1, 32, 8, 128, 16, [4096] * 64, dtype="bf16", device=dev, seed=11)
    table = torch.as_tensor(wa.page_table, device=dev)
    app = {}
    for n_per in (1, 512):
        n = 64 * n_per
        k_new = torch.randn(n, 8, 128, device=dev).to(torch.bfloat16)
        v_new = torch.randn(n, 8, 128, device=dev).to(torch.bfloat16)
        bi = torch.arange(64, dtype=torch.int32, device=dev).repeat_interleave(n_per)
        pos = (torch.arange(n_per, dtype=torch.int32, device=dev) + 3000).repeat(64)

        def run_append(k_new=k_new, v_new=v_new, bi=bi, pos=pos):
            fd.fdec_append(k_new, v_new, bi, pos, wa.k, wa.v, table, 16)

        run_append()
        med, mn = _time_calls(torch, run_append, calls, flush)
        nbytes = 2 * 2 * n * 8 * 128 * 2
        app[f"tokens_per_seq_{n_per}"] = {"us_per_call": round(med, 2), "us_min": round(mn, 2), "bytes": nbytes,
                                          "GB_per_s": round(nbytes / (med * 1e-6) / 1e9, 1)}
    points["paged_append"] = app
    del wa, table
    torch.cuda.empty_cache()

    points["long_context_e4m3_L262144"] = _e4m3_point(dev, calls, hbm_peak, flush)
    torch.cuda.empty_cache()
    points["long_context_q8_0_L262144"] = _q8_point(dev, calls, hbm_peak, flush)
    torch.cuda.empty_cache()

    # Graph-replayed long-context points where launch latency matters.
    graph = {}
    for L in (1900, 2000, 2100, 3000, 4800):
        w = W.long_context(L, device=dev)
        pd, run = runner(w)
        graph[str(L)] = round(_time_graph(torch, run, 20, flush), 2)
    points["long_context_graph_us_per_call"] = graph

    # Controlled comparison: the planned split against one split per (sequence, KV
    # head) with no reduction (the serial shape the split path replaces).
    versus = {}
    for L in (2100, 4800, 32768):
        w = W.long_context(L, device=dev)
        pd, run = runner(w)
        planned, _ = _time_calls(torch, run, calls, flush)
        splits = int(pd.info["max_splits"])
        pd1, run1 = runner(w, blocks_per_split=1 << 30)
        single, _ = _time_calls(torch, run1, max(5, calls // 5), flush)
        versus[str(L)] = {"planned_us": round(planned, 2), "planned_splits": splits, "single_split_us": round(single, 2)}
        del pd, run, pd1, run1, w
    points["planned_vs_single_split"] = versus

    # No-cliff sweep over L = 1024 ... 8192 step 64.  Each timed call reads its own
    # pages: one 512 MB pool of K/V pages, call c of a graph getting pages
    # [c * L/64, (c + 1) * L/64) in a shuffled order, so that between two reads of a
    # page the other calls of the graph have streamed about 512 MB (four times the
    # L2) and every call starts from HBM.  The graph of those calls, back to back, is
    # timed as a whole (best of 5 replays): no eviction to subtract, so the per-call
    # figure is not lost in the jitter of a 512 MB flush.
    sweep = []
    hk, D, P = 4, 128, 64
    pool_pages = (512 << 20) // (2 * hk * P * D * 2)
    kp = torch.randn(pool_pages, hk, P, D, device=dev).to(torch.bfloat16)
    vp = torch.randn(pool_pages, hk, P, D, device=dev).to(torch.bfloat16)
    qs = torch.randn(1, 1, 32, D, device=dev).to(torch.bfloat16)
    out = torch.empty((1, 1, 32, D), device=dev)
    lse = torch.empty((1, 1, 32), device=dev)
    gen = torch.Generator(device="cpu").manual_seed(17)
    for L in range(1024, 8192 + 1, 64):
        ppc = L // P
        n = min(256, pool_pages // ppc)
        perm = torch.cat([c * ppc + torch.randperm(ppc, generator=gen) for c in range(n)]).to(torch.int32)
        tables = perm.view(n, ppc).to(dev)
        lens = torch.full((1,), L, dtype=torch.int32, device=dev)
        pd = fd.PagedDecode([L], 1, P, 32, hk, D, "bf16", device=dev)

        def run_all(pd=pd, tables=tables, lens=lens, n=n):
            for c in range(n):
                pd.run(qs, kp, vp, tables[c:c + 1], lens, out, lse)

        run_all()
        torch.cuda.synchronize()
        us = _time_graph_once(torch, run_all) / n
        assert pd.device_errors() == 0
        sweep.append((L, us, int(pd.info["max_splits"])))
        del pd, run_all, tables
    del kp, vp
    torch.cuda.empty_cache()
    ratios = [b[1] / a[1] for a, b in zip(sweep, sweep[1:])]
    gbs = [L * hk * D * 4 / (us * 1e-6) / 1e9 for L, us, _ in sweep]
    changes = [i for i in range(len(sweep) - 1) if sweep[i + 1][2] != sweep[i][2]]
    drops = [(sweep[i + 1][0], round(gbs[i + 1] / gbs[i], 3)) for i in changes if gbs[i + 1] < gbs[i]]
    points["no_cliff_sweep"] = {
        "kv_lens": "1024..8192 step 64 (long-context shape: 32/4 heads, D 128, bf16, page 64)",
        "timing": "per call: a CUDA graph of n back-to-back calls (n = min(256, 512 MB / the call's K/V bytes)), "
                  "each call reading its own pages of a 512 MB pool, best of 5 replays / n",
        "max_adjacent_time_ratio": round(max(ratios), 3),
        "at_kv_len": sweep[int(np.argmax(ratios)) + 1][0],
        "split_changes": len(changes),
        "gbs_drops_at_split_changes": drops,
        "min_gbs_ratio_at_split_changes": round(min(gbs[i + 1] / gbs[i] for i in changes), 3) if changes else None,
        "us_per_call": {str(L): round(us, 3) for L, us, _ in sweep},
        "splits": {str(L): sp for L, _, sp in sweep},
    }
    del flush
    return points


# The sources each profiled kernel is built from: a committed traffic figure
# stands only while these files are unchanged.
KERNEL_SOURCES = {
    "split_mma_persist_kernel": ["device_utils.cuh", "fdec_internal.h", "split_common.cuh", "split_mma_kernel.cuh",
                                 "split_persist_kernel.cuh", "split_persist.cu"],
}
HEADLINE_KERNEL = "split_mma_persist_kernel"


def _kernel_source_hash(kernel: str = HEADLINE_KERNEL) -> str:
    csrc = os.path.join(ROOT, "paged_split_kv_gather_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _traffic_from_profile(workload: str):
    """DRAM bytes per launch of the split kernel from the committed ncu summary,
    only while the kernel sources are the ones that summary was taken from."""
    path = os.path.join(ROOT, "profiles", "split_kernel_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    entry = d.get(workload)
    if not entry or entry.get("kernel_source_hash") != _kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fdec_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: the job is done when its last replica is."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_throughput(world: int, bytes_per_rank_step: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank streams its own replica (weak scaling)."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def _headline_config(world: int, kv_bytes: int) -> dict:
    """The workload config both arms report (identical keys and values)."""
    return {"workload": "long_context_decode_L262144", "batch": 1, "q_len": 1, "num_qo_heads": 32,
            "num_kv_heads": 4, "head_dim": 128, "page_size": 64, "kv_len": HEADLINE_LENGTH,
            "kv_bytes_per_call": kv_bytes, "out": "fp32 out + lse",
            "l2": "inputs larger than L2 (537 MB of K/V per step vs 129 MB L2); every other timed call "
                  "follows a 256 MB write and a 256 MB read that evict the L2 (left holding clean lines)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def _make_inputs(length, device):
    from paged_split_kv_gather_gb300 import workloads as W

    return W.long_context(length, device=device)


def _run_fdec(args):
    import torch
    import torch.distributed as dist

    import paged_split_kv_gather_gb300 as fd

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    if world > 1:
        # Several replicas: the headline step, its roofline and end-to-end numbers only.  The
        # per-workload points characterise one GPU and would hold every GPU for another minute.
        args.no_sweep = args.no_configs = args.no_dense = True
    if args.only_q8:
        # The q8_0 long-context point alone (profiling the q8_0 kernel); not a bench line.
        peak, _ = _peaks()
        pt = _q8_point(dev, args.sweep_calls, peak, L2Flush(torch, dev))
        if rank == 0:
            print(json.dumps({"long_context_q8_0_L262144": pt}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return
    if args.only_e4m3:
        # The quantised-cache long-context point alone (profiling the E4M3 kernel); not a bench line.
        peak, _ = _peaks()
        pt = _e4m3_point(dev, args.sweep_calls, peak, L2Flush(torch, dev))
        if rank == 0:
            print(json.dumps({"long_context_e4m3_L262144": pt}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    if args.only_long:
        # Flushed calls of one long-context length alone (profiling the decode kernel); not a bench line.
        peak, _ = _peaks()
        w = _make_inputs(args.only_long, dev)
        pdl = fd.PagedDecode(w.seq_lens, 1, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype,
                             device=dev)
        tb = torch.as_tensor(w.page_table, device=dev)
        ln = torch.as_tensor(w.seq_lens, device=dev)
        o = torch.empty((1, 1, w.num_qo_heads, w.head_dim), device=dev)
        l = torch.empty((1, 1, w.num_qo_heads), device=dev)

        def run_long():
            pdl.run(w.q, w.k, w.v, tb, ln, o, l, scale=w.scale)

        for _ in range(3):
            run_long()
        med, mn = _time_calls(torch, run_long, args.sweep_calls, L2Flush(torch, dev))
        if rank == 0:
            gbs = w.kv_bytes / (med * 1e-6) / 1e9
            print(json.dumps({f"long_context_L{args.only_long}": {
                "us_per_call": round(med, 2), "us_min": round(mn, 2), "GB_per_s": round(gbs, 1),
                "frac_of_peak": round(gbs / peak, 4), "plan": pdl.info}}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    if args.only_dense:
        # The multi-token points alone (for profiling the tcgen05 kernel); not a bench line.
        peak, _ = _peaks()
        dense = _dense_query(dev, args.sweep_calls, peak, tuple(args.dense_q))
        if rank == 0:
            print(json.dumps({"dense_query": dense}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    from paged_split_kv_gather_gb300 import workloads as W

    w_host = _make_inputs(HEADLINE_LENGTH, "cpu")  # the same draws the CPU baseline reads
    w = w_host.to(dev)
    table = torch.as_tensor(w.page_table, device=dev)
    lens = torch.as_tensor(w.seq_lens, device=dev)
    out = torch.empty((1, 1, w.num_qo_heads, w.head_dim), device=dev)
    lse = torch.empty((1, 1, w.num_qo_heads), device=dev)
    pd = fd.PagedDecode(w.seq_lens, 1, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype,
                        device=dev)
    info = pd.info
    assert info["path"] == fd.FDEC_PATH_MMA, info  # the persistent tensor-core split kernel (HEADLINE_KERNEL)
    kv_bytes = w.kv_bytes

    def step():
        pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale)

    # Clocks are sampled from here to the end of the GPU work: the timed region
    # itself can be shorter than the sampling period (a few ms at small --steps).
    clocks = ClockSampler(local).__enter__()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps back to back, barrier + synchronize on
    # both sides, one event pair around the whole region (an event between the
    # split kernel and the reduction would stop the reduction's programmatic
    # early launch, so none is recorded here).
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)

    # ---- the split kernel alone, for the roofline: the same K steps again with
    # events around each split launch (on the launching stream).
    n_roof = min(args.steps, 2000)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_roof)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(n_roof)]
    for ev in mids:  # created (and marked recorded) here; fdec_run re-records them after each split launch
        ev.record(stream)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e6))  # let the host get ahead of the device
    for i in range(n_roof):
        starts[i].record(stream)
        fd.fdec_plan_set_split_event(pd.plan, mids[i])
        step()
    torch.cuda.synchronize()
    fd.fdec_plan_set_split_event(pd.plan, None)
    split_ms = float(np.mean([s.elapsed_time(m) for s, m in zip(starts, mids)]))
    total_ms = _max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    assert pd.device_errors() == 0, "device-side check fired during the benchmark"

    value = _job_throughput(world, kv_bytes, ms_per_step)
    peak, peak_kind = _peaks()
    achieved = kv_bytes / (split_ms * 1e-3) / 1e9

    # ---- end to end through the public API from pinned host buffers: the step's
    # inputs (q, page table, lengths) staged in one pinned buffer laid out like one
    # device buffer (one host-to-device copy), out and lse in one device buffer (one
    # device-to-host copy): each copy has a fixed cost whatever its size
    st_in = _Staging(torch, dev, [w.q, torch.as_tensor(w.page_table), torch.as_tensor(w.seq_lens)])
    st_res = _Staging(torch, dev, [out, lse])
    d_q, d_table, d_lens = st_in.dev_views
    d_out, d_lse = st_res.dev_views
    e2e_steps = max(10, min(args.steps, 2000))
    for i in range(args.warmup + e2e_steps):
        if i == args.warmup:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        st_in.dev.copy_(st_in.host, non_blocking=True)
        pd.run(d_q, w.k, w.v, d_table, d_lens, d_out, d_lse, scale=w.scale)
        st_res.host.copy_(st_res.dev, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    e2e_py_s = (time.perf_counter() - t0) / e2e_steps
    h2d = st_in.host.numel()
    d2h = st_res.host.numel()
    # The same steps from C (no Python or torch between the calls): the library's own
    # end-to-end cost, the headline e2e number.
    e2e_s = _e2e_from_c(fd, pd, w, st_in, st_res, stream, args.warmup, e2e_steps)
    assert torch.equal(st_res.host_views[0], out.cpu()) and torch.equal(st_res.host_views[1], lse.cpu())

    # ---- the long-context sweep: per-call time with an L2 flush before each call, and back to back
    # over rotating copies of the K/V pools (each call starting with its pages out of L2)
    sweep = []
    if not args.no_sweep:
        flush = L2Flush(torch, dev)
        for length in W.LONG_CONTEXT_LENGTHS:
            ws = w if length == HEADLINE_LENGTH else _make_inputs(length, dev)
            pds = pd if length == HEADLINE_LENGTH else fd.PagedDecode(
                ws.seq_lens, 1, ws.page_size, ws.num_qo_heads, ws.num_kv_heads, ws.head_dim, ws.dtype, device=dev)
            tb = torch.as_tensor(ws.page_table, device=dev)
            ln = torch.as_tensor(ws.seq_lens, device=dev)
            for _ in range(3):
                pds.run(ws.q, ws.k, ws.v, tb, ln, out, lse, scale=ws.scale)
            # All calls are enqueued behind a device-side delay and before one
            # final synchronise, so the device never waits on the host between a
            # call's two events; each call follows an L2 eviction (L2Flush).
            torch.cuda._sleep(int(args.sweep_calls * 2e5))
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.sweep_calls)]
            for a, b in evs:
                flush()
                a.record()
                pds.run(ws.q, ws.k, ws.v, tb, ln, out, lse, scale=ws.scale)
                b.record()
            torch.cuda.synchronize()
            times = [a.elapsed_time(b) * 1e3 for a, b in evs]
            us = float(np.median(times))
            gbs = ws.kv_bytes / (us * 1e-6) / 1e9
            # Back to back (a decode loop): calls in one CUDA graph, each reading its own copy
            # of the pools, every call starting with its pages out of L2 (no per-call events).
            b2b, n = _back_to_back_us(torch, ws, lambda k, v: pds.run(ws.q, k, v, tb, ln, out, lse, scale=ws.scale))
            gbs_b2b = ws.kv_bytes / (b2b * 1e-6) / 1e9
            # Graph-replayed after an L2 eviction: a CUDA graph of 20 (eviction, call) pairs minus a graph of
            # the 20 evictions alone (every call cold, no per-call launch or event).
            gf = _time_graph(torch, lambda: pds.run(ws.q, ws.k, ws.v, tb, ln, out, lse, scale=ws.scale), 20, flush)
            gbs_gf = ws.kv_bytes / (gf * 1e-6) / 1e9
            sweep.append({"kv_len": length, "us_per_call": round(us, 2), "us_min": round(min(times), 2),
                          "GB_per_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                          "back_to_back_us_per_call": round(b2b, 2), "back_to_back_GB_per_s": round(gbs_b2b, 1),
                          "back_to_back_frac_of_peak": round(gbs_b2b / peak, 4), "back_to_back_pool_copies": n,
                          "graph_flushed_us_per_call": round(gf, 2), "graph_flushed_GB_per_s": round(gbs_gf, 1),
                          "graph_flushed_frac_of_peak": round(gbs_gf / peak, 4),
                          "splits": int(pds.info["max_splits"]), "launches": int(pds.info["launches"])})
            if ws is not w:
                del pds, ws
        del flush

    extra = None
    if not args.no_configs:
        extra = _config_points(dev, args.sweep_calls, peak)

    dense = None
    if not args.no_dense:
        dense = _dense_query(dev, args.sweep_calls, peak, tuple(args.dense_q))
        dense["crossover"] = _crossover(dev, max(5, args.sweep_calls // 5))

    clocks.__exit__(None, None, None)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = _cpu_baseline(w_host, kv_bytes, args.cpu_seconds)

    if rank == 0:
        traffic = _traffic_from_profile("long_context_decode_L262144")
        line = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": "GB/s",
            "us_per_call": round(ms_per_step * 1e3, 2),
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded normal q/K/V, 1% spiked keys, shuffled pages)",
            "config": _headline_config(world, kv_bytes),
            "plan": {k: info[k] for k in ("blocks_per_split", "num_split_ctas", "max_splits", "reduce_passes",
                                          "launches")},
            "roofline": {"bound": "hbm", "kernel": f"{HEADLINE_KERNEL}<128,bf16>", "achieved": round(achieved, 1),
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": traffic, "algorithmic_bytes_per_launch": kv_bytes,
                         "split_kernel_us": round(split_ms * 1e3, 2)},
            "e2e": {"value": round(kv_bytes / e2e_s / 1e9, 1), "unit": "GB/s", "us_per_call": round(e2e_s * 1e6, 2),
                    "python_us_per_call": round(e2e_py_s * 1e6, 2),
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "note": "per step: one pinned H2D copy of the staged q, page table and seq_lens, "
                            "fdec_run, one D2H copy of out and lse (one device buffer), stream sync; timed from C "
                            "(value, us_per_call) and through the Python binding with torch copies "
                            "(python_us_per_call); the K/V cache stays resident (decode state)"},
            "gpu_launches": int(info["launches"]) * args.steps,
            "clocks": clocks.summary(),
            "cpu_baseline": cpu,
            "sweep": sweep,
            "dense_query": dense,
            "other_workloads": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


class _Staging:
    """Tensors packed into one pinned host buffer and one device buffer of the same
    layout (each tensor 16-byte aligned), with a view of each on both sides; the host
    views start as copies of the given tensors."""

    def __init__(self, torch, dev, tensors):
        offs, at = [], 0
        for t in tensors:
            offs.append(at)
            at = (at + t.numel() * t.element_size() + 15) // 16 * 16
        self.host = torch.zeros(at, dtype=torch.uint8).pin_memory()
        self.dev = torch.zeros(at, dtype=torch.uint8, device=dev)

        def view(buf, t, off):
            n = t.numel() * t.element_size()
            return buf[off:off + n].view(t.dtype).view(t.shape)

        self.host_views = [view(self.host, t, o) for t, o in zip(tensors, offs)]
        self.dev_views = [view(self.dev, t, o) for t, o in zip(tensors, offs)]
        for hv, t in zip(self.host_views, tensors):
            hv.copy_(t.cpu())


def _e2e_from_c(fd, pd, w, st_in, st_res, stream, warmup, iters) -> float:
    """Seconds per end-to-end step timed by the C loop in libfdec_e2e.so (e2e/e2e_loop.cu)."""
    import ctypes

    lib = ctypes.CDLL(os.path.join(ROOT, "paged_split_kv_gather_gb300", "libfdec_e2e.so"))
    P, I64, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.fdec_e2e_loop.restype = ctypes.c_int
    lib.fdec_e2e_loop.argtypes = [P, P, P, S, P, I64, I64, fd.KVDesc, fd.KVDesc, P, I64, P, ctypes.c_float, P, P,
                                  P, P, S, P, P, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    from paged_split_kv_gather_gb300.workloads import q_token_stride

    d_q, d_table, d_lens = st_in.dev_views
    d_out, d_lse = st_res.dev_views
    secs = ctypes.c_double()
    rc = lib.fdec_e2e_loop(pd.plan.handle, st_in.host.data_ptr(), st_in.dev.data_ptr(), st_in.host.numel(),
                           d_q.data_ptr(), q_token_stride(d_q), d_q.stride(2), fd.kv_desc(w.k), fd.kv_desc(w.v),
                           d_table.data_ptr(), d_table.stride(0), d_lens.data_ptr(), w.scale, d_out.data_ptr(),
                           d_lse.data_ptr(), st_res.dev.data_ptr(), st_res.host.data_ptr(), st_res.host.numel(),
                           pd.workspace.data_ptr(), stream.cuda_stream, warmup, iters, ctypes.byref(secs))
    if rc != 0:
        raise RuntimeError(f"fdec_e2e_loop failed ({rc}): {fd.fdec_last_error()}")
    return secs.value


def _cpu_baseline(c, kv_bytes, seconds):
    """Time the float64 oracle as it stands on this host's cores, over passes of
    the full headline workload (all 32 query rows), until `seconds` have elapsed."""
    import oracle  # test-infrastructure oracle: the reported CPU baseline

    from paged_split_kv_gather_gb300.workloads import q_token_stride, storage_view

    def pool(t):
        base, off, _ = storage_view(t)
        return oracle.Pool(base.view(__import__("torch").int16).numpy().view(np.uint16), off, t.shape[0],
                           t.stride(0), t.stride(1), t.stride(2))

    qb, qoff, _ = storage_view(c.q)
    q_arr = qb.view(__import__("torch").int16).numpy().view(np.uint16)
    kp, vp = pool(c.k), pool(c.v)
    cores = os.cpu_count() or 1

    def one():
        oracle.paged_attention(q_arr, qoff, q_token_stride(c.q), c.q.stride(2), kp, vp, c.page_table, c.seq_lens,
                               q_len=1, num_qo_heads=c.num_qo_heads, num_kv_heads=c.num_kv_heads,
                               head_dim=c.head_dim, page_size=c.page_size, is_bf16=True, causal=False,
                               scale=c.scale, n_threads=cores)

    one()  # warm (page in)
    passes = 0
    t0 = time.perf_counter()
    while True:
        one()
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds or passes >= 1000:
            break
    per = el / passes

    # Single-core times of the two small decode workloads (the oracle with one thread).
    from paged_split_kv_gather_gb300 import workloads as W

    single = {}
    for name, wl in (("tiny_decode", W.tiny()), ("batched_gqa_decode", W.batched_gqa())):
        qa, qo, _ = storage_view(wl.q)
        qn = qa.view(__import__("torch").int16).numpy().view(np.uint16)
        kpw, vpw = pool(wl.k), pool(wl.v)
        t1 = time.perf_counter()
        oracle.paged_attention(qn, qo, q_token_stride(wl.q), wl.q.stride(2), kpw, vpw, wl.page_table, wl.seq_lens,
                               q_len=1, num_qo_heads=wl.num_qo_heads, num_kv_heads=wl.num_kv_heads,
                               head_dim=wl.head_dim, page_size=wl.page_size, is_bf16=(wl.dtype == "bf16"),
                               causal=False, scale=wl.scale, n_threads=1)
        single[name] = round((time.perf_counter() - t1) * 1e3, 2)
    return {"value": round(kv_bytes / per / 1e9, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "ms_per_call": round(per * 1e3, 2), "cpu_model": _cpu_model(),
            "single_core_ms_per_call": single,
            "sample": f"{passes} full passes (all 32 query rows x 262144 tokens) of the headline workload in "
                      f"{el:.1f} s, float64, OpenMP over rows"}


def _cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform

    return platform.processor() or platform.machine()


def _run_reference(args):
    """The reference arm: the float64 CPU oracle, as it stands, on the same workload."""
    world, rank, local = _dist()
    if rank != 0:
        return
    import torch

    import oracle
    from paged_split_kv_gather_gb300.workloads import q_token_stride, storage_view

    c = _make_inputs(HEADLINE_LENGTH, "cpu")
    kv_bytes = c.kv_bytes

    def arr(t):
        base, off, _ = storage_view(t)
        return base.view(torch.int16).numpy().view(np.uint16), off

    def pool(t):
        a, off = arr(t)
        return oracle.Pool(a, off, t.shape[0], t.stride(0), t.stride(1), t.stride(2))

    q_arr, q_off = arr(c.q)
    kp, vp = pool(c.k), pool(c.v)
    cores = os.cpu_count() or 1
    # a bounded sample per step: 8 of the 32 query rows (two per KV head), full length
    rows = np.array([h for h in range(32) if h % 4 == 0], dtype=np.int64)
    frac = len(rows) / 32.0

    def step():
        oracle.paged_attention(q_arr, q_off, q_token_stride(c.q), c.q.stride(2), kp, vp, c.page_table,
                               c.seq_lens, q_len=1, num_qo_heads=32, num_kv_heads=4, head_dim=128, page_size=64,
                               is_bf16=True, causal=False, scale=c.scale, rows=rows, n_threads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    steps = 0
    for _ in range(args.steps):
        step()
        steps += 1
        if time.perf_counter() - t0 > args.reference_seconds:
            break  # bounded: the reference arm must finish within minutes
    el = time.perf_counter() - t0
    args.steps = steps
    per_row_sample = el / steps
    per_call = per_row_sample / frac  # the whole call's rows at the sampled rate
    value = kv_bytes / per_call / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "us_per_call": round(per_call * 1e6, 1), "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per_row_sample * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded normal q/K/V, 1% spiked keys, shuffled pages)",
        "config": _headline_config(world, kv_bytes),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step {len(rows)} of 32 query rows over all 262144 tokens; "
                                   f"value scaled to the whole call"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["fdec", "reference"], default="fdec")
    ap.add_argument("--sweep-calls", type=int, default=50)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-dense", action="store_true", help="skip the multi-token (q_len 4, 8, 2048) points")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads, the no-cliff sweep and the graph-replayed points")
    ap.add_argument("--only-dense", action="store_true",
                    help="run only the multi-token points and print them (profiling; no bench line)")
    ap.add_argument("--dense-q", type=int, nargs="+", default=[4, 8, 2048], help="q_len of the multi-token points")
    ap.add_argument("--only-long", type=int, default=0, metavar="L",
                    help="run only flushed calls of the long-context shape at L tokens and print them "
                         "(profiling; no bench line)")
    ap.add_argument("--only-q8", action="store_true",
                    help="time only the q8_0 long-context point (for profiling); prints that point, not a bench line")
    ap.add_argument("--only-e4m3", action="store_true",
                    help="run only the E4M3 (fp8) long-context point and print it (profiling; no bench line)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=120.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        _run_reference(args)
    else:
        _run_fdec(args)


if __name__ == "__main__":
    main()
