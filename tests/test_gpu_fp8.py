"""Quantised (E4M3) KV caches on the GPU against the oracle, and the scaled entry
point on 16-bit caches on every path.  The oracle decodes each stored code from
the E4M3 definition and applies k_scale / v_scale in float64."""
import numpy as np
import pytest
import torch

import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import assert_parity, gpu_run, oracle_run

pytestmark = pytest.mark.gpu

K_SCALE, V_SCALE = 0.6, 1.7


@pytest.mark.parametrize("d,dtype,page,layout", [
    (128, "bf16", 16, "hnd"),
    (128, "f16", 16, "nhd"),
    (128, "bf16", 64, "split2"),
    (128, "bf16", 256, "interleaved"),
    (128, "bf16", 1, "interleaved"),   # pages under 8 tokens: cp.async staging
    (128, "f16", 4, "hnd"),
    (256, "bf16", 16, "hnd"),
    (256, "f16", 64, "interleaved"),
    (256, "bf16", 2, "nhd"),
])
def test_e4m3_cache_matches_the_oracle(d, dtype, page, layout):
    w = W.make(3, 1, 32, 8, d, page, [1000, 77, 2500], dtype=dtype, kv_dtype="fp8", layout=layout,
               device="cuda", seed=d + page, peaked=True, nan_guard=True)
    out, lse, pd = gpu_run(w, k_scale=K_SCALE, v_scale=V_SCALE)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0 and pd.info["path"] == fd.FDEC_PATH_MMA
    ro, rl = oracle_run(w.to("cpu"), k_scale=K_SCALE, v_scale=V_SCALE)
    assert_parity(out, lse, ro, rl, f"e4m3 D{d} {dtype} P{page} {layout}")


@pytest.mark.parametrize("bps", [0, 1, 7])
def test_e4m3_split_plans_and_row_groups(bps):
    # q_len 4 x group 8 = 32 rows: two 16-row groups; causal bottom-right
    w = W.make(2, 4, 32, 4, 128, 16, [9000, 700], dtype="bf16", kv_dtype="fp8", device="cuda", seed=bps,
               causal=True, peaked=True)
    out, lse, pd = gpu_run(w, k_scale=K_SCALE, v_scale=V_SCALE, blocks_per_split=bps)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0 and pd.info["row_groups"] == 2
    ro, rl = oracle_run(w.to("cpu"), k_scale=K_SCALE, v_scale=V_SCALE)
    assert_parity(out, lse, ro, rl, f"e4m3 splits bps={bps}")


def test_e4m3_long_context_sampled_rows():
    w = W.make(1, 1, 32, 4, 128, 64, [65536], dtype="bf16", kv_dtype="fp8", device="cuda", seed=5, spikes=0.01)
    out, lse, pd = gpu_run(w, k_scale=K_SCALE, v_scale=V_SCALE)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0 and pd.info["max_splits"] > 1
    rows = np.array([0, 7, 8, 19, 31])
    ro, rl = oracle_run(w.to("cpu"), rows=rows, k_scale=K_SCALE, v_scale=V_SCALE)
    assert_parity(out.reshape(-1, 128)[rows], lse.reshape(-1)[rows], ro, rl, "e4m3 L65536")


@pytest.mark.parametrize("path,q_len", [(fd.FDEC_PATH_MMA, 1), (fd.FDEC_PATH_TC, 8), (fd.FDEC_PATH_SIMT, 1)])
def test_scaled_run_on_16bit_caches(path, q_len):
    w = W.make(2, q_len, 32, 8, 128, 16, [1500, 300], dtype="bf16", device="cuda", seed=q_len, causal=q_len > 1,
               peaked=True)
    out, lse, pd = gpu_run(w, k_scale=K_SCALE, v_scale=V_SCALE, path=path)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0 and pd.info["path"] == path
    ro, rl = oracle_run(w.to("cpu"), k_scale=K_SCALE, v_scale=V_SCALE)
    assert_parity(out, lse, ro, rl, f"scaled 16-bit path {path}")
