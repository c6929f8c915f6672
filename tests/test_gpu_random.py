"""Seeded random configurations against the float64 oracle: batch, q_len, heads,
head_dim, page size, pool layout, q layout, 16-bit dtype, cache type (16-bit,
E4M3 with scales, q8_0), causal mask, run-time lengths below capacity, split
plan, reduction fan-in and path are drawn per case, with every unread slot of
the pools poisoned with NaN, so combinations that no hand-written case names
still meet the oracle (and the input buffers stay bit-identical)."""
import numpy as np
import pytest
import torch

import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import assert_parity, gpu_run, oracle_run

pytestmark = pytest.mark.gpu

LAYOUTS = ("hnd", "nhd", "mixed", "interleaved", "split2", "interleaved_nhd")


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    kv_dtype = ["", "", "fp8", "q8_0"][rng.integers(4)]
    if kv_dtype:
        d = int(rng.choice([128, 256]))
    else:
        d = int(rng.choice([64, 128, 192, 256, 512]))
    hk = int(rng.choice([1, 2, 4]))
    group = int(rng.choice([1, 2, 4, 8]))
    q_len = int(rng.choice([1, 1, 2, 3, 5, 8, 16]))
    batch = int(rng.integers(1, 5))
    page = int(rng.choice([1, 4, 8, 16, 32, 64, 256]))
    lens = [int(x) for x in rng.integers(0, 2600, batch)]
    lens[0] = max(lens[0], q_len)
    causal = bool(q_len > 1 and rng.integers(2))
    layout = str(rng.choice(LAYOUTS))
    dtype = str(rng.choice(["bf16", "f16"]))
    q_layout = str(rng.choice(["packed", "fused_qkv", "head_major"]))
    path = fd.FDEC_PATH_AUTO
    if not kv_dtype and rng.integers(3) == 0:
        path = int(rng.choice([fd.FDEC_PATH_MMA, fd.FDEC_PATH_SIMT] + ([fd.FDEC_PATH_TC] if d <= 256 else [])))
    bps = int(rng.choice([0, 0, 1, 3, 7]))
    shorter = bool(rng.integers(3) == 0)  # run-time lengths below the planned capacities
    fanin = int(rng.choice([0, 0, 2, 5, 16]))
    scales = (float(rng.choice([0.5, 1.0, 3.0])), float(rng.choice([0.25, 1.0, 2.0]))) if kv_dtype == "fp8" else None
    return dict(batch=batch, q_len=q_len, hq=hk * group, hk=hk, d=d, page=page, lens=lens, causal=causal,
                layout=layout, dtype=dtype, q_layout=q_layout, kv_dtype=kv_dtype, path=path, bps=bps,
                shorter=shorter, fanin=fanin, scales=scales, seed=seed)


@pytest.mark.parametrize("seed", range(80))
def test_random_configuration_matches_the_oracle(seed):
    c = _draw(seed)
    w = W.make(c["batch"], c["q_len"], c["hq"], c["hk"], c["d"], c["page"], c["lens"], dtype=c["dtype"],
               layout=c["layout"], causal=c["causal"], seed=seed, q_layout=c["q_layout"], kv_dtype=c["kv_dtype"],
               nan_guard=True).to("cuda")
    caps = np.asarray(c["lens"], dtype=np.int32)
    run_lens = caps
    if c["shorter"]:
        run_lens = np.maximum(caps - np.arange(1, c["batch"] + 1) * 37, 0).astype(np.int32)
    ks, vs = c["scales"] or (None, None)
    out, lse, pd = gpu_run(w, capacities=caps, seq_lens=run_lens, path=c["path"], blocks_per_split=c["bps"],
                           reducer_fanin=c["fanin"], k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0, c
    ro, rl = oracle_run(w.to("cpu"), seq_lens=run_lens, k_scale=ks or 1.0, v_scale=vs or 1.0)
    assert_parity(out.cpu(), lse.cpu(), ro, rl, str(c))
