"""q8_0 caches on the GPU (int8 codes in blocks of 32 along head_dim, one binary16
scale per block, scales in pools of their own) against the float64 oracle: head
dims 128 and 256, bf16 and f16 queries, every pool layout, TMA boxes and the
small-page cp.async producer, causal multi-token rows, split plans with
multi-pass reductions, unread rows poisoned with NaN scales, and block scales
far from the drawn range (huge, tiny, zero, negative)."""
import pytest
import torch

import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import assert_parity, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


def _q8(*args, **kw):
    kw.setdefault("kv_dtype", "q8_0")
    return W.make(*args, **kw)


CASES = {
    "long_32768_bf16": lambda: _q8(1, 1, 32, 4, 128, 64, [32768], dtype="bf16", seed=1),
    "gqa_f16_page16": lambda: _q8(4, 1, 32, 8, 128, 16, [2048, 700, 3001, 64], dtype="f16", seed=2),
    "d256_nhd_bf16": lambda: _q8(6, 1, 16, 8, 256, 16, [5000, 17, 900, 2600, 64, 1], dtype="bf16", layout="nhd",
                                 seed=3),
    "causal_rows16_page32": lambda: _q8(3, 4, 16, 4, 128, 32, [3000, 70, 9000], dtype="bf16", causal=True,
                                        peaked=True, seed=4),
    "interleaved_page8": lambda: _q8(2, 1, 16, 2, 128, 8, [1000, 333], dtype="f16", layout="interleaved", seed=5),
    "page4_cp_async_mixed": lambda: _q8(2, 2, 8, 2, 128, 4, [777, 90], dtype="bf16", layout="mixed", causal=True,
                                        seed=6),
    "page1_split2": lambda: _q8(2, 1, 8, 1, 256, 1, [300, 65], dtype="f16", layout="split2", seed=7),
    "page256_interleaved_nhd": lambda: _q8(2, 1, 32, 4, 128, 256, [9000, 513], dtype="bf16",
                                           layout="interleaved_nhd", seed=8),
    "nan_guarded_tails": lambda: _q8(3, 2, 16, 4, 128, 16, [5, 333, 1000], dtype="bf16", causal=True,
                                     nan_guard=True, pool_pages=2 * (1000 // 16 + 8), seed=9),
}


@pytest.mark.parametrize("case", list(CASES))
def test_q8_0_matches_the_oracle(case):
    w = CASES[case]().to("cuda")
    out, lse, pd = gpu_run(w)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0
    assert pd.info["path"] == fd.FDEC_PATH_MMA
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, case)


@pytest.mark.parametrize("bps", [1, 5])
def test_q8_0_under_split_plans_with_multipass_reduction(bps):
    w = _q8(2, 1, 32, 4, 128, 16, [20000, 3000], dtype="bf16", seed=10).to("cuda")
    out, lse, pd = gpu_run(w, blocks_per_split=bps, reducer_fanin=16)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0 and pd.info["reduce_passes"] >= 2
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, f"bps {bps}")


def test_q8_0_block_scales_far_from_the_drawn_range():
    # pages of huge, tiny, zero and negative scales, and single huge scales beside
    # ordinary ones in a stage (each 32-dim block of V is normalised per stage by a
    # power of two above its largest |scale|)
    w = _q8(2, 1, 16, 2, 128, 16, [3000, 1200], dtype="bf16", seed=11)
    for k in range(3000 // 16):
        pg = int(w.page_table[0, k])
        if k % 7 == 1:
            w.v_scales[pg] *= 2.0 ** 12
        elif k % 7 == 2:
            w.v_scales[pg] *= 2.0 ** -12
        elif k % 7 == 3:
            w.v_scales[pg] = 0.0
        elif k % 7 == 4:
            w.v_scales[pg] *= -1.0
        elif k % 7 == 5:
            w.k_scales[pg] *= 4.0  # keys stay where fp32 logits keep lse within 1e-4
    pg = int(w.page_table[1, 5])
    w.v_scales[pg, 1, 3, 2] = 60000.0
    w.k_scales[pg, 0, 9, 1] = -2.0
    wg = w.to("cuda")
    out, lse, pd = gpu_run(wg)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0
    ro, rl = oracle_run(w)
    assert_parity(out.cpu(), lse.cpu(), ro, rl, "extreme scales")


def test_q8_0_plans_refuse_the_16_bit_entry_points():
    w = _q8(1, 1, 8, 2, 128, 16, [100], dtype="bf16", seed=12).to("cuda")
    pd = fd.PagedDecode(w.seq_lens, 1, 16, 8, 2, 128, "bf16", device="cuda", kv_dtype="q8_0")
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    out = torch.empty((1, 1, 8, 128), device="cuda")
    with pytest.raises(fd.FdecError):
        fd.fdec_run(pd.plan, w.q, w.k, w.v, table, lens, out, None, pd.workspace)
    pd16 = fd.PagedDecode(w.seq_lens, 1, 16, 8, 2, 128, "bf16", device="cuda")
    descs = [fd.kv_desc(t) for t in (w.k, w.k_scales, w.v, w.v_scales)]  # past the binding's dtype check
    with pytest.raises(fd.FdecError):
        fd.fdec_run_q8_0(pd16.plan, w.q, *descs, table, lens, out, None, pd16.workspace)


def test_q8_0_decode_loop_captured_in_a_cuda_graph():
    w = _q8(2, 1, 32, 4, 128, 16, [4000, 900], dtype="bf16", seed=13).to("cuda")
    pd = fd.PagedDecode(w.seq_lens, 1, 16, 32, 4, 128, "bf16", device="cuda", kv_dtype="q8_0")
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    out = torch.empty((2, 1, 32, 128), device="cuda")
    lse = torch.empty((2, 1, 32), device="cuda")

    def step():
        pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale, k_scales=w.k_scales, v_scales=w.v_scales)

    step()
    torch.cuda.synchronize()
    eager = (out.clone(), lse.clone())
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pd.device_errors() == 0
    assert torch.equal(out, eager[0]) and torch.equal(lse, eager[1])
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, "graph")
