"""CUDA path vs the float64 oracle, element by element, on seeded inputs.

Tolerance (fp32 accumulation over 16-bit K/V): per output row,
||out - ref||_inf / ||ref||_inf <= 2e-3, and |lse - ref| <= 1e-4.
"""
import numpy as np
import pytest
import torch

import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import assert_parity, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


def _check(w_gpu, rows=None, **plan_opts):
    out, lse, pd = gpu_run(w_gpu, **plan_opts)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0
    w_cpu = w_gpu.to("cpu")
    if rows is None:
        ref_o, ref_l = oracle_run(w_cpu)
        got_o, got_l = out.cpu(), lse.cpu()
    else:
        ref_o, ref_l = oracle_run(w_cpu, rows=rows)
        flat_o = out.reshape(-1, w_gpu.head_dim).cpu()
        flat_l = lse.reshape(-1).cpu()
        idx = torch.as_tensor(np.asarray(rows, dtype=np.int64))
        got_o, got_l = flat_o[idx], flat_l[idx]
    return assert_parity(got_o, got_l, ref_o, ref_l, w_gpu.name), pd


# ------------------------------------------------------------------ the five workloads

def test_tiny_decode():
    _check(W.tiny(device="cuda"))


@pytest.mark.parametrize("peaked", [False, True])
def test_batched_gqa_decode(peaked):
    _check(W.batched_gqa(device="cuda", peaked=peaked))


@pytest.mark.parametrize("length", W.LONG_CONTEXT_LENGTHS)
def test_long_context_sweep(length):
    _check(W.long_context(length, device="cuda"))


@pytest.mark.parametrize("length", [2048, 2049, 4864, 32768])
def test_long_context_peaked(length):
    _check(W.long_context(length, device="cuda", peaked=True))


def _ragged_rows(w, per_seq=2):
    rows = []
    for b in range(w.batch):
        for j in range(per_seq):
            h = (b * 7 + j * 5) % w.num_qo_heads
            rows.append(b * w.num_qo_heads + h)
    return rows


@pytest.mark.parametrize("head_dim", W.RAGGED_HEAD_DIMS)
@pytest.mark.parametrize("layout", ["interleaved", "split2"])
def test_ragged_serving_batch_full_size_sampled(head_dim, layout):
    w = W.ragged(head_dim, device="cuda", layout=layout)
    before = [t.clone() for t in w.keep[1:]]
    _check(w, rows=_ragged_rows(w))
    for a, b in zip(before, w.keep[1:]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "the KV cache changed"


@pytest.mark.parametrize("q_len", [4, 8])
def test_multi_token_spec_decode(q_len):
    _check(W.multi_token(q_len, device="cuda"))


def test_multi_token_prefill_chunk_sampled_rows():
    # every 16th query position plus the last, on one query head of every KV head (the 8
    # heads step through the groups), and every query head at the tile and CTA boundaries
    # (query rows of one 128-row tile are 32 positions x 4 heads; a CTA holds two tiles)
    w = W.multi_token(2048, device="cuda")
    strided = sorted(set(range(0, w.q_len, 16)) | {w.q_len - 1})
    boundary = [0, 1, 31, 32, 63, 64, 127, 128, 1000, 2046, 2047]
    spread_heads = [5 * k % w.num_qo_heads if k < 4 else 16 + 5 * (k - 4) for k in range(8)]
    assert sorted({h // w.group for h in spread_heads}) == list(range(w.num_kv_heads))
    rows = set()
    for b in range(w.batch):
        for i in strided:
            rows.update((b * w.q_len + i) * w.num_qo_heads + h for h in spread_heads)
        for i in boundary:
            rows.update((b * w.q_len + i) * w.num_qo_heads + h for h in range(w.num_qo_heads))
    (e_out, e_lse), pd = _check(w, rows=sorted(rows))
    assert pd.info["path"] == fd.FDEC_PATH_TC


# ------------------------------------------------------------------ both split kernels

PATHS = [fd.FDEC_PATH_SIMT, fd.FDEC_PATH_MMA]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", ["tiny", "gqa", "L2049", "L131072", "spec4", "spec8", "peaked"])
def test_fp32_simt_and_tensor_core_kernels(path, case):
    w = {"tiny": lambda: W.tiny(device="cuda"),
         "gqa": lambda: W.batched_gqa(device="cuda"),
         "L2049": lambda: W.long_context(2049, device="cuda"),
         "L131072": lambda: W.long_context(131072, device="cuda"),
         "spec4": lambda: W.multi_token(4, device="cuda"),
         "spec8": lambda: W.multi_token(8, device="cuda"),
         "peaked": lambda: W.long_context(4800, device="cuda", peaked=True)}[case]()
    (e_out, e_lse), pd = _check(w, path=path)
    assert pd.info["path"] == path


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("page_size", [1, 4, 16, 128])
def test_both_kernels_small_and_large_pages_with_nan_guard(path, page_size):
    w = W.make(3, 2, 16, 4, 128, page_size, [5, 333, 1000], dtype="bf16", device="cuda", seed=page_size,
               causal=True, nan_guard=True, pool_pages=2 * (1000 // page_size + 8))
    out, lse, pd = gpu_run(w, path=path, blocks_per_split=3)
    assert torch.isfinite(out).all()
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, f"path {path} page {page_size}")


# ------------------------------------------------------------------ the tcgen05 dense-query kernel

TC_CASES = {
    # q_len x group = 64: half of one 128-row tile; short and ragged sequences
    "half_tile": lambda: W.make(2, 16, 32, 8, 128, 16, [300, 1000], dtype="bf16", device="cuda", seed=11,
                                causal=True),
    # 160 rows: one full tile and a ragged one (row groups 2)
    "ragged_tile": lambda: W.make(2, 40, 16, 4, 128, 16, [2100, 777], dtype="bf16", device="cuda", seed=12,
                                  causal=True),
    "not_causal": lambda: W.make(2, 32, 8, 2, 128, 16, [1500, 4100], dtype="bf16", device="cuda", seed=13),
    "f16": lambda: W.make(2, 64, 8, 4, 128, 32, [900, 3000], dtype="f16", device="cuda", seed=14, causal=True),
    # 384 rows: a CTA of two tiles and a CTA whose second tile is empty
    "f16_two_tiles": lambda: W.make(2, 96, 8, 2, 128, 32, [700, 2500], dtype="f16", device="cuda", seed=19,
                                    causal=True),
    "peaked": lambda: W.make(1, 64, 8, 2, 128, 64, [6000], dtype="bf16", device="cuda", seed=15, causal=True,
                             peaked=True),
    "gqa_group1": lambda: W.make(1, 128, 4, 4, 128, 16, [2000], dtype="bf16", device="cuda", seed=16,
                                 causal=True),
    # sequences shorter than the query chunk: leading rows see nothing
    "short": lambda: W.make(3, 64, 4, 1, 128, 16, [0, 20, 64], dtype="bf16", device="cuda", seed=17,
                            causal=True),
    "hnd_interleaved": lambda: W.make(2, 32, 8, 2, 128, 16, [1234, 640], dtype="bf16", device="cuda", seed=18,
                                      causal=True, layout="interleaved"),
    # other head dims: 64 (two tiles per CTA), 192 and 256 (one tile; P V of N = 192 / 256)
    "d64_two_tiles": lambda: W.make(2, 96, 8, 2, 64, 16, [700, 2500], dtype="bf16", device="cuda", seed=31,
                                    causal=True),
    "d64_f16_page64": lambda: W.make(2, 20, 16, 4, 64, 64, [4000, 130], dtype="f16", device="cuda", seed=32,
                                     causal=True),
    "d192_ragged_tile": lambda: W.make(2, 40, 16, 4, 192, 16, [2100, 777], dtype="f16", device="cuda", seed=33,
                                       causal=True),
    "d192_bf16": lambda: W.make(1, 64, 8, 2, 192, 64, [5000], dtype="bf16", device="cuda", seed=34, causal=True),
    "d256": lambda: W.make(2, 32, 8, 2, 256, 32, [1500, 4100], dtype="bf16", device="cuda", seed=35, causal=True),
    "d256_peaked_f16": lambda: W.make(1, 64, 8, 2, 256, 64, [3000], dtype="f16", device="cuda", seed=36,
                                      causal=True, peaked=True),
    "d256_not_causal": lambda: W.make(3, 8, 32, 4, 256, 16, [900, 64, 2600], dtype="bf16", device="cuda", seed=37),
}


@pytest.mark.parametrize("case", list(TC_CASES))
def test_tcgen05_dense_query_kernel(case):
    w = TC_CASES[case]()
    (e_out, e_lse), pd = _check(w, path=fd.FDEC_PATH_TC)
    assert pd.info["path"] == fd.FDEC_PATH_TC


def test_tcgen05_bf16_v_slices_outside_the_f16_range():
    # bf16 V slices (16 tokens = one page here) that f16 cannot hold within the kernel's
    # rule -- values above 65504, a slice of values all below 2^-10, one outlier in an
    # otherwise ordinary slice -- keep the two-product P V; the others run as f16.
    w = W.make(2, 16, 32, 8, 128, 16, [3000, 700], dtype="bf16", device="cpu", seed=41, causal=True)
    for k in range(3000 // 16):
        pg = int(w.page_table[0, k])
        if k % 5 == 1:
            w.v[pg] *= 2.0 ** 17
        elif k % 5 == 3:
            w.v[pg] *= 2.0 ** -18
    w.v[int(w.page_table[1, 2]), 0, 7, 5] = 1.0e6
    (e_out, e_lse), pd = _check(w.to("cuda"), path=fd.FDEC_PATH_TC)
    assert pd.info["path"] == fd.FDEC_PATH_TC


@pytest.mark.parametrize("bps", [1, 3, 10**6])
def test_tcgen05_kernel_under_any_split_plan(bps):
    w = W.make(2, 48, 8, 2, 128, 16, [3000, 5000], dtype="bf16", device="cuda", seed=21, causal=True,
               peaked=True)
    (e_out, e_lse), pd = _check(w, path=fd.FDEC_PATH_TC, blocks_per_split=bps)
    if bps == 1:
        assert pd.info["max_splits"] == 79


@pytest.mark.parametrize("head_dim", [128, 256])
@pytest.mark.parametrize("page_size", [1, 4, 8, 16, 64, 128, 256])
def test_tcgen05_kernel_page_sizes_with_nan_guard(page_size, head_dim):
    w = W.make(3, 40, 16, 4, head_dim, page_size, [5, 333, 1000], dtype="bf16", device="cuda", seed=page_size,
               causal=True, nan_guard=True, pool_pages=2 * (1000 // page_size + 8))
    out, lse, pd = gpu_run(w, path=fd.FDEC_PATH_TC, blocks_per_split=3)
    assert pd.info["path"] == fd.FDEC_PATH_TC
    assert torch.isfinite(out).all()
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, f"tcgen05 page {page_size}")


def test_tcgen05_and_mma_kernels_agree_on_the_prefill_chunk():
    w = W.multi_token(2048, device="cuda")
    o_tc, l_tc, pd = gpu_run(w)
    assert pd.info["path"] == fd.FDEC_PATH_TC
    o_mma, l_mma, pd2 = gpu_run(w, path=fd.FDEC_PATH_MMA)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0 and pd2.device_errors() == 0
    # both within the oracle tolerance of each other on every row (not only the sampled ones)
    d = (o_tc - o_mma).abs().amax(dim=-1) / o_mma.abs().amax(dim=-1)
    assert float(d.max()) <= 2 * 2e-3
    assert float((l_tc - l_mma).abs().max()) <= 2 * 1e-4


@pytest.mark.parametrize("head_dim", [256, 512])
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("page_size", [4, 16, 64])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_large_head_dims_on_both_kernels(head_dim, path, page_size, dtype):
    # 3 q positions x 6 heads per KV head = 18 rows: two 16-row groups on the tensor-core kernel;
    # head_dim 512 splits O between the two warps of each consumer group
    w = W.make(3, 3, 12, 2, head_dim, page_size, [7, 400, 1500], dtype=dtype, device="cuda",
               seed=page_size + head_dim, causal=True, nan_guard=True, pool_pages=2 * (1500 // page_size + 8),
               peaked=True)
    out, lse, pd = gpu_run(w, path=path, blocks_per_split=2)
    assert pd.info["path"] == path
    torch.cuda.synchronize()
    assert pd.device_errors() == 0 and torch.isfinite(out).all()
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, f"D{head_dim} path {path} page {page_size} {dtype}")


# ------------------------------------------------------------------ plans and reductions

@pytest.mark.parametrize("bps,fanin", [(1, 0), (1, 4), (3, 2), (7, 0), (10**6, 0)])
def test_any_split_plan_matches_the_oracle(bps, fanin):
    w = W.long_context(4800, device="cuda", peaked=True)
    (e_out, e_lse), pd = _check(w, blocks_per_split=bps, reducer_fanin=fanin)
    info = pd.info
    if bps == 1:
        assert info["max_splits"] == 75
    if bps >= 10**6:
        assert info["max_splits"] == 1 and info["reduce_passes"] == 0


def test_multipass_reduction_at_262144_with_one_partial_per_block():
    w = W.long_context(262144, device="cuda")
    (e_out, e_lse), pd = _check(w, blocks_per_split=1)
    assert pd.info["max_splits"] == 4096 and pd.info["reduce_passes"] == 2


def test_split_plans_agree_with_each_other():
    w = W.long_context(32768, device="cuda")
    outs = []
    for bps in (1, 5, 64, 512):
        out, lse, _ = gpu_run(w, blocks_per_split=bps)
        outs.append((out, lse))
    ref = outs[-1]
    for out, lse in outs[:-1]:
        assert torch.max(torch.abs(out - ref[0])) / torch.max(torch.abs(ref[0])) < 1e-3
        assert torch.max(torch.abs(lse - ref[1])) < 1e-4


def test_results_are_deterministic_for_a_fixed_plan():
    w = W.batched_gqa(device="cuda")
    a, la, pd = gpu_run(w)
    b = torch.empty_like(a)
    lb = torch.empty_like(la)
    pd.run(w.q, w.k, w.v, torch.as_tensor(w.page_table, device="cuda"),
           torch.as_tensor(w.seq_lens, device="cuda"), b, lb, scale=w.scale)
    assert torch.equal(a, b) and torch.equal(la, lb)


# ------------------------------------------------------------------ layouts (read-only cache)

LAYOUTS = ["hnd", "nhd", "interleaved", "split2", "mixed", "interleaved_nhd"]


def _relayout(w, layout):
    """Same K/V values, another physical layout."""
    w2 = W.make(w.batch, w.q_len, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, w.seq_lens,
                dtype=w.dtype, layout=layout, causal=w.causal, device=w.q.device, pool_pages=w.k.shape[0],
                seed=999)
    w2.page_table = w.page_table.copy()
    w2.q = w.q
    w2.k.copy_(w.k)
    w2.v.copy_(w.v)
    return w2


def test_every_kv_layout_gives_bitwise_identical_results_and_leaves_the_cache_unchanged():
    base = W.make(3, 1, 16, 4, 128, 16, [700, 33, 2100], dtype="bf16", device="cuda", seed=5, peaked=True)
    ref_out, ref_lse, _ = gpu_run(base, blocks_per_split=4)
    for layout in LAYOUTS:
        w = _relayout(base, layout)
        snap = [t.clone() for t in w.keep]
        out, lse, _ = gpu_run(w, blocks_per_split=4)
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), layout
        for a, b in zip(snap, w.keep):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{layout}: cache written"
    w_cpu = base.to("cpu")
    ro, rl = oracle_run(w_cpu)
    assert_parity(ref_out.cpu(), ref_lse.cpu(), ro, rl, "layouts")


@pytest.mark.parametrize("q_layout", ["fused_qkv", "head_major"])
def test_strided_q_matches_packed_q(q_layout):
    w = W.make(3, 2, 8, 2, 64, 16, [90, 130, 64], dtype="f16", device="cuda", seed=8, causal=True,
               q_layout=q_layout, peaked=True)
    out, lse, _ = gpu_run(w)
    packed = w.q.contiguous()
    w2 = W.Workload(w.name, w.dtype, w.batch, w.q_len, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size,
                    w.causal, w.scale, w.seq_lens, w.page_table, packed, w.k, w.v, w.layout, w.keep)
    out2, lse2, _ = gpu_run(w2)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, q_layout)


def test_shorter_v_pool_only_indexed_pages_are_read():
    w = W.make(2, 1, 8, 2, 128, 16, [200, 90], dtype="bf16", device="cuda", seed=3, pool_pages=40)
    used = int(w.page_table.max()) + 1
    w.v = w.v[:used].clone()  # V holds only the pages the table uses
    out, lse, pd = gpu_run(w)
    assert pd.device_errors() == 0
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, "short V pool")


def test_unread_slots_and_pages_may_hold_nan():
    w = W.make(4, 1, 16, 4, 128, 16, [33, 1, 500, 64], dtype="bf16", device="cuda", seed=12, pool_pages=80,
               nan_guard=True)
    out, lse, _ = gpu_run(w, blocks_per_split=1)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, "nan guard")


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("head_dim", [64, 128, 192, 256, 512])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_head_dims_and_dtypes(head_dim, dtype):
    w = W.make(3, 1, 8, 2, head_dim, 16, [1, 95, 321], dtype=dtype, device="cuda", seed=head_dim, peaked=True)
    _check(w)
    _check(w, blocks_per_split=1)


@pytest.mark.parametrize("page_size", [1, 2, 8, 32, 64, 128, 256])
def test_page_sizes(page_size):
    w = W.make(2, 1, 8, 4, 64, page_size, [257, 1000], dtype="f16", device="cuda", seed=page_size)
    _check(w)


@pytest.mark.parametrize("group,q_len", [(1, 1), (3, 1), (5, 2), (16, 1), (8, 3)])
def test_group_sizes_and_row_groups(group, q_len):
    w = W.make(2, q_len, 2 * group, 2, 128, 16, [150, 77], dtype="bf16", device="cuda", seed=group,
               causal=q_len > 1)
    _check(w)


def test_empty_sequences_and_rows_with_nothing_visible():
    w = W.make(3, 1, 4, 2, 64, 16, [0, 5, 0], dtype="f16", device="cuda", seed=1)
    out, lse, _ = gpu_run(w)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert torch.all(torch.isneginf(lse[0])) and torch.all(torch.isneginf(lse[2]))
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, "empty")
    w = W.make(1, 6, 2, 1, 64, 16, [3], dtype="f16", device="cuda", seed=2, causal=True)
    out, lse, _ = gpu_run(w)
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, "causal-empty rows")


def test_run_time_lengths_below_capacity():
    caps = np.array([5000, 3000, 700], dtype=np.int32)
    w = W.make(3, 1, 16, 4, 128, 16, caps, dtype="bf16", device="cuda", seed=4)
    for lens in ([4999, 3000, 1], [64, 65, 0], [2048, 2049, 700]):
        lens = np.array(lens, dtype=np.int32)
        out, lse, _ = gpu_run(w, capacities=caps, seq_lens=lens, blocks_per_split=3)
        ro, rl = oracle_run(w.to("cpu"), seq_lens=lens)
        assert_parity(out.cpu(), lse.cpu(), ro, rl, f"lens {lens}")


# ------------------------------------------------------------------ device-side checks

def test_out_of_range_page_id_is_flagged_not_read():
    w = W.make(1, 1, 4, 1, 64, 16, [100], dtype="f16", device="cuda", seed=1)
    w.page_table[0, 2] = w.k.shape[0] + 5
    out, lse, pd = gpu_run(w)
    torch.cuda.synchronize()
    assert pd.device_errors() & fd.DEVERR_PAGE_ID
    assert pd.device_errors() == 0  # cleared by the first read


def test_length_above_capacity_is_flagged_and_clamped():
    w = W.make(1, 1, 4, 1, 64, 16, [100], dtype="f16", device="cuda", seed=1, pool_pages=20)
    out, lse, pd = gpu_run(w, capacities=[100], seq_lens=[300])
    torch.cuda.synchronize()
    assert pd.device_errors() & fd.DEVERR_SEQ_LEN
    ro, rl = oracle_run(w.to("cpu"))
    assert_parity(out.cpu(), lse.cpu(), ro, rl, "clamped")


# ------------------------------------------------------------------ merge of states

@pytest.mark.parametrize("n", [1, 2, 7, 33, 100])
def test_merge_states_matches_the_oracle_merge(n):
    import oracle

    rng = np.random.default_rng(n)
    rows, d = 37, 128
    o = rng.standard_normal((n, rows, d)).astype(np.float32)
    l = (rng.standard_normal((n, rows)) * 4).astype(np.float32)
    l[0, 3] = -np.inf
    if n > 1:
        l[:, 5] = -np.inf   # a row where every state is empty
    ot, lt = torch.as_tensor(o, device="cuda"), torch.as_tensor(l, device="cuda")
    oo = torch.empty((rows, d), device="cuda")
    lo = torch.empty((rows,), device="cuda")
    fd.fdec_merge_states(ot, lt, oo, lo)
    ro, rl = oracle.merge_states(o.astype(np.float64), l.astype(np.float64))
    assert_parity(oo.cpu(), lo.cpu(), ro, rl, f"merge n={n}")


def test_two_runs_over_disjoint_ranges_merge_to_the_whole():
    # cascade: attend to a prefix and a suffix separately, merge the states
    w = W.make(1, 1, 8, 2, 128, 16, [1000], dtype="bf16", device="cuda", seed=6, peaked=True)
    full_o, full_l, _ = gpu_run(w)
    cut_pages = 640 // 16
    pre = W.Workload(w.name, w.dtype, 1, 1, 8, 2, 128, 16, False, w.scale, np.array([640], np.int32),
                     w.page_table[:, :cut_pages].copy(), w.q, w.k, w.v)
    suf = W.Workload(w.name, w.dtype, 1, 1, 8, 2, 128, 16, False, w.scale, np.array([360], np.int32),
                     w.page_table[:, cut_pages:].copy(), w.q, w.k, w.v)
    o1, l1, _ = gpu_run(pre)
    o2, l2, _ = gpu_run(suf)
    oo = torch.empty((8, 128), device="cuda")
    lo = torch.empty((8,), device="cuda")
    fd.fdec_merge_states(torch.stack([o1.reshape(8, 128), o2.reshape(8, 128)]).contiguous(),
                         torch.stack([l1.reshape(8), l2.reshape(8)]).contiguous(), oo, lo)
    assert torch.max(torch.abs(oo - full_o.reshape(8, 128))) / torch.max(torch.abs(full_o)) < 1e-4
    assert torch.max(torch.abs(lo - full_l.reshape(8))) < 1e-5


@pytest.mark.parametrize("kv_dtype", ["", "fp8", "q8_0"])
def test_rows_that_see_nothing_of_a_consumer_groups_only_stage(kv_dtype):
    # One 64-token block per split, run-time lengths below capacity and a causal
    # 5-token query: the last split of a sequence has a stage past the early rows'
    # limits that is its consumer group's only stage, while later rows of the same
    # warp see tokens there.  Those early rows must keep an empty state (their
    # running max is still -inf), not a NaN sum that empties the whole row.
    w = W.make(2, 5, 4, 1, 128, 8, [617, 1452], dtype="bf16", causal=True, seed=6, kv_dtype=kv_dtype,
               q_layout="fused_qkv").to("cuda")
    run_lens = np.asarray([580, 1378], dtype=np.int32)
    out, lse, pd = gpu_run(w, capacities=np.asarray([617, 1452], dtype=np.int32), seq_lens=run_lens,
                           blocks_per_split=1, path=fd.FDEC_PATH_MMA if not kv_dtype else fd.FDEC_PATH_AUTO)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0 and pd.info["path"] == fd.FDEC_PATH_MMA
    ro, rl = oracle_run(w.to("cpu"), seq_lens=run_lens)
    assert_parity(out.cpu(), lse.cpu(), ro, rl, kv_dtype or "16-bit")
