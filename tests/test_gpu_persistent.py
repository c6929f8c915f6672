"""The persistent split kernel (resident CTAs taking work units from a counter)
against the one-CTA-per-item kernel and the oracle.

Both kernels run the same plan: the persistent one when q's rows are 16-byte
aligned, the other when they are not (q offset by one element).  A unit is
computed by the same code in the same order whichever CTA takes it, so the two
must agree bit for bit, call after call (the ticket counter carries over from
call to call and must hand out every unit exactly once each time)."""
import numpy as np
import pytest
import torch

import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import assert_parity, oracle_run

pytestmark = pytest.mark.gpu


def _misaligned_copy(q):
    """The same values as q, with rows that start 2 bytes past a 16-byte boundary."""
    flat = torch.empty(q.numel() + 1, dtype=q.dtype, device=q.device)
    qm = flat[1:].view(q.shape)
    qm.copy_(q)
    assert qm.data_ptr() % 16 != 0
    return qm


def _run(pd, w, q, table, lens):
    out = torch.full((w.batch, w.q_len, w.num_qo_heads, w.head_dim), float("nan"), device="cuda")
    lse = torch.full((w.batch, w.q_len, w.num_qo_heads), float("nan"), device="cuda")
    pd.run(q, w.k, w.v, table, lens, out, lse, scale=w.scale)
    return out, lse


CASES = {
    "long_32768": lambda: W.long_context(32768, device="cuda"),
    "long_131072": lambda: W.long_context(131072, device="cuda"),
    "gqa": lambda: W.batched_gqa(device="cuda"),
    "tiny_d64": lambda: W.tiny(device="cuda"),
    "ragged_d192": lambda: W.ragged(192, device="cuda"),
    "spec4_causal": lambda: W.multi_token(4, device="cuda"),
    "page1_f16": lambda: W.make(3, 1, 8, 2, 128, 1, [700, 64, 2050], dtype="f16", device="cuda", seed=5),
    "page4_rows32": lambda: W.make(2, 2, 32, 2, 64, 4, [3000, 4500], dtype="bf16", causal=True, device="cuda",
                                   seed=6),
    "page256_nhd": lambda: W.make(2, 1, 16, 4, 128, 256, [20000, 9000], dtype="bf16", layout="nhd", device="cuda",
                                  seed=7),
    "many_sequences": lambda: W.make(40, 1, 8, 1, 128, 16, list(range(100, 40 * 997, 997)), dtype="bf16",
                                     device="cuda", seed=8),
    # head_dim 256 (query rows re-read from shared memory, one query buffer) and 512 (two
    # warps per stage, one CTA per SM), over more units than CTAs
    "d256_many_units": lambda: W.make(12, 1, 16, 8, 256, 16, list(range(700, 12 * 1900, 1900)), dtype="f16",
                                      device="cuda", seed=9),
    "d256_page64_rows16": lambda: W.make(2, 2, 16, 2, 256, 64, [9000, 3100], dtype="bf16", causal=True,
                                         device="cuda", seed=10),
    "d512_many_units": lambda: W.make(10, 1, 16, 8, 512, 16, list(range(300, 10 * 2300, 2300)), dtype="bf16",
                                      device="cuda", seed=13),
    "d512_page32_causal": lambda: W.make(2, 3, 8, 2, 512, 32, [5000, 77], dtype="f16", causal=True,
                                         device="cuda", seed=14),
    # more units than CTAs at head_dim 256 and 512 (one query buffer, unit after unit)
    "ragged_d256_interleaved": lambda: W.ragged(256, device="cuda", layout="interleaved"),
    "ragged_d512_split2": lambda: W.ragged(512, device="cuda", layout="split2"),
}


@pytest.mark.parametrize("case", list(CASES))
def test_persistent_and_grid_kernels_agree_bitwise(case):
    w = CASES[case]()
    pd = fd.PagedDecode(w.seq_lens, w.q_len, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype,
                        w.causal, device="cuda", path=fd.FDEC_PATH_MMA)  # (a tiny decode would plan on SIMT)
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    assert w.q.data_ptr() % 16 == 0
    first = _run(pd, w, w.q, table, lens)
    qm = _misaligned_copy(w.q)
    grid = _run(pd, w, qm, table, lens)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0
    assert torch.equal(first[0], grid[0]) and torch.equal(first[1], grid[1]), "persistent != one CTA per item"
    # the persistent kernel again, several times: the counter must stay in step
    for _ in range(5):
        again = _run(pd, w, w.q, table, lens)
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
    torch.cuda.synchronize()
    assert pd.device_errors() == 0


@pytest.mark.parametrize("case", ["long_131072", "ragged_d192", "page1_f16", "many_sequences", "d256_many_units",
                                  "d512_many_units", "d512_page32_causal", "ragged_d256_interleaved",
                                  "ragged_d512_split2"])
def test_persistent_kernel_matches_the_oracle(case):
    w = CASES[case]()
    pd = fd.PagedDecode(w.seq_lens, w.q_len, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype,
                        w.causal, device="cuda")
    info = pd.info
    assert info["path"] == fd.FDEC_PATH_MMA
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    out, lse = _run(pd, w, w.q, table, lens)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0
    wc = w.to("cpu")
    rows = None
    if case.startswith("ragged"):  # a sample of output rows: two query heads of every sequence
        rows = [b * w.num_qo_heads + h for b in range(w.batch) for h in (0, w.num_qo_heads - 1)]
    ref_o, ref_l = oracle_run(wc, rows=rows)
    if rows is None:
        assert_parity(out.cpu(), lse.cpu(), ref_o, ref_l, case)
    else:
        idx = torch.as_tensor(np.asarray(rows, dtype=np.int64))
        assert_parity(out.reshape(-1, w.head_dim).cpu()[idx], lse.reshape(-1).cpu()[idx], ref_o, ref_l, case)


def test_run_time_lengths_below_capacity_and_empty_sequences():
    # capacities fix the units; shorter run-time lengths leave some units empty
    w = W.make(4, 1, 16, 2, 128, 16, [9000, 7000, 300, 5000], dtype="bf16", device="cuda", seed=12)
    pd = fd.PagedDecode(w.seq_lens, 1, 16, 16, 2, 128, "bf16", device="cuda")
    table = torch.as_tensor(w.page_table, device="cuda")
    wc = w.to("cpu")
    for run_lens in ([9000, 7000, 300, 5000], [4100, 0, 299, 64], [1, 6999, 0, 0]):
        lens = torch.as_tensor(np.asarray(run_lens, dtype=np.int32), device="cuda")
        out, lse = _run(pd, w, w.q, table, lens)
        grid = _run(pd, w, _misaligned_copy(w.q), table, lens)
        torch.cuda.synchronize()
        assert pd.device_errors() == 0
        assert torch.equal(out, grid[0]) and torch.equal(lse, grid[1])
        ref_o, ref_l = oracle_run(wc, seq_lens=np.asarray(run_lens, dtype=np.int32))
        assert_parity(out.cpu(), lse.cpu(), ref_o, ref_l, str(run_lens))


def test_many_more_units_than_ctas():
    # 1024 short sequences (GQA 8/2, page 16): about 7 units per resident CTA, all but the
    # first of each CTA handed out by the ticket counter; sampled rows against the oracle,
    # bitwise against one CTA per item
    n = 1024
    lens = np.random.default_rng(41).integers(1, 400, n).astype(np.int32).tolist()
    w = W.make(n, 1, 8, 2, 128, 16, lens, dtype="bf16", device="cuda", seed=41)
    pd = fd.PagedDecode(w.seq_lens, 1, 16, 8, 2, 128, "bf16", device="cuda")
    info = pd.info
    assert info["num_items"] * 2 > 4 * info["num_split_ctas"]
    table = torch.as_tensor(w.page_table, device="cuda")
    lens_d = torch.as_tensor(w.seq_lens, device="cuda")
    out, lse = _run(pd, w, w.q, table, lens_d)
    grid = _run(pd, w, _misaligned_copy(w.q), table, lens_d)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0
    assert torch.equal(out, grid[0]) and torch.equal(lse, grid[1])
    for _ in range(3):  # the counter stays in step
        again = _run(pd, w, w.q, table, lens_d)
        assert torch.equal(out, again[0]) and torch.equal(lse, again[1])
    rows = [b * 8 + h for b in range(0, n, 17) for h in (0, 7)]
    ref_o, ref_l = oracle_run(w.to("cpu"), rows=rows)
    idx = torch.as_tensor(np.asarray(rows, dtype=np.int64))
    assert_parity(out.reshape(-1, 128).cpu()[idx], lse.reshape(-1).cpu()[idx], ref_o, ref_l, "1024 sequences")
