"""Paged KV append (the write side of the cache): the oracle's scatter pinned on
CPU by a gather round trip, then the library's kernel against it on the GPU,
bit for bit, in every K/V layout, and append-then-decode parity."""
import numpy as np
import pytest
import torch

import oracle
import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import assert_parity, gather_tokens, oracle_run


def _new_tokens(w, lens, n_per_seq, seed):
    """n_per_seq new tokens for each sequence at positions lens[b] .. lens[b]+n-1."""
    g = torch.Generator().manual_seed(seed)
    n = n_per_seq * w.batch
    shape = (n, w.num_kv_heads, w.head_dim)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    k_new = torch.randn(shape, generator=g).to(dt)
    v_new = torch.randn(shape, generator=g).to(dt)
    bi = np.repeat(np.arange(w.batch, dtype=np.int32), n_per_seq)
    pos = np.concatenate([np.arange(lens[b], lens[b] + n_per_seq, dtype=np.int32) for b in range(w.batch)])
    perm = np.random.default_rng(seed).permutation(n)  # any token order
    return k_new[perm], v_new[perm], bi[perm], pos[perm]


def test_oracle_append_round_trips_through_the_page_table():
    w = W.make(3, 1, 8, 2, 64, 16, [100, 250, 37], dtype="bf16", seed=3, layout="interleaved")
    lens = [60, 200, 5]
    k_new, v_new, bi, pos = _new_tokens(w, lens, 30, seed=1)
    k_before, v_before = w.k.clone(), w.v.clone()
    flags = oracle.append_paged(k_new, v_new, bi, pos, w.k, w.v, w.page_table, w.page_size)
    assert flags == 0
    for i in range(len(bi)):
        b, t = int(bi[i]), int(pos[i])
        for h in range(w.num_kv_heads):
            got_k = gather_tokens(w, w.k, b, h, t + 1)[t]
            got_v = gather_tokens(w, w.v, b, h, t + 1)[t]
            assert np.array_equal(got_k, k_new[i, h].double().numpy())
            assert np.array_equal(got_v, v_new[i, h].double().numpy())
    # every other (page, head, slot) row is unchanged
    written = {(int(w.page_table[b, t // 16]), t % 16) for b, t in zip(bi, pos)}
    for page in range(w.k.shape[0]):
        for slot in range(16):
            if (page, slot) not in written:
                assert torch.equal(w.k[page, :, slot], k_before[page, :, slot])
                assert torch.equal(w.v[page, :, slot], v_before[page, :, slot])


def test_oracle_append_skips_and_flags_bad_tokens():
    w = W.make(2, 1, 4, 1, 64, 16, [40, 40], dtype="f16", seed=5)
    k_new = torch.ones(3, 1, 64, dtype=torch.float16)
    v_new = torch.ones(3, 1, 64, dtype=torch.float16)
    before = w.k.clone()
    table = w.page_table.copy()
    table[1, 0] = w.k.shape[0] + 3  # a page outside the pool
    flags = oracle.append_paged(k_new, v_new, [0, 1, 2], [10_000, 3, 0], w.k, w.v, table, 16)
    assert flags == 3 and torch.equal(w.k, before)


@pytest.mark.gpu
@pytest.mark.parametrize("layout", ["hnd", "nhd", "interleaved", "split2"])
@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_append_matches_the_oracle_scatter_bit_for_bit(layout, page_size):
    caps = [300, 1000, 64]
    w = W.make(3, 1, 16, 4, 128, page_size, caps, dtype="bf16", device="cuda", seed=page_size, layout=layout)
    lens = [250, 900, 10]
    k_new, v_new, bi, pos = _new_tokens(w, lens, 40 if page_size > 1 else 7, seed=page_size)
    cpu = w.to("cpu")
    flags = oracle.append_paged(k_new, v_new, bi, pos, cpu.k, cpu.v, cpu.page_table, page_size)
    assert flags == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    table = torch.as_tensor(w.page_table, device="cuda")
    fd.fdec_append(k_new.cuda(), v_new.cuda(), torch.as_tensor(bi, device="cuda"), torch.as_tensor(pos, device="cuda"),
                   w.k, w.v, table, page_size, device_errors=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert len(w.keep) == len(cpu.keep)
    for got, ref in zip(w.keep, cpu.keep):  # q and every pool storage (whole, flattened), bit for bit
        assert torch.equal(got.reshape(-1).cpu().view(torch.int16), ref.reshape(-1).view(torch.int16))


@pytest.mark.gpu
def test_append_then_decode_matches_the_oracle():
    caps = [700, 2100, 129]
    w = W.make(3, 1, 32, 8, 128, 16, caps, dtype="bf16", device="cuda", seed=7, peaked=True)
    lens = [600, 2000, 100]
    k_new, v_new, bi, pos = _new_tokens(w, lens, 29, seed=7)
    table = torch.as_tensor(w.page_table, device="cuda")
    fd.fdec_append(k_new.cuda(), v_new.cuda(), torch.as_tensor(bi, device="cuda"), torch.as_tensor(pos, device="cuda"),
                   w.k, w.v, table, 16)
    new_lens = np.array(lens, dtype=np.int32) + 29
    pd = fd.PagedDecode(caps, 1, 16, 32, 8, 128, "bf16", device="cuda")
    out = torch.empty(3, 1, 32, 128, device="cuda")
    lse = torch.empty(3, 1, 32, device="cuda")
    pd.run(w.q, w.k, w.v, table, torch.as_tensor(new_lens, device="cuda"), out, lse, scale=w.scale)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0
    ro, rl = oracle_run(w.to("cpu"), seq_lens=new_lens)
    assert_parity(out.cpu(), lse.cpu(), ro, rl, "append then decode")


@pytest.mark.gpu
def test_append_flags_out_of_range_tokens_and_writes_nothing_for_them():
    w = W.make(2, 1, 4, 1, 64, 16, [40, 40], dtype="f16", device="cuda", seed=5)
    table = w.page_table.copy()
    table[1, 0] = w.k.shape[0] + 3
    before = [t.clone() for t in w.keep]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ones = torch.ones(3, 1, 64, dtype=torch.float16, device="cuda")
    fd.fdec_append(ones, ones, torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda"),
                   torch.tensor([10_000, 3, 0], dtype=torch.int32, device="cuda"), w.k, w.v,
                   torch.as_tensor(table, device="cuda"), 16, device_errors=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 3
    for a, b in zip(before, w.keep):
        assert torch.equal(a, b)


def test_append_rejects_bad_arguments_on_the_host():
    lib = fd._load()
    kd = fd.KVDesc(0x100000, 4, 4 * 16 * 64, 16 * 64, 64)
    p = 0x200000
    assert fd.STATUS_NAMES[lib.fdec_append(p, p, 64, 64, p, p, 1, 1, 100, 16, kd, kd, p, 1, 4, None, None)] == \
        "FDEC_ERR_UNSUPPORTED"
    assert fd.STATUS_NAMES[lib.fdec_append(p, p, 64, 64, p, p, 1, 1, 64, 12, kd, kd, p, 1, 4, None, None)] == \
        "FDEC_ERR_UNSUPPORTED"
    assert fd.STATUS_NAMES[lib.fdec_append(p + 2, p, 64, 64, p, p, 1, 1, 64, 16, kd, kd, p, 1, 4, None, None)] == \
        "FDEC_ERR_LAYOUT"
    assert fd.STATUS_NAMES[lib.fdec_append(None, p, 64, 64, p, p, 1, 1, 64, 16, kd, kd, p, 1, 4, None, None)] == \
        "FDEC_ERR_INVALID_ARG"
    assert fd.STATUS_NAMES[lib.fdec_append(p, p, 64, 64, p, p, 0, 1, 64, 16, kd, kd, p, 1, 4, None, None)] == "FDEC_OK"


@pytest.mark.gpu
@pytest.mark.parametrize("layout,page_size", [("hnd", 16), ("interleaved", 64), ("nhd", 1)])
def test_e4m3_append_matches_the_oracle_scatter_bit_for_bit(layout, page_size):
    caps = [300, 1000, 64]
    w = W.make(3, 1, 16, 4, 128, page_size, caps, dtype="bf16", kv_dtype="fp8", device="cuda", seed=page_size,
               layout=layout)
    lens = [250, 900, 10]
    k16, v16, bi, pos = _new_tokens(w, lens, 40 if page_size > 1 else 7, seed=page_size + 1)
    k_new, v_new = k16.float().to(torch.float8_e4m3fn), v16.float().to(torch.float8_e4m3fn)
    cpu = w.to("cpu")
    assert oracle.append_paged(k_new, v_new, bi, pos, cpu.k, cpu.v, cpu.page_table, page_size) == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fd.fdec_append_e4m3(k_new.cuda(), v_new.cuda(), torch.as_tensor(bi, device="cuda"),
                        torch.as_tensor(pos, device="cuda"), w.k, w.v, torch.as_tensor(w.page_table, device="cuda"),
                        page_size, device_errors=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for got, ref in zip(w.keep, cpu.keep):
        assert torch.equal(got.reshape(-1).cpu().view(torch.uint8), ref.reshape(-1).view(torch.uint8))


@pytest.mark.gpu
def test_e4m3_append_then_decode_matches_the_oracle():
    caps = [700, 2100, 129]
    w = W.make(3, 1, 32, 8, 128, 16, caps, dtype="bf16", kv_dtype="fp8", device="cuda", seed=9, peaked=True)
    lens = [600, 2000, 100]
    k16, v16, bi, pos = _new_tokens(w, lens, 29, seed=9)
    k_new, v_new = k16.float().to(torch.float8_e4m3fn), v16.float().to(torch.float8_e4m3fn)
    table = torch.as_tensor(w.page_table, device="cuda")
    fd.fdec_append_e4m3(k_new.cuda(), v_new.cuda(), torch.as_tensor(bi, device="cuda"),
                        torch.as_tensor(pos, device="cuda"), w.k, w.v, table, 16)
    new_lens = np.array(lens, dtype=np.int32) + 29
    pd = fd.PagedDecode(caps, 1, 16, 32, 8, 128, "bf16", device="cuda", kv_dtype="fp8")
    out = torch.empty(3, 1, 32, 128, device="cuda")
    lse = torch.empty(3, 1, 32, device="cuda")
    pd.run(w.q, w.k, w.v, table, torch.as_tensor(new_lens, device="cuda"), out, lse, scale=w.scale,
           k_scale=0.7, v_scale=1.3)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0
    ro, rl = oracle_run(w.to("cpu"), seq_lens=new_lens, k_scale=0.7, v_scale=1.3)
    assert_parity(out.cpu(), lse.cpu(), ro, rl, "e4m3 append then decode")


def test_e4m3_append_checks_byte_strides_and_element_sizes():
    lib = fd._load()
    p = 0x200000
    good = fd.KVDesc(0x100000, 4, 4 * 16 * 128, 16 * 128, 128)
    # 8-element strides are 16 bytes of a 16-bit cache but 8 bytes of codes
    assert fd.STATUS_NAMES[lib.fdec_append_e4m3(p, p, 128, 8, p, p, 1, 1, 128, 16, good, good, p, 1, 4, None,
                                                None)] == "FDEC_ERR_LAYOUT"
    bad = fd.KVDesc(0x100000, 4, 4 * 16 * 128, 16 * 128, 136)
    assert fd.STATUS_NAMES[lib.fdec_append_e4m3(p, p, 128, 128, p, p, 1, 1, 128, 16, good, bad, p, 1, 4, None,
                                                None)] == "FDEC_ERR_LAYOUT"
    odd16 = fd.KVDesc(0x100000, 4, 4 * 16 * 128, 16 * 128, 132)  # 132 x 2 bytes is not a multiple of 16
    assert fd.STATUS_NAMES[lib.fdec_append(p, p, 128, 8, p, p, 1, 1, 128, 16, good, odd16, p, 1, 4, None,
                                           None)] == "FDEC_ERR_LAYOUT"
    k16 = torch.zeros(2, 1, 128, dtype=torch.bfloat16)
    pool8 = torch.zeros(4, 1, 16, 128, dtype=torch.float8_e4m3fn)
    idx = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError):
        fd.fdec_append_e4m3(k16, k16, idx, idx, pool8, pool8, torch.zeros(1, 4, dtype=torch.int32), 16)
    with pytest.raises(ValueError):
        fd.fdec_append(k16, k16, idx, idx, pool8, pool8, torch.zeros(1, 4, dtype=torch.int32), 16)
