"""Cascade (shared-prefix) decode composed from the library's calls: the shared
prefix is attended once for all sequences that share it (their queries are the
query rows of one non-causal call over the prefix pages), each sequence's own
suffix by an ordinary decode call, and the two normalised states of every row
are merged by fdec_merge_states.  The FlashInfer PR "Stop declaring the paged KV
cache mutated on read-only attention ops" runs its cascade tests against the
decode path; here the composition is checked against the oracle over each whole
sequence (prefix pages followed by the sequence's own pages)."""
import dataclasses

import numpy as np
import pytest
import torch

import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import assert_parity, oracle_run


def _cascade_case(hq, hk, d, prefix_len, suffix_lens, dtype, seed):
    """One pool holding the prefix (sequence 0 of the table) and every suffix."""
    P = 16
    assert prefix_len % P == 0
    s = len(suffix_lens)
    w = W.make(s + 1, 1, hq, hk, d, P, [prefix_len, *suffix_lens], dtype=dtype, device="cuda", seed=seed,
               peaked=True)
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    q = (torch.randn((s, 1, hq, d), generator=g, device="cuda") * 8).to(tdt)  # one query per sequence
    return w, q


def _full_sequence_oracle(w, q, prefix_len, suffix_lens):
    """Oracle over each whole sequence: table row = prefix pages + own pages."""
    P = w.page_size
    s = len(suffix_lens)
    npre = prefix_len // P
    width = npre + max(1, -(-max(suffix_lens) // P))
    table = np.full((s, width), -1, dtype=np.int32)
    for b, L in enumerate(suffix_lens):
        table[b, :npre] = w.page_table[0, :npre]
        own = -(-L // P)
        table[b, npre:npre + own] = w.page_table[1 + b, :own]
    cpu = w.to("cpu")
    full = dataclasses.replace(cpu, batch=s, q_len=1, q=q.cpu(), page_table=table,
                               seq_lens=np.array([prefix_len + L for L in suffix_lens], dtype=np.int32))
    return oracle_run(full)


def _cascade(w, q, prefix_len, suffix_lens):
    s = len(suffix_lens)
    hq, d = w.num_qo_heads, w.head_dim
    table = torch.as_tensor(w.page_table, device="cuda")
    o_states = torch.empty((2, s * hq, d), device="cuda")
    lse_states = torch.empty((2, s * hq), device="cuda")
    # shared prefix: one sequence whose s query tokens are the s sequences' queries
    pre = fd.PagedDecode([prefix_len], s, w.page_size, hq, w.num_kv_heads, d, w.dtype, causal=False,
                         device="cuda")
    pre.run(q.view(1, s, hq, d), w.k, w.v, table[0:1], torch.tensor([prefix_len], dtype=torch.int32,
                                                                     device="cuda"),
            o_states[0].view(1, s, hq, d), lse_states[0].view(1, s, hq), scale=w.scale)
    # each sequence's own suffix
    suf = fd.PagedDecode(suffix_lens, 1, w.page_size, hq, w.num_kv_heads, d, w.dtype, device="cuda")
    suf.run(q, w.k, w.v, table[1:], torch.as_tensor(np.asarray(suffix_lens, dtype=np.int32), device="cuda"),
            o_states[1].view(s, 1, hq, d), lse_states[1].view(s, 1, hq), scale=w.scale)
    out = torch.empty((s * hq, d), device="cuda")
    lse = torch.empty((s * hq,), device="cuda")
    fd.fdec_merge_states(o_states, lse_states, out, lse)
    torch.cuda.synchronize()
    assert pre.device_errors() == 0 and suf.device_errors() == 0
    return out.view(s, 1, hq, d), lse.view(s, 1, hq), pre.info


@pytest.mark.gpu
@pytest.mark.parametrize("hq,hk,d,dtype,suffix_lens,want_path", [
    (32, 8, 128, "bf16", [1, 37, 0, 500, 64, 129, 2000, 15], fd.FDEC_PATH_TC),   # 32 prefix rows: tcgen05
    (8, 2, 64, "f16", [300, 0, 17], fd.FDEC_PATH_MMA),                            # 12 prefix rows: mma.sync
    (16, 8, 256, "bf16", [65, 1000], fd.FDEC_PATH_MMA),
])
def test_cascade_matches_the_oracle_on_whole_sequences(hq, hk, d, dtype, suffix_lens, want_path):
    prefix_len = 3008
    w, q = _cascade_case(hq, hk, d, prefix_len, suffix_lens, dtype, seed=d)
    out, lse, info = _cascade(w, q, prefix_len, suffix_lens)
    assert int(info["path"]) == want_path
    ro, rl = _full_sequence_oracle(w, q, prefix_len, suffix_lens)
    assert_parity(out.cpu(), lse.cpu(), ro, rl, "cascade")


def test_cascade_reading_holds_in_the_oracle():
    """CPU pin of the cascade reading, oracle only: the prefix attended as the
    non-causal query rows of one call, merged by log-sum-exp with each sequence's
    own-suffix attention, equals attention over prefix + suffix (to 1e-12)."""
    import oracle

    prefix_len, suffix_lens = 192, [5, 0, 70]
    hq, hk, d, P = 8, 2, 64, 16
    s = len(suffix_lens)
    w = W.make(s + 1, 1, hq, hk, d, P, [prefix_len, *suffix_lens], dtype="bf16", seed=3, peaked=True)
    q = (torch.randn((s, 1, hq, d), generator=torch.Generator().manual_seed(4)) * 8).to(torch.bfloat16)
    pre = dataclasses.replace(w, batch=1, q_len=s, q=q.view(1, s, hq, d), causal=False,
                              page_table=w.page_table[0:1], seq_lens=np.array([prefix_len], dtype=np.int32))
    suf = dataclasses.replace(w, batch=s, q_len=1, q=q, page_table=w.page_table[1:],
                              seq_lens=np.array(suffix_lens, dtype=np.int32))
    po, pl = oracle_run(pre)
    so, sl = oracle_run(suf)
    mo, ml = oracle.merge_states(np.stack([po.reshape(s * hq, d), so.reshape(s * hq, d)]),
                                 np.stack([pl.reshape(-1), sl.reshape(-1)]))
    ro, rl = _full_sequence_oracle_cpu(w, q, prefix_len, suffix_lens)
    assert np.abs(mo - ro.reshape(s * hq, d)).max() < 1e-12
    assert np.abs(ml - rl.reshape(-1)).max() < 1e-12


def _full_sequence_oracle_cpu(w, q, prefix_len, suffix_lens):
    P = w.page_size
    s = len(suffix_lens)
    npre = prefix_len // P
    width = npre + max(1, -(-max(suffix_lens) // P))
    table = np.full((s, width), -1, dtype=np.int32)
    for b, L in enumerate(suffix_lens):
        table[b, :npre] = w.page_table[0, :npre]
        own = -(-L // P)
        table[b, npre:npre + own] = w.page_table[1 + b, :own]
    full = dataclasses.replace(w, batch=s, q_len=1, q=q, page_table=table,
                               seq_lens=np.array([prefix_len + L for L in suffix_lens], dtype=np.int32))
    return oracle_run(full)
