"""Stream order around the decode kernel's programmatic dependent launch: inputs that
the kernel just before the call writes on the same stream (q, lengths, page table)
are the ones the call reads, and back-to-back calls into the same out / lse leave
the last call's result.  Each call is compared bitwise with the same call made after
a device synchronisation (a fixed plan is deterministic)."""
import numpy as np
import pytest
import torch

import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _cases():
    return {
        "long_context_page64": lambda: W.long_context(4224, device="cuda"),   # region-major stages
        "batched_gqa_page16": lambda: W.batched_gqa(device="cuda"),           # box-major stages
        # the tcgen05 kernel (32 rows per KV head) and the one-CTA-per-item kernel (E4M3 codes)
        "spec_decode_q8_tcgen05": lambda: W.make(2, 8, 32, 8, 128, 16, [3000, 1700], dtype="bf16", causal=True,
                                                 device="cuda", seed=31),
        "e4m3_page32": lambda: W.make(2, 1, 16, 2, 128, 32, [5000, 2222], dtype="bf16", kv_dtype="fp8",
                                      device="cuda", seed=32),
    }


@pytest.mark.parametrize("case", list(_cases()))
def test_inputs_written_just_before_the_call_are_read(case):
    w = _cases()[case]()
    opts = {"kv_dtype": w.kv_dtype} if w.kv_dtype else {}
    pd = fd.PagedDecode(w.seq_lens, w.q_len, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype,
                        w.causal, device="cuda", **opts)
    sc = {"k_scale": 0.5, "v_scale": 2.0} if w.kv_dtype == "fp8" else {}
    gen = torch.Generator(device="cuda").manual_seed(5)
    n = 12
    qs = [torch.randn(w.q.shape, generator=gen, device="cuda").to(w.q.dtype) for _ in range(n)]
    caps = np.asarray(w.seq_lens, dtype=np.int32)
    lens_k = [torch.as_tensor(np.maximum(caps - 3 * k, 0).astype(np.int32), device="cuda") for k in range(n)]
    table0 = torch.as_tensor(w.page_table, device="cuda")
    tables = [table0.clone() for _ in range(n)]
    for k in range(1, n, 3):  # some steps permute two pages of sequence 0 (K/V follow the table)
        t = tables[k]
        t[0, 0], t[0, 1] = table0[0, 1].item(), table0[0, 0].item()
    q = torch.empty_like(w.q)
    lens = torch.empty_like(lens_k[0])
    table = torch.empty_like(table0)
    out = torch.empty((w.batch, w.q_len, w.num_qo_heads, w.head_dim), device="cuda")
    lse = torch.empty((w.batch, w.q_len, w.num_qo_heads), device="cuda")

    refs = []
    for k in range(n):
        q.copy_(qs[k])
        lens.copy_(lens_k[k])
        table.copy_(tables[k])
        torch.cuda.synchronize()
        pd.run(q, w.k, w.v, table, lens, out, lse, scale=w.scale, **sc)
        torch.cuda.synchronize()
        refs.append((out.clone(), lse.clone()))

    # the same steps with no synchronisation: each copy kernel runs right before its call
    got = []
    for k in range(n):
        q.copy_(qs[k])
        lens.copy_(lens_k[k])
        table.copy_(tables[k])
        pd.run(q, w.k, w.v, table, lens, out, lse, scale=w.scale, **sc)
        got.append((out.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert pd.device_errors() == 0
    for k in range(n):
        assert torch.equal(got[k][0], refs[k][0]), (case, k)
        assert torch.equal(got[k][1], refs[k][1]), (case, k)

    # back-to-back calls into the same out / lse: the last one's result stays
    for k in range(n):
        q.copy_(qs[k])
        pd.run(q, w.k, w.v, table0, torch.as_tensor(caps, device="cuda"), out, lse, scale=w.scale, **sc)
    torch.cuda.synchronize()
    q.copy_(qs[n - 1])
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    pd.run(q, w.k, w.v, table0, torch.as_tensor(caps, device="cuda"), out2, lse2, scale=w.scale, **sc)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def _packed(tensors, device):
    """One uint8 buffer holding every tensor at a 16-byte-aligned offset, and a view of each."""
    offs, at = [], 0
    for t in tensors:
        offs.append(at)
        at = (at + t.numel() * t.element_size() + 15) // 16 * 16
    buf = torch.zeros(at, dtype=torch.uint8, device=device)
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(tensors, offs)]
    for v, t in zip(views, tensors):
        v.copy_(t)
    return buf, views


@pytest.mark.parametrize("case", ["long_context_page64", "spec_decode_q8_tcgen05"])
def test_inputs_and_outputs_packed_in_one_buffer(case):
    # q, the page table and the lengths as views of one device buffer (one host-to-device
    # copy per step), out and lse as views of another (one copy back): the same result,
    # bitwise, as separate tensors
    w = _cases()[case]()
    pd = fd.PagedDecode(w.seq_lens, w.q_len, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype,
                        w.causal, device="cuda")
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    out = torch.empty((w.batch, w.q_len, w.num_qo_heads, w.head_dim), device="cuda")
    lse = torch.empty((w.batch, w.q_len, w.num_qo_heads), device="cuda")
    pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale)
    _, (q_p, table_p, lens_p) = _packed([w.q, table, lens], "cuda")
    _, (out_p, lse_p) = _packed([torch.full_like(out, float("nan")), torch.full_like(lse, float("nan"))], "cuda")
    pd.run(q_p, w.k, w.v, table_p, lens_p, out_p, lse_p, scale=w.scale)
    torch.cuda.synchronize()
    assert pd.device_errors() == 0
    assert torch.equal(out_p, out) and torch.equal(lse_p, lse)
