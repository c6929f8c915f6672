"""Glue between the seeded workloads and the float64 oracle (test side only)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_split_kv_gather_gb300.workloads import Workload, q_token_stride, storage_view


def np_storage(t: torch.Tensor):
    """(numpy array over t's whole CPU storage, element offset): uint16 for 16-bit
    tensors, uint8 (E4M3 codes) for float8_e4m3fn, int8 (q8_0 codes) for int8."""
    flat, off, _ = storage_view(t)
    if t.dtype == torch.float8_e4m3fn:
        return flat.view(torch.uint8).numpy(), off
    if t.dtype == torch.int8:
        return flat.numpy(), off
    return flat.view(torch.int16).numpy().view(np.uint16), off


def oracle_pool(t: torch.Tensor) -> oracle.Pool:
    arr, off = np_storage(t)
    return oracle.Pool(arr, off, t.shape[0], t.stride(0), t.stride(1), t.stride(2))


def oracle_run(w: Workload, rows=None, n_threads: int = 0, seq_lens=None, k_scale=1.0, v_scale=1.0):
    """Oracle (out, lse) for a CPU workload."""
    assert w.q.device.type == "cpu"
    q_arr, q_off = np_storage(w.q)
    lens = w.seq_lens if seq_lens is None else seq_lens
    q8 = w.kv_dtype == "q8_0"
    return oracle.paged_attention(
        q_arr, q_off, q_token_stride(w.q), w.q.stride(2), oracle_pool(w.k), oracle_pool(w.v),
        w.page_table, lens, q_len=w.q_len, num_qo_heads=w.num_qo_heads,
        num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=w.page_size,
        is_bf16=(w.dtype == "bf16"), causal=w.causal, scale=w.scale, rows=rows,
        n_threads=n_threads, k_scale=k_scale, v_scale=v_scale,
        k_scales=oracle_pool(w.k_scales) if q8 else None, v_scales=oracle_pool(w.v_scales) if q8 else None)


def gather_tokens(w: Workload, pool: torch.Tensor, b: int, kvh: int, n: int) -> np.ndarray:
    """float64 rows pool[table[b][t//P], kvh, t%P, :] for t < n (test-side gather)."""
    t = np.arange(n)
    pages = torch.as_tensor(w.page_table[b, t // w.page_size].astype(np.int64))
    slots = torch.as_tensor((t % w.page_size).astype(np.int64))
    return pool[pages, kvh, slots].double().numpy()


def visible(w: Workload, b: int, i: int) -> int:
    L = int(w.seq_lens[b])
    if not w.causal:
        return L
    return max(0, min(L, L - w.q_len + i + 1))


def row_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of ||got - ref||_inf / ||ref||_inf (rows = leading dims, last = D)."""
    got = np.asarray(got, dtype=np.float64).reshape(-1, ref.shape[-1])
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-1])
    num = np.max(np.abs(got - ref), axis=1)
    den = np.max(np.abs(ref), axis=1)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(num / den)) if num.size else 0.0


def lse_abs_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(got - ref))
    return float(np.max(d)) if d.size else 0.0


# ---------------------------------------------------------------------------
# running the CUDA library on a workload (GPU tests only)
# ---------------------------------------------------------------------------

OUT_TOL = 2e-3   # max over rows of ||out - ref||_inf / ||ref||_inf
LSE_TOL = 1e-4   # max |lse - ref|


def gpu_run(w: Workload, capacities=None, seq_lens=None, stream=None, k_scale=None, v_scale=None, **plan_opts):
    """Plan, upload and run the library on a CUDA workload; returns (out, lse, PagedDecode).
    With k_scale / v_scale the scaled entry point runs."""
    import paged_split_kv_gather_gb300 as fd

    dev = w.q.device
    if w.kv_dtype:
        plan_opts.setdefault("kv_dtype", w.kv_dtype)
    caps = w.seq_lens if capacities is None else capacities
    pd = fd.PagedDecode(caps, w.q_len, w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype,
                        w.causal, device=dev, stream=stream, **plan_opts)
    out = torch.full((w.batch, w.q_len, w.num_qo_heads, w.head_dim), float("nan"), device=dev)
    lse = torch.full((w.batch, w.q_len, w.num_qo_heads), float("nan"), device=dev)
    table = torch.as_tensor(w.page_table, device=dev)
    lens = torch.as_tensor(w.seq_lens if seq_lens is None else seq_lens, dtype=torch.int32, device=dev)
    # every storage the workload holds (q and the K/V pools) must come back bit-identical
    before = [t.clone() for t in w.keep]
    if w.kv_dtype == "q8_0":
        pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale, stream=stream, k_scales=w.k_scales,
               v_scales=w.v_scales)
    else:
        pd.run(w.q, w.k, w.v, table, lens, out, lse, scale=w.scale, stream=stream, k_scale=k_scale,
               v_scale=v_scale)
    for a, b in zip(before, w.keep):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), "an input buffer changed"
    return out, lse, pd


def assert_parity(out, lse, ref_out, ref_lse, what=""):
    o = out.detach().cpu().double().numpy() if hasattr(out, "detach") else np.asarray(out)
    l = lse.detach().cpu().double().numpy() if hasattr(lse, "detach") else np.asarray(lse)
    e_out = row_rel_err(o, ref_out)
    e_lse = lse_abs_err(l, ref_lse)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, f"{what}: out rel {e_out:.3g}, lse abs {e_lse:.3g}"
    return e_out, e_lse
