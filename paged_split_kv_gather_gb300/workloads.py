"""Seeded synthetic inputs for paged-KV attention decode.

This module only draws and lays out inputs: random q/K/V values, sequence
lengths, page tables and the physical arrangement of the K/V pools.  It holds
none of the attention arithmetic, so the float64 oracle and the CUDA library
can both be fed from it.

Recipe (all draws seeded):
  * integer structure (lengths, page permutations, spike positions) from
    ``numpy.random.Generator(PCG64(seed))``, in the order: lengths, page
    permutation, spike positions;
  * q, then K, then V from one ``torch.Generator(device).manual_seed(seed)``,
    standard normal in float32, then rounded to the storage dtype;
  * "spikes" (long-context sweep): for 1% of the token positions (without
    replacement) and every KV head, K_t += alpha * qbar where qbar is the mean
    of that head's query group and alpha = 8 / (scale * |qbar|^2), which lifts
    that token's logit by about +8 for every head of the group; the sum is
    rounded to the storage dtype, and both sides read the stored values;
  * "peaked": q multiplied by 8 (exact in 16-bit), so the softmax is sharp and
    a misread key or value moves the output well past the tolerance;
  * quantised caches (kv_dtype "fp8"): K and V drawn the same way and rounded
    to 8-bit E4M3 (torch.float8_e4m3fn), q stays 16-bit;
  * q8_0 caches (kv_dtype "q8_0"): K codes, V codes (uniform int8 in
    [-128, 127]), then K and V block scales (log-uniform in [0.005, 0.05],
    stored as binary16: the size of max|x| / 127 for unit-variance values), each
    pool in the same layout as the codes with head_dim / 32 scales per row.  No
    quantisation is done: codes and scales are drawn as they are stored.

The five named workloads follow the shapes of the pages' workloads: a tiny
decode, a batched GQA decode at exactly 32 blocks of 64 tokens, the 32q/4kv/128
long-context sweep across the 2048-token boundary up to 262144 tokens, a ragged
serving batch with large head dims over an interleaved cache, and multi-token
(spec-decode / prefill-chunk) queries with a causal mask.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

LONG_CONTEXT_LENGTHS = (1900, 2000, 2100, 3000, 4800, 32768, 131072, 262144)
RAGGED_HEAD_DIMS = (192, 256, 512)
MULTI_TOKEN_Q_LENS = (4, 8, 2048)

_TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "fp8": torch.float8_e4m3fn, "q8_0": torch.int8,
                "q8_0_scale": torch.float16}
_NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "fp8": 0x7F}


@dataclass
class Workload:
    """One set of inputs.  K and V are 4-D views indexed [page, kv_head, slot, dim]."""

    name: str
    dtype: str
    batch: int
    q_len: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    causal: bool
    scale: float
    seq_lens: np.ndarray          # int32 [batch]
    page_table: np.ndarray        # int32 [batch, max_pages]; unused entries are -1
    q: torch.Tensor               # [batch, q_len, Hq, D] (any token/head strides, dim stride 1)
    k: torch.Tensor               # [pages, Hk, P, D] view
    v: torch.Tensor               # [pages, Hk, P, D] view
    layout: str = "hnd"
    keep: List[torch.Tensor] = field(default_factory=list)
    kv_dtype: str = ""            # "" = the q dtype; "fp8" = E4M3 K/V codes; "q8_0" = int8 codes + block scales
    k_scales: Optional[torch.Tensor] = None  # q8_0: binary16 [pages, Hk, P, D / 32] views
    v_scales: Optional[torch.Tensor] = None

    @property
    def kv_fp8(self) -> bool:
        return self.kv_dtype == "fp8"

    @property
    def group(self) -> int:
        return self.num_qo_heads // self.num_kv_heads

    @property
    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one call reads: sum_b L_b * Hk * 2 (K and V) * (D * element bytes, plus
        D / 32 binary16 block scales for q8_0)."""
        row = self.head_dim * (1 if self.kv_dtype in ("fp8", "q8_0") else 2)
        if self.kv_dtype == "q8_0":
            row += (self.head_dim // 32) * 2
        return int(np.sum(self.seq_lens.astype(np.int64))) * self.num_kv_heads * 2 * row

    def to(self, device) -> "Workload":
        """Copy every tensor to ``device`` keeping views and strides (storage is copied whole)."""
        memo = {}

        def move(t):
            base = _flat_storage(t)
            key = base.data_ptr()
            if key not in memo:
                memo[key] = base.to(device)
            nb = memo[key]
            return nb.as_strided(t.shape, t.stride(), t.storage_offset())

        ks = None if self.k_scales is None else move(self.k_scales)
        vs = None if self.v_scales is None else move(self.v_scales)
        return Workload(self.name, self.dtype, self.batch, self.q_len, self.num_qo_heads,
                        self.num_kv_heads, self.head_dim, self.page_size, self.causal, self.scale,
                        self.seq_lens.copy(), self.page_table.copy(), move(self.q), move(self.k),
                        move(self.v), self.layout, list(memo.values()), self.kv_dtype, ks, vs)


def _flat_storage(t: torch.Tensor) -> torch.Tensor:
    """A 1-D tensor of t's dtype over t's whole storage (offset 0)."""
    n = t.untyped_storage().nbytes() // t.element_size()
    return torch.empty(0, dtype=t.dtype, device=t.device).set_(t.untyped_storage(), 0, (n,), (1,))


def q_token_stride(q: torch.Tensor) -> int:
    """Element stride between consecutive flattened tokens b*Q + i of a [B, Q, Hq, D] view."""
    batch, q_len = q.shape[0], q.shape[1]
    if q_len == 1:
        return q.stride(0)
    if batch > 1 and q.stride(0) != q_len * q.stride(1):
        raise ValueError("q tokens do not flatten to a single stride (b*Q + i)")
    return q.stride(1)


def storage_view(t: torch.Tensor):
    """(flat storage tensor, element offset, strides) of a view."""
    return _flat_storage(t), t.storage_offset(), t.stride()


def _randn(gen: torch.Generator, shape, device, dtype: str) -> torch.Tensor:
    if dtype == "q8_0":          # codes, uniform over the signed bytes
        return torch.randint(-128, 128, shape, generator=gen, device=device, dtype=torch.int8)
    if dtype == "q8_0_scale":    # block scales, log-uniform in [0.005, 0.05]
        u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
        return torch.exp(math.log(0.005) + u * (math.log(0.05) - math.log(0.005))).to(torch.float16)
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return x.to(_TORCH_DTYPE[dtype])


def _alloc_pool(num_pages: int, hk: int, p: int, d: int, layout: str, gen, device, dtype):
    """Draw K then V and arrange them as ``layout``; returns (k_view, v_view, keep)."""
    shape_hnd = (num_pages, hk, p, d)
    if layout == "hnd":          # separate pools [pages, Hk, P, D]
        k = _randn(gen, shape_hnd, device, dtype)
        v = _randn(gen, shape_hnd, device, dtype)
        return k, v, [k, v]
    if layout == "nhd":          # separate pools [pages, P, Hk, D]
        k = _randn(gen, (num_pages, p, hk, d), device, dtype)
        v = _randn(gen, (num_pages, p, hk, d), device, dtype)
        return k.permute(0, 2, 1, 3), v.permute(0, 2, 1, 3), [k, v]
    if layout == "mixed":        # K as NHD [pages, P, Hk, D], V as HND [pages, Hk, P, D]
        k = _randn(gen, (num_pages, p, hk, d), device, dtype)
        v = _randn(gen, shape_hnd, device, dtype)
        return k.permute(0, 2, 1, 3), v, [k, v]
    if layout == "interleaved":  # one tensor [pages, 2, Hk, P, D]
        kv = torch.empty((num_pages, 2, hk, p, d), device=device, dtype=_TORCH_DTYPE[dtype])
        kv[:, 0] = _randn(gen, shape_hnd, device, dtype)
        kv[:, 1] = _randn(gen, shape_hnd, device, dtype)
        return kv[:, 0], kv[:, 1], [kv]
    if layout == "split2":       # one tensor [2, pages, Hk, P, D]
        kv = torch.empty((2, num_pages, hk, p, d), device=device, dtype=_TORCH_DTYPE[dtype])
        kv[0] = _randn(gen, shape_hnd, device, dtype)
        kv[1] = _randn(gen, shape_hnd, device, dtype)
        return kv[0], kv[1], [kv]
    if layout == "interleaved_nhd":  # one tensor [pages, P, 2, Hk, D] (token-major pairs)
        kv = torch.empty((num_pages, p, 2, hk, d), device=device, dtype=_TORCH_DTYPE[dtype])
        kv[:, :, 0] = _randn(gen, (num_pages, p, hk, d), device, dtype)
        kv[:, :, 1] = _randn(gen, (num_pages, p, hk, d), device, dtype)
        return kv[:, :, 0].permute(0, 2, 1, 3), kv[:, :, 1].permute(0, 2, 1, 3), [kv]
    raise ValueError(f"unknown layout {layout!r}")


def _page_tables(rng: np.random.Generator, lens, page_size: int, pool_pages: Optional[int]):
    """Give each sequence ceil(L/P) distinct physical pages drawn from a shuffled pool."""
    need = [max(1, -(-int(L) // page_size)) for L in lens]
    total = sum(need)
    pool = total if pool_pages is None else int(pool_pages)
    if pool < total:
        raise ValueError("pool too small")
    perm = rng.permutation(pool)[:total]
    width = max(need)
    table = np.full((len(lens), width), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n]
        at += n
    return table, pool


def make(batch: int, q_len: int, num_qo_heads: int, num_kv_heads: int, head_dim: int,
         page_size: int, seq_lens, *, dtype: str = "bf16", layout: str = "hnd",
         causal: bool = False, seed: int = 0, device="cpu", pool_pages: Optional[int] = None,
         q_layout: str = "packed", peaked: bool = False, spikes: float = 0.0,
         nan_guard: bool = False, name: str = "custom", scale: Optional[float] = None,
         kv_dtype: str = "") -> Workload:
    """General seeded workload.

    q_layout: "packed" [B,Q,Hq,D]; "fused_qkv" (head slice of a [B*Q, Hq+2Hk, D] tensor);
    "head_major" (a [Hq, B*Q, D] tensor viewed as [B,Q,Hq,D]).
    nan_guard: fill every K/V element that must never be read (slots past L in a
    sequence's last page, and pages no sequence references) with NaN.
    kv_dtype: "" (K/V in the q dtype), "fp8" (E4M3 K/V codes) or "q8_0" (int8 codes and
    binary16 block-scale pools in the same layout).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = np.asarray(seq_lens, dtype=np.int64).reshape(-1)
    if lens.shape[0] != batch:
        raise ValueError("seq_lens must have batch entries")
    table, pool = _page_tables(rng, lens, page_size, pool_pages)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    tdt = _TORCH_DTYPE[dtype]
    hq, hk, d = num_qo_heads, num_kv_heads, head_dim
    sc = 1.0 / math.sqrt(head_dim) if scale is None else float(scale)

    ntok = batch * q_len
    if q_layout == "packed":
        q = _randn(gen, (batch, q_len, hq, d), device, dtype)
        q_keep = [q]
    elif q_layout == "fused_qkv":
        fused = torch.zeros((ntok, hq + 2 * hk, d), device=device, dtype=tdt)
        fused[:, :hq] = _randn(gen, (ntok, hq, d), device, dtype)
        q = fused[:, :hq].view(batch, q_len, hq, d)
        q_keep = [fused]
    elif q_layout == "head_major":
        hm = _randn(gen, (hq, ntok, d), device, dtype)
        q = hm.permute(1, 0, 2).view(batch, q_len, hq, d)
        q_keep = [hm]
    else:
        raise ValueError(f"unknown q_layout {q_layout!r}")
    if peaked:
        q.mul_(8)

    kvd = kv_dtype or dtype
    k, v, keep = _alloc_pool(pool, hk, page_size, d, layout, gen, device, kvd)
    ks = vs = None
    if kvd == "q8_0":
        if d % 32 != 0:
            raise ValueError("q8_0 rows are blocks of 32")
        if spikes > 0:
            raise ValueError("spikes are drawn into 16-bit or E4M3 keys only")
        ks, vs, skeep = _alloc_pool(pool, hk, page_size, d // 32, layout, gen, device, "q8_0_scale")
        keep = keep + skeep

    if spikes > 0:
        _add_spikes(rng, k, q, table, lens, page_size, sc, spikes, hq // hk)
    if nan_guard:
        if kvd == "q8_0":  # int8 codes have no NaN: the scales of unread rows carry it
            _nan_fill_unread(ks, vs, table, lens, page_size, "f16")
        else:
            _nan_fill_unread(k, v, table, lens, page_size, kvd)

    return Workload(name, dtype, batch, q_len, hq, hk, d, page_size, causal, sc,
                    lens.astype(np.int32), table, q, k, v, layout, q_keep + keep, kv_dtype, ks, vs)


def _add_spikes(rng, k, q, table, lens, page_size, scale, frac, g):
    batch, _, hq, d = q.shape
    hk = k.shape[1]
    for b in range(batch):
        L = int(lens[b])
        n_sp = int(math.ceil(frac * L))
        if n_sp == 0:
            continue
        pos = rng.choice(L, size=n_sp, replace=False)
        pages = torch.as_tensor(table[b, pos // page_size].astype(np.int64), device=k.device)
        slots = torch.as_tensor((pos % page_size).astype(np.int64), device=k.device)
        for kvh in range(hk):
            qbar = q[b, :, kvh * g:(kvh + 1) * g].float().mean(dim=(0, 1))
            alpha = 8.0 / (scale * float(qbar.pow(2).sum()))
            rows = (k[pages, kvh, slots].float() + alpha * qbar).to(k.dtype)
            if k.element_size() == 1:  # write E4M3 codes through a byte view
                k.view(torch.uint8)[pages, kvh, slots] = rows.view(torch.uint8)
            else:
                k[pages, kvh, slots] = rows


def _nan_fill_unread(k, v, table, lens, page_size, dtype):
    raw_dtype = torch.uint8 if dtype == "fp8" else torch.int16
    nan = torch.tensor(_NAN_BITS[dtype], dtype=torch.int32).to(raw_dtype).item()
    used = np.zeros(k.shape[0], dtype=bool)
    for b in range(table.shape[0]):
        n = max(1, -(-int(lens[b]) // page_size))
        used[table[b, :n]] = True
    for pool in (k, v):
        raw = pool.view(raw_dtype)
        unused = torch.as_tensor(np.nonzero(~used)[0], device=pool.device)
        if unused.numel():
            raw[unused] = nan
        for b in range(table.shape[0]):
            L = int(lens[b])
            n = max(1, -(-L // page_size))
            tail = L - (n - 1) * page_size
            if tail < page_size:
                raw[int(table[b, n - 1]), :, tail:] = nan


# ----------------------------------------------------------------------------
# The named workloads
# ----------------------------------------------------------------------------

def tiny(seed: int = 0, device="cpu", **kw) -> Workload:
    """Batch 1, q_len 1, 4 q heads / 1 KV head, D 64, L 300, page 16, f16, NHD pools of 19 pages."""
    kw.setdefault("layout", "nhd")
    return make(1, 1, 4, 1, 64, 16, [300], dtype="f16", seed=seed, device=device,
                pool_pages=19, name="tiny_decode", **kw)


def batched_gqa(seed: int = 0, device="cpu", **kw) -> Workload:
    """Batch 8, 32/8 heads, D 128, every L = 2048 (32 blocks of 64), page 16, bf16,
    separate K/V pools of 2048 pages of which 1024 are used."""
    return make(8, 1, 32, 8, 128, 16, [2048] * 8, dtype="bf16", seed=seed, device=device,
                pool_pages=2048, name="batched_gqa_decode", **kw)


def long_context(length: int, seed: int = 0, device="cpu", **kw) -> Workload:
    """Batch 1, 32/4 heads, D 128, page 64, bf16, shuffled pages, 1% of tokens spiked by ~+8 logit."""
    kw.setdefault("spikes", 0.01)
    return make(1, 1, 32, 4, 128, 64, [length], dtype="bf16", seed=seed, device=device,
                name=f"long_context_decode_L{length}", **kw)


def ragged_lengths(seed: int = 0, batch: int = 64, lo: int = 16, hi: int = 32768) -> np.ndarray:
    """L_b = round(exp(U(ln lo, ln hi))), drawn from its own stream."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    return np.round(np.exp(rng.uniform(math.log(lo), math.log(hi), size=batch))).astype(np.int32)


def ragged(head_dim: int, seed: int = 0, device="cpu", layout: str = "interleaved", **kw) -> Workload:
    """64 sequences, log-uniform L in [16, 32768], 16/8 heads, page 16, f16, one
    [pages,2,Hk,16,D] tensor ("interleaved") or [2,pages,...] views ("split2")."""
    lens = ragged_lengths(seed)
    return make(64, 1, 16, 8, head_dim, 16, lens, dtype="f16", seed=seed, device=device,
                layout=layout, name=f"ragged_serving_D{head_dim}_{layout}", **kw)


def multi_token(q_len: int, seed: int = 0, device="cpu", **kw) -> Workload:
    """Batch 4, 32/8 heads, D 128, bf16, page 16, KV length 8192 + q_len, causal (bottom-right)."""
    return make(4, q_len, 32, 8, 128, 16, [8192 + q_len] * 4, dtype="bf16", seed=seed,
                device=device, causal=True, name=f"multi_token_Q{q_len}", **kw)
