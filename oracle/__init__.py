"""float64 CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  The
product library never imports or links it, and it shares no code with the
CUDA path.

The arithmetic lives in ``oracle.c`` (plain C, OpenMP over output rows); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
What it computes is stated at the top of ``oracle.c``: softmax(q K^T * scale) V
and its log-sum-exp over the tokens gathered through the page table, and the
log-sum-exp merge of normalised attention states.  ``append_paged`` (the write
side of the cache, a plain scatter) is written here in Python.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    lib.oracle_f16_to_double.restype = ctypes.c_double
    lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_paged_attention.restype = I
    lib.oracle_paged_attention.argtypes = (
        [P, I64, I64, I64]
        + [P, I64, I64, I64, I64, I64]
        + [P, I64, I64, I64, I64, I64]
        + [P, I64, P]
        + [I, I, I, I, I, I, I, I, ctypes.c_double, I, ctypes.c_double, ctypes.c_double]
        + [P, I64, I64, I64, I64, P, I64, I64, I64, I64]
        + [P, I64, P, P, I]
    )
    lib.oracle_merge_states.restype = I
    lib.oracle_merge_states.argtypes = [P, P, I, I64, I, P, P]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB)
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Temporarily route every call through another build of oracle.c (used by the
    mutation tests, which plant a mistake in a copy of the source)."""
    global _lib
    _load()
    with _lock:
        saved = _lib
        _lib = _bind(path)
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"16-bit storage expected, got {a.dtype}")
    return a.reshape(-1)


def f16_to_double(bits: int) -> float:
    return _load().oracle_f16_to_double(int(bits) & 0xFFFF)


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits) & 0xFFFF)


def e4m3_to_double(bits: int) -> float:
    return _load().oracle_e4m3_to_double(int(bits) & 0xFF)


KV_16BIT, KV_E4M3, KV_Q8_0 = 0, 1, 2  # storage formats (oracle.c)


class Pool:
    """A K or V pool as flat storage plus element offset, page count and strides.

    Element (page, head, slot, dim) is at ``offset + page*stride_page +
    head*stride_head + slot*stride_token + dim``.  The storage is 16-bit (the
    query's type, or the binary16 scales of a q8_0 cache) or, for a quantised
    cache, uint8 holding E4M3 codes or int8 holding q8_0 codes.
    """

    def __init__(self, storage, offset: int, num_pages: int, stride_page: int,
                 stride_head: int, stride_token: int):
        a = np.asarray(storage)
        self.fp8 = a.dtype == np.uint8
        self.fmt = KV_E4M3 if self.fp8 else (KV_Q8_0 if a.dtype == np.int8 else KV_16BIT)
        self.storage = np.ascontiguousarray(a).reshape(-1) if self.fmt != KV_16BIT else _u16(storage)
        self.offset = int(offset)
        self.num_pages = int(num_pages)
        self.stride_page = int(stride_page)
        self.stride_head = int(stride_head)
        self.stride_token = int(stride_token)


def paged_attention(q_storage, q_offset: int, q_stride_tok: int, q_stride_head: int,
                    k: Pool, v: Pool, page_table, seq_lens, *, q_len: int, num_qo_heads: int,
                    num_kv_heads: int, head_dim: int, page_size: int, is_bf16: bool,
                    causal: bool, scale: float, rows=None, n_threads: int = 0, k_scale: float = 1.0,
                    v_scale: float = 1.0, k_scales: Pool | None = None, v_scales: Pool | None = None):
    """Return (out, lse) in float64.

    K and V are k_scale and v_scale times their stored values (decoded from
    16-bit, from E4M3 when the pools hold uint8 codes, or from q8_0 when they hold
    int8 codes: then k_scales / v_scales are the binary16 block-scale pools, scale
    j of (page, head, slot) at the pool's address of "dim" j).

    Without ``rows``: out has shape [batch, q_len, Hq, D] and lse [batch, q_len, Hq].
    With ``rows`` (flat indices (b*q_len + i)*Hq + h): out is [len(rows), D], lse [len(rows)].
    """
    lib = _load()
    if k.fmt != v.fmt:
        raise ValueError("K and V pools must have the same storage type")
    q8 = k.fmt == KV_Q8_0
    if q8 and (k_scales is None or v_scales is None):
        raise ValueError("q8_0 pools need k_scales and v_scales")
    ks = k_scales if q8 else None
    vs = v_scales if q8 else None
    qs = _u16(q_storage)
    table = np.ascontiguousarray(page_table, dtype=np.int32)
    if table.ndim != 2:
        raise ValueError("page_table must be 2-D [batch, max_pages]")
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32).reshape(-1)
    batch = lens.shape[0]
    if rows is None:
        n_rows = batch * q_len * num_qo_heads
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
        n_rows = rows_arr.shape[0]
    out = np.empty((n_rows, head_dim), dtype=np.float64)
    lse = np.empty((n_rows,), dtype=np.float64)
    st = lib.oracle_paged_attention(
        qs.ctypes.data, q_offset, q_stride_tok, q_stride_head,
        k.storage.ctypes.data, k.offset, k.num_pages, k.stride_page, k.stride_head, k.stride_token,
        v.storage.ctypes.data, v.offset, v.num_pages, v.stride_page, v.stride_head, v.stride_token,
        table.ctypes.data, table.shape[1], lens.ctypes.data,
        batch, q_len, num_qo_heads, num_kv_heads, head_dim, page_size, int(bool(is_bf16)),
        int(bool(causal)), float(scale), int(k.fmt), float(k_scale), float(v_scale),
        None if ks is None else ks.storage.ctypes.data, 0 if ks is None else ks.offset,
        0 if ks is None else ks.stride_page, 0 if ks is None else ks.stride_head, 0 if ks is None else ks.stride_token,
        None if vs is None else vs.storage.ctypes.data, 0 if vs is None else vs.offset,
        0 if vs is None else vs.stride_page, 0 if vs is None else vs.stride_head, 0 if vs is None else vs.stride_token,
        None if rows_arr is None else rows_arr.ctypes.data, n_rows,
        out.ctypes.data, lse.ctypes.data, int(n_threads))
    if st != 0:
        raise ValueError(f"oracle_paged_attention failed with status {st}")
    if rows is None:
        return (out.reshape(batch, q_len, num_qo_heads, head_dim),
                lse.reshape(batch, q_len, num_qo_heads))
    return out, lse


def merge_states(o, lse):
    """Merge normalised states: o [n, rows, D], lse [n, rows] -> (o [rows, D], lse [rows])."""
    lib = _load()
    o = np.ascontiguousarray(o, dtype=np.float64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    n, rows, d = o.shape
    if lse.shape != (n, rows):
        raise ValueError("lse must be [n_states, rows]")
    o_out = np.empty((rows, d), dtype=np.float64)
    lse_out = np.empty((rows,), dtype=np.float64)
    st = lib.oracle_merge_states(o.ctypes.data, lse.ctypes.data, n, rows, d,
                                 o_out.ctypes.data, lse_out.ctypes.data)
    if st != 0:
        raise ValueError(f"oracle_merge_states failed with status {st}")
    return o_out, lse_out


def append_paged(k_new, v_new, batch_indices, positions, k_view, v_view, page_table, page_size: int) -> int:
    """Paged KV append, by definition (FlashInfer PR "Stop declaring the paged KV
    cache mutated on read-only attention ops", append notes: append writes the
    cache): new token i of sequence b = batch_indices[i] at position
    t = positions[i] goes to page = page_table[b][t // page_size], slot
    t % page_size, for every KV head:  K[page, h, slot, :] = k_new[i, h, :] and
    V likewise.  A token whose sequence, position or page id is out of range is
    skipped; the returned flags are those of the library (1 = page id,
    2 = sequence / position).  Plain Python over the tokens on CPU tensors
    (k_view / v_view are written in place through their strides)."""
    table = np.asarray(page_table)
    flags = 0
    n_pages_k, n_pages_v = k_view.shape[0], v_view.shape[0]
    for i in range(k_new.shape[0]):
        b, t = int(batch_indices[i]), int(positions[i])
        if b < 0 or b >= table.shape[0] or t < 0 or t // page_size >= table.shape[1]:
            flags |= 2
            continue
        page = int(table[b, t // page_size])
        if page < 0 or page >= n_pages_k or page >= n_pages_v:
            flags |= 1
            continue
        slot = t % page_size
        k_view[page, :, slot, :] = k_new[i]
        v_view[page, :, slot, :] = v_new[i]
    return flags
