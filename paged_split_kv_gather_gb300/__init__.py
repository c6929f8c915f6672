"""paged_split_kv_gather_gb300 -- paged split-KV flash-decoding on GB300 (sm_103a).

A thin Python binding over the C ABI in ``include/fdec.h`` (``libfdec.so``):
the functions below carry the same names and only marshal arguments (tensor
pointers, strides, streams).  Every step of the computation runs in the CUDA
kernels of the library; PyTorch only provides device memory and streams.
There is no CPU fallback: if the library is not built, the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "FdecError", "KVDesc", "Plan", "PlanInfo", "fdec_plan", "fdec_plan_upload", "fdec_run",
    "fdec_merge_states", "fdec_plan_destroy", "fdec_plan_get_info", "fdec_plan_get_splits",
    "fdec_plan_set_split_event", "fdec_read_device_errors", "fdec_last_error", "fdec_version",
    "fdec_run_static_workspace", "fdec_append", "kv_desc", "library_path", "PagedDecode", "EXPORTED_SYMBOLS",
    "FDEC_F16", "FDEC_BF16", "FDEC_PATH_AUTO", "FDEC_PATH_SIMT", "FDEC_PATH_MMA", "FDEC_PATH_TC",
    "FDEC_KV_SAME", "FDEC_KV_E4M3", "FDEC_KV_Q8_0", "fdec_run_scaled", "fdec_append_e4m3", "fdec_run_q8_0",
    "DEVERR_PAGE_ID", "DEVERR_SEQ_LEN", "DEVERR_TIMEOUT",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfdec.so")

FDEC_F16, FDEC_BF16 = 0, 1
FDEC_PATH_AUTO, FDEC_PATH_SIMT, FDEC_PATH_MMA, FDEC_PATH_TC = 0, 1, 2, 3
FDEC_KV_SAME, FDEC_KV_E4M3, FDEC_KV_Q8_0 = 0, 1, 2
DEVERR_PAGE_ID, DEVERR_SEQ_LEN, DEVERR_TIMEOUT = 0x1, 0x2, 0x4

STATUS_NAMES = {
    0: "FDEC_OK", 1: "FDEC_ERR_INVALID_ARG", 2: "FDEC_ERR_LAYOUT", 3: "FDEC_ERR_UNSUPPORTED",
    4: "FDEC_ERR_CAPACITY", 5: "FDEC_ERR_CAPTURING", 6: "FDEC_ERR_WORKSPACE", 7: "FDEC_ERR_CUDA",
    8: "FDEC_ERR_DEVICE",
}

# Every entry point include/fdec.h declares.
EXPORTED_SYMBOLS = (
    "fdec_plan", "fdec_plan_upload", "fdec_run", "fdec_merge_states", "fdec_plan_destroy",
    "fdec_plan_get_info", "fdec_plan_get_splits", "fdec_plan_set_split_event",
    "fdec_read_device_errors", "fdec_last_error", "fdec_version", "fdec_run_static_workspace", "fdec_append",
    "fdec_run_scaled", "fdec_append_e4m3", "fdec_run_q8_0",
)


class FdecError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{self.status_name}: {message}")


class KVDesc(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("stride_page", ctypes.c_int64), ("stride_head", ctypes.c_int64),
                ("stride_token", ctypes.c_int64)]


class PlanOpts(ctypes.Structure):
    _fields_ = [("blocks_per_split", ctypes.c_int), ("reducer_fanin", ctypes.c_int),
                ("path", ctypes.c_int), ("num_sms", ctypes.c_int), ("kv_dtype", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("blocks_per_split", ctypes.c_int),
                ("num_items", ctypes.c_int), ("num_split_ctas", ctypes.c_int),
                ("row_groups", ctypes.c_int), ("rows_per_group", ctypes.c_int),
                ("max_splits", ctypes.c_int), ("reduce_passes", ctypes.c_int),
                ("launches", ctypes.c_int), ("num_sms", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
                "(or paged_split_kv_gather_gb300/_build.py) first; there is no fallback path")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, I64, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        lib.fdec_plan.restype = I
        lib.fdec_plan.argtypes = [P, I, I, I, I, I, I, I, I, ctypes.POINTER(PlanOpts), ctypes.POINTER(P),
                                  ctypes.POINTER(S)]
        lib.fdec_plan_upload.restype = I
        lib.fdec_plan_upload.argtypes = [P, P, P]
        lib.fdec_run.restype = I
        lib.fdec_run.argtypes = [P, P, I64, I64, KVDesc, KVDesc, P, I64, P, ctypes.c_float, P, P, P, P]
        lib.fdec_run_scaled.restype = I
        lib.fdec_run_scaled.argtypes = [P, P, I64, I64, KVDesc, KVDesc, P, I64, P, ctypes.c_float, ctypes.c_float,
                                        ctypes.c_float, P, P, P, P]
        lib.fdec_run_static_workspace.restype = I
        lib.fdec_run_q8_0.restype = I
        lib.fdec_run_q8_0.argtypes = [P, P, I64, I64, KVDesc, KVDesc, KVDesc, KVDesc, P, I64, P, ctypes.c_float, P,
                                      P, P, P]
        lib.fdec_run_static_workspace.argtypes = [P, P, I64, I64, KVDesc, KVDesc, P, I64, P, ctypes.c_float, P,
                                                  P, P]
        lib.fdec_merge_states.restype = I
        lib.fdec_merge_states.argtypes = [P, P, I, I, I, P, P, P]
        lib.fdec_append.restype = I
        lib.fdec_append.argtypes = [P, P, I64, I64, P, P, I, I, I, I, KVDesc, KVDesc, P, I, I64, P, P]
        lib.fdec_append_e4m3.restype = I
        lib.fdec_append_e4m3.argtypes = [P, P, I64, I64, P, P, I, I, I, I, KVDesc, KVDesc, P, I, I64, P, P]
        lib.fdec_plan_destroy.restype = I
        lib.fdec_plan_destroy.argtypes = [P]
        lib.fdec_plan_get_info.restype = I
        lib.fdec_plan_get_info.argtypes = [P, ctypes.POINTER(PlanInfo)]
        lib.fdec_plan_get_splits.restype = I
        lib.fdec_plan_get_splits.argtypes = [P, P, I]
        lib.fdec_plan_set_split_event.restype = I
        lib.fdec_plan_set_split_event.argtypes = [P, P]
        lib.fdec_read_device_errors.restype = I
        lib.fdec_read_device_errors.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32), I, P]
        lib.fdec_last_error.restype = ctypes.c_char_p
        lib.fdec_last_error.argtypes = []
        lib.fdec_version.restype = ctypes.c_char_p
        lib.fdec_version.argtypes = []
        _lib = lib
    return _lib


def _check(status: int):
    if status != 0:
        raise FdecError(status, fdec_last_error())


def fdec_last_error() -> str:
    return _load().fdec_last_error().decode()


def fdec_version() -> str:
    return _load().fdec_version().decode()


def _stream_handle(stream) -> Optional[int]:
    """cudaStream_t of a torch stream (None -> torch's current stream)."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owns an fdec_plan_t (host memory) and remembers what it was planned for."""

    def __init__(self, handle: int, workspace_bytes: int, batch: int, meta: dict):
        self.handle = handle
        self.workspace_bytes = workspace_bytes
        self.batch = batch
        self.meta = meta

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.fdec_plan_destroy(self.handle)
            self.handle = None


def fdec_plan(seq_lens: Sequence[int], q_len: int, page_size: int, num_qo_heads: int, num_kv_heads: int,
              head_dim: int, dtype: str = "bf16", causal: bool = False, blocks_per_split: int = 0,
              reducer_fanin: int = 0, path: int = FDEC_PATH_AUTO, num_sms: int = 0, kv_dtype: str = "") -> Plan:
    """kv_dtype: "" (K/V in the q dtype), "fp8" (E4M3 codes; scales go to fdec_run_scaled) or
    "q8_0" (int8 codes with binary16 block scales; see fdec_run_q8_0)."""
    lib = _load()
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(-1))
    kvd = {"": FDEC_KV_SAME, "fp8": FDEC_KV_E4M3, "q8_0": FDEC_KV_Q8_0}[kv_dtype]
    opts = PlanOpts(blocks_per_split, reducer_fanin, path, num_sms, kvd)
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    dt = {"f16": FDEC_F16, "bf16": FDEC_BF16}[dtype]
    _check(lib.fdec_plan(lens.ctypes.data, lens.shape[0], q_len, page_size, num_qo_heads, num_kv_heads,
                         head_dim, dt, int(bool(causal)), ctypes.byref(opts), ctypes.byref(handle),
                         ctypes.byref(ws)))
    meta = dict(q_len=q_len, page_size=page_size, num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, dtype=dtype, causal=causal, capacity=lens.copy(), kv_dtype=kv_dtype)
    return Plan(handle.value, ws.value, lens.shape[0], meta)


def fdec_plan_upload(plan: Plan, workspace, stream=None) -> None:
    _check(_load().fdec_plan_upload(plan.handle, workspace.data_ptr(), _stream_handle(stream)))


def fdec_plan_destroy(plan: Plan) -> None:
    if plan.handle:
        _check(_load().fdec_plan_destroy(plan.handle))
        plan.handle = None


def fdec_plan_get_info(plan: Plan) -> dict:
    info = PlanInfo()
    _check(_load().fdec_plan_get_info(plan.handle, ctypes.byref(info)))
    return info.as_dict()


def fdec_plan_get_splits(plan: Plan) -> np.ndarray:
    out = np.zeros(plan.batch, dtype=np.int32)
    _check(_load().fdec_plan_get_splits(plan.handle, out.ctypes.data, plan.batch))
    return out


def fdec_plan_set_split_event(plan: Plan, event) -> None:
    """event: a torch.cuda.Event (created), a raw cudaEvent_t int, or None."""
    if event is None:
        handle = None
    elif isinstance(event, int):
        handle = event
    else:
        handle = event.cuda_event
    _check(_load().fdec_plan_set_split_event(plan.handle, handle))


def fdec_read_device_errors(plan: Plan, workspace, clear: bool = True, stream=None) -> int:
    flags = ctypes.c_uint32()
    _check(_load().fdec_read_device_errors(plan.handle, workspace.data_ptr(), ctypes.byref(flags),
                                           int(bool(clear)), _stream_handle(stream)))
    return flags.value


def kv_desc(t) -> KVDesc:
    """Descriptor of a 4-D K or V view indexed [page, kv_head, slot, dim] (dim stride 1)."""
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("K/V views must be 4-D [page, kv_head, slot, dim] with a unit dim stride")
    return KVDesc(t.data_ptr(), t.shape[0], t.stride(0), t.stride(1), t.stride(2))


def _q_strides(q):
    batch, q_len = q.shape[0], q.shape[1]
    if q.stride(3) != 1:
        raise ValueError("q must have a unit head_dim stride")
    if q_len == 1:
        tok = q.stride(0)
    else:
        if batch > 1 and q.stride(0) != q_len * q.stride(1):
            raise ValueError("q tokens must flatten to one stride (b*q_len + i)")
        tok = q.stride(1)
    return tok, q.stride(2)


def fdec_run(plan: Plan, q, k, v, page_table, seq_lens, out, lse, workspace, scale: Optional[float] = None,
             stream=None) -> None:
    """q [B,Q,Hq,D] 16-bit; k, v: 4-D views [page, kv_head, slot, dim] or KVDesc; page_table int32
    [B, W]; seq_lens int32 [B]; out float32 [B,Q,Hq,D] contiguous; lse float32 [B,Q,Hq] or None."""
    kd = k if isinstance(k, KVDesc) else kv_desc(k)
    vd = v if isinstance(v, KVDesc) else kv_desc(v)
    if not out.is_contiguous() or (lse is not None and not lse.is_contiguous()):
        raise ValueError("out and lse must be contiguous")
    tok, head = _q_strides(q)
    if page_table.stride(1) != 1:
        raise ValueError("page_table rows must be contiguous")
    sc = 1.0 / math.sqrt(plan.meta["head_dim"]) if scale is None else float(scale)
    _check_kv_type(plan, k, v)
    _check(_load().fdec_run(plan.handle, q.data_ptr(), tok, head, kd, vd, page_table.data_ptr(),
                            page_table.stride(0), seq_lens.data_ptr(), sc, out.data_ptr(),
                            None if lse is None else lse.data_ptr(), workspace.data_ptr(),
                            _stream_handle(stream)))


def _check_kv_type(plan: Plan, k, v) -> None:
    """K/V tensors must hold the element type the plan was made for (1-byte E4M3 codes or 16-bit)."""
    want = 1 if plan.meta.get("kv_dtype") in ("fp8", "q8_0") else 2
    for t in (k, v):
        if not isinstance(t, KVDesc) and t.element_size() != want:
            raise ValueError(f"this plan reads {want}-byte K/V elements, got {t.dtype}")


def fdec_run_scaled(plan: Plan, q, k, v, page_table, seq_lens, out, lse, workspace, scale: Optional[float] = None,
                    k_scale: float = 1.0, v_scale: float = 1.0, stream=None) -> None:
    """fdec_run over a scaled cache: K = k_scale x stored K, V = v_scale x stored V (host floats)."""
    kd = k if isinstance(k, KVDesc) else kv_desc(k)
    vd = v if isinstance(v, KVDesc) else kv_desc(v)
    if not out.is_contiguous() or (lse is not None and not lse.is_contiguous()):
        raise ValueError("out and lse must be contiguous")
    tok, head = _q_strides(q)
    if page_table.stride(1) != 1:
        raise ValueError("page_table rows must be contiguous")
    sc = 1.0 / math.sqrt(plan.meta["head_dim"]) if scale is None else float(scale)
    _check_kv_type(plan, k, v)
    _check(_load().fdec_run_scaled(plan.handle, q.data_ptr(), tok, head, kd, vd, page_table.data_ptr(),
                                   page_table.stride(0), seq_lens.data_ptr(), sc, float(k_scale), float(v_scale),
                                   out.data_ptr(), None if lse is None else lse.data_ptr(), workspace.data_ptr(),
                                   _stream_handle(stream)))


def fdec_run_q8_0(plan: Plan, q, k, k_scales, v, v_scales, page_table, seq_lens, out, lse, workspace,
                  scale: Optional[float] = None, stream=None) -> None:
    """fdec_run over a q8_0 cache: k / v int8 code views [page, kv_head, slot, D], k_scales /
    v_scales binary16 views [page, kv_head, slot, D / 32] (element e of a row is
    scale[e // 32] * code[e])."""
    descs = [t if isinstance(t, KVDesc) else kv_desc(t) for t in (k, k_scales, v, v_scales)]
    if not out.is_contiguous() or (lse is not None and not lse.is_contiguous()):
        raise ValueError("out and lse must be contiguous")
    tok, head = _q_strides(q)
    if page_table.stride(1) != 1:
        raise ValueError("page_table rows must be contiguous")
    sc = 1.0 / math.sqrt(plan.meta["head_dim"]) if scale is None else float(scale)
    _check_kv_type(plan, k, v)
    for t in (k_scales, v_scales):
        if not isinstance(t, KVDesc) and t.element_size() != 2:
            raise ValueError(f"q8_0 scales are binary16, got {t.dtype}")
    _check(_load().fdec_run_q8_0(plan.handle, q.data_ptr(), tok, head, *descs, page_table.data_ptr(),
                                 page_table.stride(0), seq_lens.data_ptr(), sc, out.data_ptr(),
                                 None if lse is None else lse.data_ptr(), workspace.data_ptr(),
                                 _stream_handle(stream)))


def fdec_run_static_workspace(plan: Plan, q, k, v, page_table, seq_lens, out, lse, scale: Optional[float] = None,
                              stream=None) -> None:
    """fdec_run with the library's built-in workspace: no device allocation by anyone (see fdec.h)."""
    kd = k if isinstance(k, KVDesc) else kv_desc(k)
    vd = v if isinstance(v, KVDesc) else kv_desc(v)
    if not out.is_contiguous() or (lse is not None and not lse.is_contiguous()):
        raise ValueError("out and lse must be contiguous")
    tok, head = _q_strides(q)
    if page_table.stride(1) != 1:
        raise ValueError("page_table rows must be contiguous")
    sc = 1.0 / math.sqrt(plan.meta["head_dim"]) if scale is None else float(scale)
    _check_kv_type(plan, k, v)
    _check(_load().fdec_run_static_workspace(plan.handle, q.data_ptr(), tok, head, kd, vd, page_table.data_ptr(),
                                             page_table.stride(0), seq_lens.data_ptr(), sc, out.data_ptr(),
                                             None if lse is None else lse.data_ptr(), _stream_handle(stream)))


def _append(entry, elem_bytes, k_new, v_new, batch_indices, positions, k, v, page_table, page_size, device_errors,
            stream):
    if k_new.dim() != 3 or v_new.shape != k_new.shape or k_new.stride(2) != 1 or v_new.stride(2) != 1:
        raise ValueError("k_new and v_new must be [n, Hk, D] with a unit dim stride")
    if k_new.stride() != v_new.stride():
        raise ValueError("k_new and v_new must have the same strides")
    for t in (k_new, v_new, k, v):
        if t.element_size() != elem_bytes:
            raise ValueError(f"expected {elem_bytes}-byte elements, got {t.dtype}")
    n, hk, d = k_new.shape
    _check(entry(k_new.data_ptr(), v_new.data_ptr(), k_new.stride(0), k_new.stride(1), batch_indices.data_ptr(),
                 positions.data_ptr(), n, hk, d, page_size, kv_desc(k), kv_desc(v), page_table.data_ptr(),
                 page_table.shape[0], page_table.stride(0),
                 None if device_errors is None else device_errors.data_ptr(), _stream_handle(stream)))


def fdec_append(k_new, v_new, batch_indices, positions, k, v, page_table, page_size: int, device_errors=None,
                stream=None) -> None:
    """Write new tokens into the paged cache: k_new / v_new [n, Hk, D] (16-bit, unit
    dim stride), batch_indices / positions int32 [n] (device); k / v the cache
    views [page, kv_head, slot, dim]; page_table int32 [batch, stride];
    device_errors an optional int32/uint32 device tensor of one element."""
    _append(_load().fdec_append, 2, k_new, v_new, batch_indices, positions, k, v, page_table, page_size,
            device_errors, stream)


def fdec_append_e4m3(k_new, v_new, batch_indices, positions, k, v, page_table, page_size: int, device_errors=None,
                     stream=None) -> None:
    """fdec_append for E4M3 caches: k_new / v_new and the pools hold 1-byte codes
    (torch.float8_e4m3fn or uint8), copied unchanged."""
    _append(_load().fdec_append_e4m3, 1, k_new, v_new, batch_indices, positions, k, v, page_table, page_size,
            device_errors, stream)


def fdec_merge_states(o, lse, o_out, lse_out=None, stream=None) -> None:
    """o [n, rows, D] float32, lse [n, rows] float32 -> o_out [rows, D], lse_out [rows]."""
    if not (o.is_contiguous() and lse.is_contiguous() and o_out.is_contiguous()):
        raise ValueError("merge_states needs contiguous tensors")
    n, rows, d = o.shape
    _check(_load().fdec_merge_states(o.data_ptr(), lse.data_ptr(), n, rows, d, o_out.data_ptr(),
                                     None if lse_out is None else lse_out.data_ptr(),
                                     _stream_handle(stream)))


class PagedDecode:
    """Convenience holder: a plan, its torch-allocated workspace, uploaded once."""

    def __init__(self, capacities, q_len, page_size, num_qo_heads, num_kv_heads, head_dim, dtype="bf16",
                 causal=False, device=None, stream=None, **opts):
        import torch

        self.plan = fdec_plan(capacities, q_len, page_size, num_qo_heads, num_kv_heads, head_dim, dtype,
                              causal, **opts)
        self.workspace = torch.empty(max(self.plan.workspace_bytes, 256), dtype=torch.uint8,
                                     device=device or "cuda")
        fdec_plan_upload(self.plan, self.workspace, stream)

    def run(self, q, k, v, page_table, seq_lens, out, lse=None, scale=None, stream=None, k_scale=None,
            v_scale=None, k_scales=None, v_scales=None):
        if k_scales is not None or v_scales is not None:  # q8_0 block scales
            if k_scale is not None or v_scale is not None:
                raise ValueError("q8_0 caches take block scales, not k_scale / v_scale")
            fdec_run_q8_0(self.plan, q, k, k_scales, v, v_scales, page_table, seq_lens, out, lse, self.workspace,
                          scale, stream)
        elif k_scale is None and v_scale is None:
            fdec_run(self.plan, q, k, v, page_table, seq_lens, out, lse, self.workspace, scale, stream)
        else:
            fdec_run_scaled(self.plan, q, k, v, page_table, seq_lens, out, lse, self.workspace, scale,
                            1.0 if k_scale is None else k_scale, 1.0 if v_scale is None else v_scale, stream)

    def device_errors(self, clear=True, stream=None) -> int:
        return fdec_read_device_errors(self.plan, self.workspace, clear, stream)

    @property
    def info(self) -> dict:
        return fdec_plan_get_info(self.plan)
