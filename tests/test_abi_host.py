"""Host-side tests of the C ABI (no GPU): symbols, planning, argument checks."""
import ctypes
import json
import os
import re
import subprocess

import numpy as np
import pytest

import paged_split_kv_gather_gb300 as fd
from paged_split_kv_gather_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fdec.h")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    if not os.path.exists(fd.library_path()):
        _build.build()
    return fd.library_path()


def declared_entry_points():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fdec_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_match_binding_list():
    assert declared_entry_points() == sorted(fd.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(fd.library_path())
    for name in declared_entry_points():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", fd.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (fdec_\w+)", out))
    assert set(declared_entry_points()) <= exported


def test_version_and_empty_error():
    assert "sm_103a" in fd.fdec_version()


def _plan(lens, **kw):
    args = dict(q_len=1, page_size=16, num_qo_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16")
    args.update(kw)
    args.setdefault("num_sms", 152)
    return fd.fdec_plan(lens, **args)


def test_capacity_rounds_up_to_64_token_blocks_golden():
    g = json.load(open(os.path.join(GOLDEN, "capacity_blocks.json")))
    for length, blocks in g["rows"]:
        p = _plan([length], blocks_per_split=1)
        assert int(fd.fdec_plan_get_splits(p)[0]) == blocks, (length, blocks)
        assert fd.fdec_plan_get_info(p)["max_splits"] == blocks


def test_split_path_is_planned_at_every_length_across_the_2048_boundary():
    # the pages' cliff: past 32 blocks the old matcher fell back to a serial kernel
    for length in (1900, 2000, 2048, 2049, 2100, 3000, 4800, 4864, 8192, 32768, 131072, 262144):
        p = _plan([length], num_qo_heads=32, num_kv_heads=4, page_size=64)
        info = fd.fdec_plan_get_info(p)
        assert info["path"] == fd.FDEC_PATH_MMA  # tensor-core split kernel by default for head_dim 128
        units = -(-length // 64) * 4
        assert info["num_split_ctas"] >= min(units, 152) // 2, (length, info)  # the grid fills the SMs
        if info["max_splits"] > 1:
            assert info["reduce_passes"] >= 1


def test_forced_one_block_per_split_uses_two_reduction_passes():
    p = _plan([262144], num_qo_heads=32, num_kv_heads=4, page_size=64, blocks_per_split=1)
    info = fd.fdec_plan_get_info(p)
    assert info["max_splits"] == 4096
    assert info["reduce_passes"] == 2          # 4096 -> 4 -> 1 with the default fan-in 1024
    assert info["launches"] == 3
    p = _plan([262144], num_qo_heads=32, num_kv_heads=4, page_size=64, blocks_per_split=1, reducer_fanin=4)
    assert fd.fdec_plan_get_info(p)["reduce_passes"] == 6   # 4096 = 4^6


def test_single_split_needs_no_reduction():
    p = _plan([300], num_qo_heads=4, num_kv_heads=1, head_dim=64, blocks_per_split=8)
    info = fd.fdec_plan_get_info(p)
    assert info["max_splits"] == 1 and info["reduce_passes"] == 0 and info["launches"] == 1


def test_auto_plan_balances_ragged_batches():
    lens = np.round(np.exp(np.random.default_rng(0).uniform(np.log(16), np.log(32768), 64))).astype(np.int32)
    p = _plan(lens, num_qo_heads=16, num_kv_heads=8, head_dim=256, dtype="f16")
    info = fd.fdec_plan_get_info(p)
    splits = fd.fdec_plan_get_splits(p)
    C = info["blocks_per_split"]
    nb = np.maximum(1, -(-lens // 64))
    assert np.array_equal(splits, -(-nb // C))
    assert info["num_items"] == int(splits.sum())


def test_path_selection():
    assert fd.fdec_plan_get_info(_plan([100], path=fd.FDEC_PATH_SIMT))["path"] == fd.FDEC_PATH_SIMT
    for d in (64, 128, 192, 256, 512):  # (1000 tokens: past the tiny-decode bound)
        assert fd.fdec_plan_get_info(_plan([1000], head_dim=d))["path"] == fd.FDEC_PATH_MMA
        assert fd.fdec_plan_get_info(_plan([100], head_dim=d, path=fd.FDEC_PATH_SIMT))["path"] == fd.FDEC_PATH_SIMT
    for d in (64, 128, 192, 256):
        assert fd.fdec_plan_get_info(_plan([100], head_dim=d, path=fd.FDEC_PATH_TC))["path"] == fd.FDEC_PATH_TC
    # head_dim 512: O alone would take all 512 tensor-memory columns
    with pytest.raises(fd.FdecError) as ei:
        _plan([100], head_dim=512, path=fd.FDEC_PATH_TC)
    assert ei.value.status_name == "FDEC_ERR_UNSUPPORTED"


def test_dense_query_rows_take_the_tcgen05_path():
    # q_len x group: 4 x 4 = 16 rows fit one group of the 16-row kernel; 8 x 4 = 32 would need two
    assert fd.fdec_plan_get_info(_plan([8200] * 4, q_len=4, num_qo_heads=32, num_kv_heads=8,
                                       causal=True))["path"] == fd.FDEC_PATH_MMA
    assert fd.fdec_plan_get_info(_plan([8200] * 4, q_len=8, num_qo_heads=32, num_kv_heads=8,
                                       causal=True))["path"] == fd.FDEC_PATH_TC
    assert fd.fdec_plan_get_info(_plan([1000], q_len=1, num_qo_heads=32, num_kv_heads=2))["path"] == fd.FDEC_PATH_MMA
    info = fd.fdec_plan_get_info(_plan([8200] * 4, q_len=16, num_qo_heads=32, num_kv_heads=8, causal=True))
    assert info["path"] == fd.FDEC_PATH_TC and info["rows_per_group"] == 128 and info["row_groups"] == 1
    info = fd.fdec_plan_get_info(_plan([10240] * 4, q_len=2048, num_qo_heads=32, num_kv_heads=8, causal=True))
    # more than 128 rows: two 128-row tiles per CTA share each staged K/V block
    assert info["path"] == fd.FDEC_PATH_TC and info["rows_per_group"] == 256
    assert info["row_groups"] == 2048 * 4 // 256
    assert info["num_split_ctas"] == info["num_items"] * 8 * info["row_groups"]
    # every head_dim the tcgen05 kernel is built for takes it above 16 rows (measured crossover);
    # two tiles per CTA where tensor memory holds them (head_dim up to 128)
    for d, tiles in ((64, 2), (128, 2), (192, 1), (256, 1)):
        info = fd.fdec_plan_get_info(_plan([1000], q_len=64, head_dim=d))
        assert info["path"] == fd.FDEC_PATH_TC and info["rows_per_group"] == 128 * tiles, (d, info)
        assert fd.fdec_plan_get_info(_plan([1000], q_len=4, head_dim=d))["path"] == fd.FDEC_PATH_MMA
    # head_dim 512 keeps the 16-row kernel at any row count
    assert fd.fdec_plan_get_info(_plan([1000], q_len=64, head_dim=512))["path"] == fd.FDEC_PATH_MMA


def test_row_groups_cover_all_query_rows():
    p = _plan([8200] * 4, q_len=8, num_qo_heads=32, num_kv_heads=8, causal=True)
    info = fd.fdec_plan_get_info(p)
    assert info["rows_per_group"] * info["row_groups"] >= 32
    p = _plan([1000], num_qo_heads=16, num_kv_heads=8, head_dim=512, q_len=3, path=fd.FDEC_PATH_SIMT)
    info = fd.fdec_plan_get_info(p)
    assert info["rows_per_group"] <= 4 and info["rows_per_group"] * info["row_groups"] >= 6
    p = _plan([1000], num_qo_heads=16, num_kv_heads=8, head_dim=512, q_len=3)  # tensor cores: one 16-row group
    info = fd.fdec_plan_get_info(p)
    assert info["rows_per_group"] == 16 and info["row_groups"] == 1


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=100), "FDEC_ERR_UNSUPPORTED"),
    (dict(page_size=3), "FDEC_ERR_UNSUPPORTED"),
    (dict(page_size=512), "FDEC_ERR_UNSUPPORTED"),
    (dict(num_qo_heads=30, num_kv_heads=8), "FDEC_ERR_INVALID_ARG"),
    (dict(q_len=0), "FDEC_ERR_INVALID_ARG"),
    (dict(reducer_fanin=1), "FDEC_ERR_INVALID_ARG"),
    (dict(path=7), "FDEC_ERR_INVALID_ARG"),
])
def test_plan_rejects_bad_arguments(kw, status):
    with pytest.raises(fd.FdecError) as ei:
        _plan([100], **kw)
    assert ei.value.status_name == status


def test_plan_rejects_negative_capacity():
    with pytest.raises(fd.FdecError) as ei:
        _plan([10, -1])
    assert ei.value.status_name == "FDEC_ERR_INVALID_ARG"


def test_plan_without_device_or_sm_count_reports_cuda_error():
    import torch

    if torch.cuda.is_available():
        pytest.skip("a device is present")
    with pytest.raises(fd.FdecError) as ei:
        fd.fdec_plan([100], 1, 16, 4, 1, 64, "f16", num_sms=0)
    assert ei.value.status_name == "FDEC_ERR_CUDA"


class _FakeTensor:
    """Just enough of a tensor for argument marshalling (never dereferenced on the host)."""

    def __init__(self, ptr, shape, strides):
        self._ptr, self.shape, self._strides = ptr, shape, strides

    def data_ptr(self):
        return self._ptr

    def stride(self, i=None):
        return self._strides if i is None else self._strides[i]

    def dim(self):
        return len(self.shape)

    def is_contiguous(self):
        return True


def _run_raw(plan, k, v, q=0x10000, out=0x20000, ws=0x30000, lse=None, pt_stride=None):
    lib = fd._load()
    st = lib.fdec_run(plan.handle, q, 128, 128 * 8, k, v, 0x40000, pt_stride or 256, 0x50000,
                      ctypes.c_float(0.1), out, lse, ws, None)
    return fd.STATUS_NAMES[st], fd.fdec_last_error()


def test_run_layout_checks_happen_before_any_launch():
    plan = _plan([2048], num_qo_heads=8, num_kv_heads=1, head_dim=128)
    good = fd.KVDesc(0x100000, 10, 16 * 128, 0, 128)
    assert _run_raw(plan, fd.KVDesc(0x100008, 10, 16 * 128, 0, 128), good)[0] == "FDEC_ERR_LAYOUT"
    assert _run_raw(plan, good, fd.KVDesc(0x100000, 10, 16 * 128 + 4, 0, 128))[0] == "FDEC_ERR_LAYOUT"
    assert _run_raw(plan, good, fd.KVDesc(0x100000, 10, 16 * 128, 0, 130))[0] == "FDEC_ERR_LAYOUT"
    assert _run_raw(plan, good, fd.KVDesc(0, 10, 16 * 128, 0, 128))[0] == "FDEC_ERR_INVALID_ARG"
    assert _run_raw(plan, good, fd.KVDesc(0x100000, 0, 16 * 128, 0, 128))[0] == "FDEC_ERR_INVALID_ARG"
    assert _run_raw(plan, good, good, pt_stride=100)[0] == "FDEC_ERR_CAPACITY"   # needs 128 pages
    assert _run_raw(plan, good, good, out=0x20002)[0] == "FDEC_ERR_LAYOUT"
    # everything valid but never uploaded: the workspace check
    assert _run_raw(plan, good, good)[0] == "FDEC_ERR_WORKSPACE"


def test_merge_states_rejects_bad_sizes():
    lib = fd._load()
    assert fd.STATUS_NAMES[lib.fdec_merge_states(0x1000, 0x2000, 0, 4, 64, 0x3000, None, None)] == \
        "FDEC_ERR_INVALID_ARG"
    assert fd.STATUS_NAMES[lib.fdec_merge_states(0x1000, 0x2000, 2, 4, 513, 0x3000, None, None)] == \
        "FDEC_ERR_INVALID_ARG"
    assert fd.STATUS_NAMES[lib.fdec_merge_states(None, 0x2000, 2, 4, 64, 0x3000, None, None)] == \
        "FDEC_ERR_INVALID_ARG"


def test_upload_refuses_null_and_misaligned_workspace():
    plan = _plan([100])
    lib = fd._load()
    assert fd.STATUS_NAMES[lib.fdec_plan_upload(plan.handle, None, None)] == "FDEC_ERR_INVALID_ARG"
    assert fd.STATUS_NAMES[lib.fdec_plan_upload(plan.handle, 0x1008, None)] == "FDEC_ERR_WORKSPACE"


def test_binding_refuses_views_without_a_unit_dim_stride():
    import torch

    kv = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16)
    assert fd.kv_desc(kv).stride_token == 64
    with pytest.raises(ValueError):
        fd.kv_desc(kv.transpose(2, 3))          # dim stride 16
    with pytest.raises(ValueError):
        fd.kv_desc(kv[:, :, :, ::2])             # dim stride 2
    q = torch.zeros(2, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fd._q_strides(q.transpose(2, 3).contiguous().transpose(2, 3))


def test_e4m3_cache_plans_on_the_mma_path_only():
    for d in (128, 256):
        info = fd.fdec_plan_get_info(_plan([1000], head_dim=d, kv_dtype="fp8"))
        assert info["path"] == fd.FDEC_PATH_MMA
    # rows above 16 stay on the 16-row kernel (row groups) for E4M3 caches
    info = fd.fdec_plan_get_info(_plan([8200] * 4, q_len=8, causal=True, kv_dtype="fp8"))
    assert info["path"] == fd.FDEC_PATH_MMA and info["row_groups"] == 2
    for kw in (dict(head_dim=64), dict(head_dim=192), dict(head_dim=512), dict(path=fd.FDEC_PATH_TC),
               dict(path=fd.FDEC_PATH_SIMT)):
        with pytest.raises(fd.FdecError) as ei:
            _plan([1000], kv_dtype="fp8", **kw)
        assert ei.value.status_name == "FDEC_ERR_UNSUPPORTED"


def _run_scaled_raw(plan, k, v, k_scale=1.0, v_scale=1.0):
    lib = fd._load()
    st = lib.fdec_run_scaled(plan.handle, 0x10000, 128, 128 * 8, k, v, 0x40000, 256, 0x50000, ctypes.c_float(0.1),
                             ctypes.c_float(k_scale), ctypes.c_float(v_scale), 0x20000, None, 0x30000, None)
    return fd.STATUS_NAMES[st]


def test_e4m3_strides_are_checked_in_bytes_and_scales_must_be_finite():
    plan = _plan([2048], num_qo_heads=8, num_kv_heads=1, head_dim=128, kv_dtype="fp8")
    good = fd.KVDesc(0x100000, 10, 16 * 128, 0, 128)
    assert _run_scaled_raw(plan, good, good) == "FDEC_ERR_WORKSPACE"  # valid, never uploaded
    # 8 elements is 16 bytes of a 16-bit cache but only 8 bytes of codes
    assert _run_scaled_raw(plan, good, fd.KVDesc(0x100000, 10, 16 * 128 + 8, 0, 128)) == "FDEC_ERR_LAYOUT"
    assert _run_scaled_raw(plan, good, fd.KVDesc(0x100000, 10, 16 * 128 + 16, 0, 128)) == "FDEC_ERR_WORKSPACE"
    for ks, vs in ((float("inf"), 1.0), (1.0, float("nan")), (-float("inf"), 1.0)):
        assert _run_scaled_raw(plan, good, good, ks, vs) == "FDEC_ERR_INVALID_ARG"


def test_q8_0_cache_plans_on_the_mma_path_only():
    for d in (128, 256):
        info = fd.fdec_plan_get_info(_plan([1000], head_dim=d, kv_dtype="q8_0"))
        assert info["path"] == fd.FDEC_PATH_MMA
        assert info["num_split_ctas"] == info["num_items"] * info["row_groups"] * 8  # one CTA per unit (8 KV heads)
    for kw in (dict(head_dim=64), dict(head_dim=192), dict(head_dim=512), dict(path=fd.FDEC_PATH_TC),
               dict(path=fd.FDEC_PATH_SIMT)):
        with pytest.raises(fd.FdecError) as ei:
            _plan([1000], kv_dtype="q8_0", **kw)
        assert ei.value.status_name == "FDEC_ERR_UNSUPPORTED"


def _run_q8_raw(plan, k, ks, v, vs):
    lib = fd._load()
    st = lib.fdec_run_q8_0(plan.handle, 0x10000, 128, 128 * 8, k, ks, v, vs, 0x40000, 256, 0x50000,
                           ctypes.c_float(0.1), 0x20000, None, 0x30000, None)
    return fd.STATUS_NAMES[st]


def test_q8_0_entry_points_and_scale_pool_layout_checks():
    plan = _plan([2048], num_qo_heads=8, num_kv_heads=1, head_dim=128, kv_dtype="q8_0")
    codes = fd.KVDesc(0x100000, 10, 16 * 128, 0, 128)
    scales = fd.KVDesc(0x200000, 10, 16 * 4, 0, 4)  # [pages, 1, 16, 4] binary16
    assert _run_q8_raw(plan, codes, scales, codes, scales) == "FDEC_ERR_WORKSPACE"  # valid, never uploaded
    # the 16-bit entry points refuse a q8_0 plan (they have no scale pools)
    assert _run_scaled_raw(plan, codes, codes) == "FDEC_ERR_INVALID_ARG"
    # scale rows must start on head_dim / 16 bytes: base, then each stride
    assert _run_q8_raw(plan, codes, fd.KVDesc(0x200004, 10, 64, 0, 4), codes, scales) == "FDEC_ERR_LAYOUT"
    assert _run_q8_raw(plan, codes, scales, codes, fd.KVDesc(0x200000, 10, 66, 0, 4)) == "FDEC_ERR_LAYOUT"
    assert _run_q8_raw(plan, codes, fd.KVDesc(0x200000, 10, 64, 0, 6), codes, scales) == "FDEC_ERR_LAYOUT"
    assert _run_q8_raw(plan, codes, fd.KVDesc(0x200000, 0, 64, 0, 4), codes, scales) == "FDEC_ERR_INVALID_ARG"
    assert _run_q8_raw(plan, codes, fd.KVDesc(0, 10, 64, 0, 4), codes, scales) == "FDEC_ERR_INVALID_ARG"
    # the q8_0 entry point refuses a plan of another cache type
    plan16 = _plan([2048], num_qo_heads=8, num_kv_heads=1, head_dim=128)
    assert _run_q8_raw(plan16, codes, scales, codes, scales) == "FDEC_ERR_INVALID_ARG"


def test_binding_refuses_k_v_of_the_wrong_element_size():
    import torch

    plan = _plan([64], num_qo_heads=8, num_kv_heads=1, head_dim=128, kv_dtype="fp8")
    k16 = torch.zeros(4, 1, 16, 128, dtype=torch.bfloat16)
    k8 = torch.zeros(4, 1, 16, 128, dtype=torch.float8_e4m3fn)
    q = torch.zeros(1, 1, 8, 128, dtype=torch.bfloat16)
    out = torch.zeros(1, 1, 8, 128)
    with pytest.raises(ValueError):
        fd.fdec_run_scaled(plan, q, k16, k16, torch.zeros(1, 4, dtype=torch.int32), torch.zeros(1, dtype=torch.int32),
                           out, None, torch.zeros(256, dtype=torch.uint8), k_scale=0.5)
    plan16 = _plan([64], num_qo_heads=8, num_kv_heads=1, head_dim=128)
    with pytest.raises(ValueError):
        fd.fdec_run(plan16, q, k8, k8, torch.zeros(1, 4, dtype=torch.int32), torch.zeros(1, dtype=torch.int32),
                    out, None, torch.zeros(256, dtype=torch.uint8))


def test_tiny_decodes_plan_on_the_simt_kernel():
    # one token, <= 4 rows per KV head, head_dim <= 128, every sequence within 5 blocks, <= one
    # (sequence, KV head) pair per SM: the SIMT kernel; one step past any bound: the tensor-core one
    info = fd.fdec_plan_get_info(_plan([300], num_qo_heads=4, num_kv_heads=1, head_dim=64))
    assert info["path"] == fd.FDEC_PATH_SIMT and info["launches"] == 1
    assert fd.fdec_plan_get_info(_plan([320] * 4, num_qo_heads=32, num_kv_heads=8, head_dim=128))["path"] == \
        fd.FDEC_PATH_SIMT
    for kw in (dict(lens=[321]), dict(num_qo_heads=8), dict(head_dim=192), dict(q_len=2),
               dict(lens=[64] * 153)):
        args = dict(lens=[300], num_qo_heads=4, num_kv_heads=1, head_dim=64)
        args.update(kw)
        lens = args.pop("lens")
        assert fd.fdec_plan_get_info(_plan(lens, **args))["path"] == fd.FDEC_PATH_MMA, kw
    # quantised caches stay on the tensor-core kernel
    assert fd.fdec_plan_get_info(_plan([300], num_qo_heads=4, num_kv_heads=1, head_dim=128, kv_dtype="fp8"))[
        "path"] == fd.FDEC_PATH_MMA


def test_plan_invariants_hold_for_random_batches():
    """Property check of the planner over random batches: split counts follow the
    chosen blocks per split, items and CTAs cover every (split, KV head, row group),
    the reduction has exactly the passes a fan-in F tree needs, the path choice
    follows the row count, and the workspace holds every partial."""
    hypothesis = pytest.importorskip("hypothesis")
    st = hypothesis.strategies

    @hypothesis.settings(max_examples=60, deadline=None, derandomize=True)
    @hypothesis.given(lens=st.lists(st.integers(0, 100000), min_size=1, max_size=12), q_len=st.integers(1, 12),
                      group=st.sampled_from([1, 2, 4, 8]), hk=st.sampled_from([1, 2, 8]),
                      d=st.sampled_from([64, 128, 192, 256, 512]), bps=st.integers(0, 40),
                      fanin=st.sampled_from([0, 2, 3, 16]), kv8=st.booleans())
    def check(lens, q_len, group, hk, d, bps, fanin, kv8):
        if kv8 and d not in (128, 256):
            d = 128
        p = _plan(lens, q_len=q_len, num_qo_heads=hk * group, num_kv_heads=hk, head_dim=d, blocks_per_split=bps,
                  reducer_fanin=fanin, kv_dtype="fp8" if kv8 else "", causal=q_len > 1)
        info = fd.fdec_plan_get_info(p)
        splits = fd.fdec_plan_get_splits(p).astype(np.int64)
        C = info["blocks_per_split"]
        if bps:
            assert C == bps
        nb = np.maximum(1, -(-np.asarray(lens, dtype=np.int64) // 64))
        rows = q_len * group
        tiny = (not kv8 and q_len == 1 and rows <= 4 and d <= 128 and len(lens) * hk <= 152
                and max(lens) <= 5 * 64)
        want_path = (fd.FDEC_PATH_SIMT if tiny else
                     fd.FDEC_PATH_TC if (not kv8 and d in (64, 128, 192, 256) and rows > (32 if d == 256 else 16))
                     else fd.FDEC_PATH_MMA)
        assert info["path"] == want_path
        # the persistent kernel (16-bit caches on the 16-row path; one CTA per SM at head_dim 512)
        persistent = want_path == fd.FDEC_PATH_MMA and not kv8
        assert np.array_equal(splits, -(-nb // C))
        assert info["num_items"] == int(splits.sum()) and info["max_splits"] == int(splits.max())
        assert info["row_groups"] == -(-rows // info["rows_per_group"])
        units = info["num_items"] * hk * info["row_groups"]
        assert info["num_split_ctas"] == (min(units, 152 * (1 if d == 512 else 2)) if persistent else units)
        F = fanin or 1024
        n, passes = int(splits.max()), 0
        while n > 1:
            n, passes = -(-n // F), passes + 1
        assert info["reduce_passes"] == passes and info["launches"] == 1 + passes
        partial_rows = int(splits[splits > 1].sum()) * hk * rows
        assert info["workspace_bytes"] >= partial_rows * (4 * d + 8)

    check()
