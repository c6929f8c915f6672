"""Pins of the oracle's quantised-cache path (K/V stored as 8-bit E4M3 codes with
a k_scale and a v_scale), to facts that do not come from the oracle: the E4M3
format's definition on every code, torch's float8_e4m3fn conversion, a 16-bit
cache holding the same values, scale identities and a float64 softmax on the
dequantised gathered rows.  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import gather_tokens, oracle_run, visible


def test_e4m3_decoder_matches_torch_on_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # only S.1111.111
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decoder_format_facts():
    assert oracle.e4m3_to_double(0x38) == 1.0          # exponent 7 = bias
    assert oracle.e4m3_to_double(0xB8) == -1.0
    assert oracle.e4m3_to_double(0x7E) == 448.0        # largest: 1.75 * 2^8
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6    # smallest normal
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9    # smallest subnormal
    assert oracle.e4m3_to_double(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_to_double(0x00) == 0.0 and math.copysign(1, oracle.e4m3_to_double(0x80)) == -1
    assert math.isnan(oracle.e4m3_to_double(0x7F)) and math.isnan(oracle.e4m3_to_double(0xFF))
    # consecutive codes within a binade differ by one ulp = 2^(e-7) / 8
    for e in range(1, 15):
        base = e << 3
        vals = [oracle.e4m3_to_double(base + m) for m in range(8)]
        assert np.allclose(np.diff(vals), 2.0 ** (e - 7) / 8, rtol=0, atol=0)


def _fp8_case(seed, **kw):
    kw.setdefault("layout", "hnd")
    return W.make(2, kw.pop("q_len", 1), 8, 2, 64, 16, [70, 33], dtype="bf16", seed=seed, kv_dtype="fp8", **kw)


def _as_bf16_cache(w, k_scale, v_scale):
    """The same workload with K/V stored as bf16 holding scale * decoded E4M3 values
    (exact for power-of-two scales: E4M3 has 3 fraction bits, bf16 has 7)."""
    k = (w.k.to(torch.float64) * k_scale).to(torch.bfloat16)
    v = (w.v.to(torch.float64) * v_scale).to(torch.bfloat16)
    assert torch.equal(k.to(torch.float64), w.k.to(torch.float64) * k_scale)
    return W.Workload(w.name, w.dtype, w.batch, w.q_len, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size,
                      w.causal, w.scale, w.seq_lens, w.page_table, w.q, k, v, w.layout, [w.q, k, v])


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.5, 4.0), (2.0 ** -3, 2.0 ** 5)])
def test_fp8_cache_equals_bf16_cache_of_the_dequantised_values(k_scale, v_scale):
    w = _fp8_case(1, peaked=True)
    o8, l8 = oracle_run(w, k_scale=k_scale, v_scale=v_scale)
    o16, l16 = oracle_run(_as_bf16_cache(w, k_scale, v_scale))
    assert np.array_equal(o8, o16) and np.array_equal(l8, l16)


def test_v_scale_scales_out_and_leaves_lse():
    w = _fp8_case(2, q_len=3, causal=True)
    o1, l1 = oracle_run(w)
    o3, l3 = oracle_run(w, v_scale=0.37)
    assert np.array_equal(l1, l3)
    assert np.abs(o3 - 0.37 * o1).max() <= 1e-14 * np.abs(o1).max()  # summation order only


def test_k_scale_acts_as_a_logit_scale():
    w = _fp8_case(3)
    o1, l1 = oracle_run(w, k_scale=0.37)
    w2 = W.Workload(**{**w.__dict__, "scale": w.scale * 0.37})
    o2, l2 = oracle_run(w2)
    assert np.allclose(o1, o2, rtol=0, atol=1e-13) and np.allclose(l1, l2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("layout", ["hnd", "nhd", "interleaved"])
def test_fp8_matches_torch_float64_softmax_on_dequantised_rows(layout):
    w = _fp8_case(4, layout=layout, q_len=2, causal=True)
    ks, vs = 0.8, 1.7
    out, lse = oracle_run(w, k_scale=ks, v_scale=vs)
    g = w.group
    for b in range(w.batch):
        for i in range(w.q_len):
            n = visible(w, b, i)
            for h in range(w.num_qo_heads):
                kvh = h // g
                K = torch.from_numpy(gather_tokens(w, w.k, b, kvh, n)) * ks
                V = torch.from_numpy(gather_tokens(w, w.v, b, kvh, n)) * vs
                q = w.q[b, i, h].double()
                z = w.scale * (K @ q)
                ref = torch.softmax(z, 0) @ V
                assert torch.allclose(torch.from_numpy(out[b, i, h]), ref, rtol=0, atol=1e-12)
                assert abs(lse[b, i, h] - torch.logsumexp(z, 0).item()) < 1e-12
