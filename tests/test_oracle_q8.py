"""Pins of the oracle's q8_0 path (K/V stored as blocks of 32 int8 codes with one
binary16 scale each: element e of a row is scale[e // 32] * code[e]), to facts
that do not come from the oracle: closed forms of attention (a single token, a
one-hot logit, identical keys), the block structure built into the inputs, and
a 16-bit cache holding the same values through the separately pinned 16-bit
path.  CPU only."""
import math

import numpy as np
import pytest

import oracle

D, P, HK, HQ = 64, 4, 2, 4  # two q8_0 blocks per row, pages of 4 tokens, two query heads per KV head


def _pools(codes, scales, layout="hnd"):
    """Code pool (int8) and scale pool (binary16 bits) from [pages, HK, P, D] and
    [pages, HK, P, D // 32] arrays, stored head-major ("hnd") or token-major ("nhd")."""
    pages = codes.shape[0]
    if layout == "nhd":
        c = np.ascontiguousarray(codes.transpose(0, 2, 1, 3))
        s = np.ascontiguousarray(scales.transpose(0, 2, 1, 3))
        cp = oracle.Pool(c.astype(np.int8), 0, pages, P * HK * D, D, HK * D)
        sp = oracle.Pool(s.astype(np.float16).view(np.uint16), 0, pages, P * HK * (D // 32), D // 32, HK * (D // 32))
    else:
        cp = oracle.Pool(np.ascontiguousarray(codes).astype(np.int8), 0, pages, HK * P * D, P * D, D)
        sp = oracle.Pool(np.ascontiguousarray(scales).astype(np.float16).view(np.uint16), 0, pages,
                         HK * P * (D // 32), P * (D // 32), D // 32)
    return cp, sp


def _run(q, k_codes, k_sc, v_codes, v_sc, table, lens, *, scale=1.0, layout="hnd", causal=False):
    """q: float16 [batch, q_len, HQ, D]."""
    kp, ksp = _pools(k_codes, k_sc, layout)
    vp, vsp = _pools(v_codes, v_sc, layout)
    b, ql = q.shape[0], q.shape[1]
    return oracle.paged_attention(q.astype(np.float16).view(np.uint16), 0, HQ * D, D, kp, vp, table, lens,
                                  q_len=ql, num_qo_heads=HQ, num_kv_heads=HK, head_dim=D, page_size=P,
                                  is_bf16=False, causal=causal, scale=scale, k_scales=ksp, v_scales=vsp)


def _zeros(pages):
    return (np.zeros((pages, HK, P, D), np.int8), np.ones((pages, HK, P, D // 32), np.float16))


def test_single_token_gives_its_dequantised_value():
    rng = np.random.default_rng(1)
    kc, ks = _zeros(3)
    vc, vs = _zeros(3)
    kc[2, 1, 0] = rng.integers(-128, 128, D)
    vc[2, 1, 0] = rng.integers(-128, 128, D)
    vs[2, 1, 0] = [0.75, -2.5]                      # a negative scale flips its block
    table = np.array([[2]], np.int32)               # the one token: slot 0 of physical page 2
    q = rng.standard_normal((1, 1, HQ, D)).astype(np.float16)
    out, _ = _run(q, kc, ks, vc, vs, table, np.array([1], np.int32))
    want = np.concatenate([0.75 * vc[2, 1, 0, :32].astype(float), -2.5 * vc[2, 1, 0, 32:].astype(float)])
    for h in (2, 3):                                 # query heads of KV head 1
        assert np.array_equal(out[0, 0, h], want)


def test_block_scales_apply_to_their_own_32_elements():
    kc, ks = _zeros(1)
    vc, vs = _zeros(1)
    vc[0, 0, 0] = 1                                  # every code 1
    vs[0, 0, 0] = [2.0 ** -3, 2.0 ** 5]
    out, _ = _run(np.zeros((1, 1, HQ, D), np.float16), kc, ks, vc, vs, np.array([[0]], np.int32),
                  np.array([1], np.int32))
    assert np.array_equal(out[0, 0, 0], np.array([2.0 ** -3] * 32 + [2.0 ** 5] * 32))


def test_codes_are_signed_bytes():
    kc, ks = _zeros(1)
    vc, vs = _zeros(1)
    vc[0, 0, 0] = np.concatenate([np.arange(-128, -96), np.arange(96, 128)]).astype(np.int8)
    out, _ = _run(np.zeros((1, 1, HQ, D), np.float16), kc, ks, vc, vs, np.array([[0]], np.int32),
                  np.array([1], np.int32))
    assert np.array_equal(out[0, 0, 1], np.concatenate([np.arange(-128, -96), np.arange(96, 128)]).astype(float))


@pytest.mark.parametrize("j", [3, 40])
def test_logits_carry_the_key_block_scale(j):
    # q is the unit vector on dim j; token t's key is code c_t on dim j with its block's scale d_t:
    # z_t = scale * d_t * c_t, so lse = ln sum_t exp(z_t) and out weighs V rows by softmax(z)
    c, d = [5, -7, 12], [0.5, 1.5, -0.25]
    kc, ks = _zeros(1)
    vc, vs = _zeros(1)
    for t in range(3):
        kc[0, 0, t, j] = c[t]
        ks[0, 0, t, j // 32] = d[t]
        ks[0, 0, t, 1 - j // 32] = 99.0             # the other block's scale must not matter
        vc[0, 0, t, 0] = t + 1
        vs[0, 0, t] = [4.0, 8.0]                     # V scales differ from K scales
    q = np.zeros((1, 1, HQ, D), np.float16)
    q[0, 0, 0, j] = 1.0
    out, lse = _run(q, kc, ks, vc, vs, np.array([[0]], np.int32), np.array([3], np.int32), scale=0.125)
    z = [0.125 * d[t] * c[t] for t in range(3)]
    m = max(z)
    sw = sum(math.exp(x - m) for x in z)
    assert abs(lse[0, 0, 0] - (m + math.log(sw))) < 1e-14
    want0 = sum(math.exp(z[t] - m) * 4.0 * (t + 1) for t in range(3)) / sw
    assert abs(out[0, 0, 0, 0] - want0) < 1e-13


def test_identical_keys_average_the_values():
    rng = np.random.default_rng(2)
    pages = 4
    kc = np.broadcast_to(rng.integers(-128, 128, D), (pages, HK, P, D)).astype(np.int8)
    ks = np.full((pages, HK, P, 2), 0.5, np.float16)
    vc = rng.integers(-128, 128, (pages, HK, P, D)).astype(np.int8)
    vs = rng.choice([0.25, 0.5, 1.0, 3.0], (pages, HK, P, 2)).astype(np.float16)
    table = np.array([[3, 0, 2, 1]], np.int32)
    q = rng.standard_normal((1, 1, HQ, D)).astype(np.float16)
    out, _ = _run(q, kc, ks, vc, vs, table, np.array([14], np.int32))
    for h in range(HQ):
        rows = [(table[0, t // P], h // 2, t % P) for t in range(14)]
        vals = np.array([np.repeat(vs[p, kh, s].astype(float), 32) * vc[p, kh, s] for p, kh, s in rows])
        assert np.allclose(out[0, 0, h], vals.mean(axis=0), rtol=0, atol=1e-12)


@pytest.mark.parametrize("layout", ["hnd", "nhd"])
def test_q8_0_cache_equals_f16_cache_of_the_same_values(layout):
    # power-of-two block scales keep scale * code exact in binary16, so an f16 cache can hold the
    # dequantised values; the separately pinned 16-bit path must then give the same doubles
    rng = np.random.default_rng(3)
    pages = 6
    kc = rng.integers(-128, 128, (pages, HK, P, D)).astype(np.int8)
    vc = rng.integers(-128, 128, (pages, HK, P, D)).astype(np.int8)
    ks = (2.0 ** rng.integers(-9, -2, (pages, HK, P, 2))).astype(np.float16)
    vs = (2.0 ** rng.integers(-6, 1, (pages, HK, P, 2))).astype(np.float16)
    table = np.array([[5, 1, 4, 0, 2], [3, 2, 0, 1, 4]], np.int32)
    lens = np.array([19, 7], np.int32)
    q = rng.standard_normal((2, 3, HQ, D)).astype(np.float16)
    o8, l8 = _run(q, kc, ks, vc, vs, table, lens, scale=0.2, layout=layout, causal=True)
    kf = (np.repeat(ks.astype(np.float64), 32, axis=-1) * kc).astype(np.float16)
    vf = (np.repeat(vs.astype(np.float64), 32, axis=-1) * vc).astype(np.float16)
    assert np.array_equal(kf.astype(np.float64), np.repeat(ks.astype(np.float64), 32, axis=-1) * kc)
    kp = oracle.Pool(kf.view(np.uint16), 0, pages, HK * P * D, P * D, D)
    vp = oracle.Pool(vf.view(np.uint16), 0, pages, HK * P * D, P * D, D)
    o16, l16 = oracle.paged_attention(q.view(np.uint16), 0, HQ * D, D, kp, vp, table, lens, q_len=3,
                                      num_qo_heads=HQ, num_kv_heads=HK, head_dim=D, page_size=P,
                                      is_bf16=False, causal=True, scale=0.2)
    assert np.array_equal(o8, o16) and np.array_equal(l8, l16)


def test_permuting_physical_pages_leaves_the_result():
    rng = np.random.default_rng(4)
    pages = 5
    kc = rng.integers(-128, 128, (pages, HK, P, D)).astype(np.int8)
    vc = rng.integers(-128, 128, (pages, HK, P, D)).astype(np.int8)
    ks = rng.uniform(0.01, 0.05, (pages, HK, P, 2)).astype(np.float16)
    vs = rng.uniform(0.01, 0.05, (pages, HK, P, 2)).astype(np.float16)
    table = np.array([[0, 1, 2, 3, 4]], np.int32)
    q = rng.standard_normal((1, 2, HQ, D)).astype(np.float16)
    o1, l1 = _run(q, kc, ks, vc, vs, table, np.array([18], np.int32), causal=True)
    perm = np.array([3, 0, 4, 1, 2])                 # physical page of logical page i
    kc2, vc2, ks2, vs2 = (np.empty_like(a) for a in (kc, vc, ks, vs))
    kc2[perm], vc2[perm], ks2[perm], vs2[perm] = kc, vc, ks, vs
    o2, l2 = _run(q, kc2, ks2, vc2, vs2, perm[None, :].astype(np.int32), np.array([18], np.int32), causal=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("layout", ["hnd", "nhd", "interleaved", "split2", "mixed", "interleaved_nhd"])
def test_q8_0_workloads_through_the_helpers_match_a_float64_softmax(layout):
    # the seeded q8_0 workloads and the test helpers that hand their pools to the oracle
    # (code and scale strides of every layout) against a float64 softmax over rows
    # gathered and dequantised here by plain indexing
    from paged_split_kv_gather_gb300 import workloads as W
    from tests.helpers import gather_tokens, oracle_run, visible

    w = W.make(2, 3, 8, 2, 64, 4, [30, 9], dtype="f16", seed=5, kv_dtype="q8_0", layout=layout, causal=True)
    out, lse = oracle_run(w)
    q = w.q.double().numpy()
    for b in range(w.batch):
        for kvh in range(w.num_kv_heads):
            n = int(w.seq_lens[b])
            k = gather_tokens(w, w.k, b, kvh, n) * np.repeat(gather_tokens(w, w.k_scales, b, kvh, n), 32, axis=1)
            v = gather_tokens(w, w.v, b, kvh, n) * np.repeat(gather_tokens(w, w.v_scales, b, kvh, n), 32, axis=1)
            for i in range(w.q_len):
                m = visible(w, b, i)
                for h in range(kvh * w.group, (kvh + 1) * w.group):
                    z = w.scale * (k[:m] @ q[b, i, h])
                    zm = z.max()
                    p = np.exp(z - zm)
                    assert np.allclose(out[b, i, h], p @ v[:m] / p.sum(), rtol=0, atol=1e-12)
                    assert abs(lse[b, i, h] - (zm + np.log(p.sum()))) < 1e-12
