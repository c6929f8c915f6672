"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Closed forms, invariants, special cases that reduce to a library routine, and
brute force on tiny inputs.  The definition pinned is softmax(q K^T * scale) V
with its log-sum-exp over the tokens gathered through the page table (see the
header of oracle/oracle.c).  CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_split_kv_gather_gb300 import workloads as W
from tests.helpers import gather_tokens, oracle_run, visible

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# storage decoders: every bit pattern against numpy / torch
# --------------------------------------------------------------------------

def _decode_all(fn):
    return np.array([fn(b) for b in range(65536)], dtype=np.float64)


def test_f16_decoder_matches_numpy_on_all_bit_patterns():
    ref = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    got = _decode_all(oracle.f16_to_double)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decoder_matches_torch_on_all_bit_patterns():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).double().numpy()
    got = _decode_all(oracle.bf16_to_double)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

CASES = [
    dict(batch=1, q_len=1, hq=4, hk=1, d=64, p=16, lens=[300], dtype="f16", layout="nhd"),
    dict(batch=3, q_len=1, hq=8, hk=2, d=32, p=4, lens=[1, 13, 40], dtype="bf16", layout="hnd"),
    dict(batch=2, q_len=1, hq=6, hk=3, d=16, p=8, lens=[17, 64], dtype="f16", layout="interleaved"),
    dict(batch=2, q_len=1, hq=4, hk=2, d=16, p=2, lens=[9, 5], dtype="bf16", layout="split2"),
    dict(batch=2, q_len=1, hq=4, hk=2, d=16, p=4, lens=[6, 11], dtype="f16", layout="mixed"),
]


def _make(c, seed=0, **kw):
    return W.make(c["batch"], c["q_len"], c["hq"], c["hk"], c["d"], c["p"], c["lens"],
                  dtype=c["dtype"], layout=c["layout"], seed=seed, **kw)


@pytest.mark.parametrize("c", CASES)
def test_zero_query_gives_mean_of_values_and_log_count(c):
    w = _make(c)
    w.q.zero_()
    out, lse = oracle_run(w)
    g = w.group
    for b in range(w.batch):
        n = int(w.seq_lens[b])
        for h in range(w.num_qo_heads):
            vt = gather_tokens(w, w.v, b, h // g, n)
            np.testing.assert_allclose(out[b, 0, h], vt.mean(axis=0), rtol=0, atol=1e-13)
            assert abs(lse[b, 0, h] - math.log(n)) < 1e-13


@pytest.mark.parametrize("c", CASES)
def test_identical_keys_give_mean_and_shifted_lse(c):
    w = _make(c, seed=3)
    g = w.group
    for kvh in range(w.num_kv_heads):
        row = w.k[0, kvh, 0].clone()
        w.k[:, kvh] = row  # every key of this head is the same vector
    out, lse = oracle_run(w)
    for b in range(w.batch):
        n = int(w.seq_lens[b])
        for h in range(w.num_qo_heads):
            kvec = w.k[0, h // g, 0].double().numpy()
            qvec = w.q[b, 0, h].double().numpy()
            z = w.scale * float(qvec @ kvec)
            vt = gather_tokens(w, w.v, b, h // g, n)
            np.testing.assert_allclose(out[b, 0, h], vt.mean(axis=0), rtol=0, atol=1e-12)
            assert abs(lse[b, 0, h] - (z + math.log(n))) < 1e-12


def test_single_token_returns_its_value_exactly():
    w = W.make(2, 1, 4, 2, 32, 16, [1, 1], dtype="bf16", seed=5)
    out, lse = oracle_run(w)
    for b in range(2):
        for h in range(4):
            kvh = h // 2
            page = int(w.page_table[b, 0])
            v0 = w.v[page, kvh, 0].double().numpy()
            k0 = w.k[page, kvh, 0].double().numpy()
            q = w.q[b, 0, h].double().numpy()
            assert np.array_equal(out[b, 0, h], v0)
            assert abs(lse[b, 0, h] - w.scale * float(q @ k0)) < 1e-13


def test_one_hot_large_logit_selects_its_value():
    w = W.make(1, 1, 1, 1, 64, 16, [200], dtype="f16", seed=9)
    q = w.q[0, 0, 0]
    w.k.mul_(0.01)
    t_star = 137
    page = int(w.page_table[0, t_star // 16])
    # K_t* parallel to q and long enough that z_t* - max_others >= 40
    w.k[page, 0, t_star % 16] = (q.float() * (48.0 / (w.scale * q.float().pow(2).sum()))).half()
    out, lse = oracle_run(w)
    kq = w.k[page, 0, t_star % 16].double().numpy()
    z_star = w.scale * float(q.double().numpy() @ kq)
    ks = gather_tokens(w, w.k, 0, 0, 200)
    z = w.scale * ks @ q.double().numpy()
    others = np.delete(z, t_star)
    assert z_star - others.max() >= 40
    v_star = w.v[page, 0, t_star % 16].double().numpy()
    vnorm = np.abs(gather_tokens(w, w.v, 0, 0, 200)).max()
    assert np.max(np.abs(out[0, 0, 0] - v_star)) <= 200 * math.exp(-40) * vnorm * 2
    assert abs(lse[0, 0, 0] - z_star) <= 200 * math.exp(-40) + 1e-13


def test_causal_mask_is_bottom_right_aligned():
    # q = 0: row i sees exactly the first L - Q + i + 1 tokens, with equal weight
    w = W.make(2, 5, 4, 2, 16, 4, [20, 7], dtype="bf16", causal=True, seed=11)
    w.q.zero_()
    out, lse = oracle_run(w)
    for b in range(2):
        L = int(w.seq_lens[b])
        for i in range(5):
            n = L - 5 + i + 1
            for h in range(4):
                vt = gather_tokens(w, w.v, b, h // 2, n)
                np.testing.assert_allclose(out[b, i, h], vt.mean(axis=0), rtol=0, atol=1e-13)
                assert abs(lse[b, i, h] - math.log(n)) < 1e-13


def test_causal_rows_with_nothing_visible_are_empty():
    w = W.make(1, 6, 2, 1, 16, 4, [3], dtype="f16", causal=True, seed=2)
    out, lse = oracle_run(w)
    for i in range(6):
        if 3 - 6 + i + 1 <= 0:
            assert np.all(out[0, i] == 0) and np.all(np.isneginf(lse[0, i]))
        else:
            assert np.all(np.isfinite(lse[0, i]))


def test_empty_sequence_gives_zero_output_and_minus_inf_lse():
    w = W.make(2, 1, 4, 2, 16, 4, [0, 5], dtype="f16", seed=4)
    out, lse = oracle_run(w)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_bad_page_id_is_reported():
    w = W.make(1, 1, 2, 1, 16, 4, [8], dtype="f16", seed=4)
    w.page_table[0, 1] = w.k.shape[0] + 3
    with pytest.raises(ValueError):
        oracle_run(w)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def _repage(w, b, tokens, page_size, seed):
    """A batch-1 workload holding only ``tokens`` of sequence b (in that order), freshly paged."""
    n = len(tokens)
    sub = W.make(1, 1, w.num_qo_heads, w.num_kv_heads, w.head_dim, page_size, [n],
                 dtype=w.dtype, seed=seed)
    sub.q.copy_(w.q[b:b + 1])
    t = np.asarray(tokens)
    src_p = torch.as_tensor(w.page_table[b, t // w.page_size].astype(np.int64))
    src_s = torch.as_tensor((t % w.page_size).astype(np.int64))
    j = np.arange(n)
    dst_p = torch.as_tensor(sub.page_table[0, j // page_size].astype(np.int64))
    dst_s = torch.as_tensor((j % page_size).astype(np.int64))
    for kvh in range(w.num_kv_heads):
        sub.k[dst_p, kvh, dst_s] = w.k[src_p, kvh, src_s]
        sub.v[dst_p, kvh, dst_s] = w.v[src_p, kvh, src_s]
    return sub


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_any_partition_merged_by_lse_equals_unsplit(seed):
    rng = np.random.default_rng(seed)
    w = W.make(1, 1, 8, 2, 32, 16, [333], dtype="bf16", seed=seed, peaked=True)
    full_o, full_lse = oracle_run(w)
    L = 333
    if seed == 2:  # an arbitrary (non-contiguous) partition
        perm = rng.permutation(L)
        pieces = np.array_split(perm, 5)
    else:          # contiguous pieces of random sizes
        cuts = np.sort(rng.choice(np.arange(1, L), size=6, replace=False))
        pieces = np.split(np.arange(L), cuts)
    os_, ls_ = [], []
    for k, piece in enumerate(pieces):
        sub = _repage(w, 0, list(piece), page_size=8, seed=100 + k)
        o, l = oracle_run(sub)
        os_.append(o.reshape(-1, 32))
        ls_.append(l.reshape(-1))
    mo, ml = oracle.merge_states(np.stack(os_), np.stack(ls_))
    ref = full_o.reshape(-1, 32)
    assert np.max(np.abs(mo - ref)) <= 1e-12 * max(1.0, np.abs(ref).max())
    assert np.max(np.abs(ml - full_lse.reshape(-1))) <= 1e-12


def test_physical_page_permutation_is_bitwise_invisible():
    w = W.make(3, 1, 8, 4, 64, 16, [100, 250, 33], dtype="f16", seed=7, pool_pages=60)
    out0, lse0 = oracle_run(w)
    perm = np.random.default_rng(1).permutation(60)  # new position of every page
    inv = np.argsort(perm)
    k2 = w.k[torch.as_tensor(inv)].contiguous()
    v2 = w.v[torch.as_tensor(inv)].contiguous()
    w.k, w.v = k2, v2
    t = w.page_table
    w.page_table = np.where(t >= 0, perm[np.maximum(t, 0)], -1).astype(np.int32)
    out1, lse1 = oracle_run(w)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_gqa_equals_mha_with_replicated_kv_heads():
    w = W.make(2, 1, 8, 2, 32, 16, [70, 41], dtype="bf16", seed=8)
    out0, lse0 = oracle_run(w)
    g = 4
    w.k = w.k.repeat_interleave(g, dim=1)
    w.v = w.v.repeat_interleave(g, dim=1)
    w.num_kv_heads = 8
    out1, lse1 = oracle_run(w)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_logit_shift_moves_lse_only():
    w = W.make(2, 1, 4, 2, 32, 16, [50, 77], dtype="f16", seed=12)
    w.k[..., -1] = 1.0          # every key has a 1 in its last coordinate
    w.q[..., -1] = 0.5
    out0, lse0 = oracle_run(w)
    w.q[..., -1] = 2.5          # q' = q + 2 u, K u = 1  =>  z' = z + 2 * scale
    out1, lse1 = oracle_run(w)
    np.testing.assert_allclose(out1, out0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse1, lse0 + 2.0 * w.scale, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# library routine and brute force on tiny inputs
# --------------------------------------------------------------------------

TINY = [
    dict(batch=2, q_len=1, hq=4, hk=2, d=16, p=4, lens=[9, 23], dtype="bf16", layout="hnd"),
    dict(batch=1, q_len=3, hq=2, hk=1, d=8, p=2, lens=[11], dtype="f16", layout="nhd", causal=True),
    dict(batch=2, q_len=2, hq=6, hk=2, d=16, p=8, lens=[30, 3], dtype="bf16", layout="interleaved",
         causal=True, q_layout="fused_qkv"),
    dict(batch=2, q_len=1, hq=4, hk=4, d=8, p=1, lens=[7, 40], dtype="f16", layout="split2",
         q_layout="head_major"),
    dict(batch=2, q_len=1, hq=4, hk=2, d=8, p=4, lens=[10, 13], dtype="bf16", layout="mixed"),
]


def _make_tiny(c, seed):
    return W.make(c["batch"], c["q_len"], c["hq"], c["hk"], c["d"], c["p"], c["lens"],
                  dtype=c["dtype"], layout=c["layout"], causal=c.get("causal", False),
                  q_layout=c.get("q_layout", "packed"), seed=seed)


@pytest.mark.parametrize("c", TINY)
def test_matches_torch_float64_softmax_on_gathered_kv(c):
    w = _make_tiny(c, seed=21)
    out, lse = oracle_run(w)
    g = w.group
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        for h in range(w.num_qo_heads):
            K = torch.from_numpy(gather_tokens(w, w.k, b, h // g, L))
            V = torch.from_numpy(gather_tokens(w, w.v, b, h // g, L))
            for i in range(w.q_len):
                n = visible(w, b, i)
                q = w.q[b, i, h].double()
                s = (K[:n] @ q) * w.scale
                ref = torch.softmax(s, dim=0) @ V[:n]
                assert np.max(np.abs(out[b, i, h] - ref.numpy())) <= 1e-13
                assert abs(lse[b, i, h] - torch.logsumexp(s, dim=0).item()) <= 1e-13


@pytest.mark.parametrize("c", TINY)
def test_matches_pure_python_brute_force(c):
    w = _make_tiny(c, seed=33)
    out, lse = oracle_run(w)
    g = w.group
    D = w.head_dim
    for b in range(w.batch):
        for i in range(w.q_len):
            for h in range(w.num_qo_heads):
                qv = [float(x) for x in w.q[b, i, h].double()]
                num = [0.0] * D
                den = 0.0
                for t in range(visible(w, b, i)):
                    page = int(w.page_table[b][t // w.page_size])
                    slot = t % w.page_size
                    kv = [float(x) for x in w.k[page, h // g, slot].double()]
                    vv = [float(x) for x in w.v[page, h // g, slot].double()]
                    z = w.scale * sum(qv[e] * kv[e] for e in range(D))
                    assert abs(z) < 50
                    e_z = math.exp(z)  # no max subtraction
                    den += e_z
                    for e in range(D):
                        num[e] += e_z * vv[e]
                ref = [x / den for x in num]
                assert max(abs(out[b, i, h, e] - ref[e]) for e in range(D)) <= 1e-13
                assert abs(lse[b, i, h] - math.log(den)) <= 1e-13


# --------------------------------------------------------------------------
# the merge of normalised states
# --------------------------------------------------------------------------

def test_merge_single_state_is_identity():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((1, 5, 16))
    l = rng.standard_normal((1, 5))
    mo, ml = oracle.merge_states(o, l)
    np.testing.assert_allclose(mo, o[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(ml, l[0], rtol=0, atol=1e-15)


def test_merge_with_empty_state_is_identity_and_all_empty_is_empty():
    rng = np.random.default_rng(1)
    o = rng.standard_normal((3, 4, 8))
    l = np.array([[0.5, -1.0, 2.0, 7.0], [-np.inf] * 4, [-np.inf] * 4])
    mo, ml = oracle.merge_states(o, l)
    np.testing.assert_allclose(mo, o[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(ml, l[0], rtol=0, atol=1e-15)
    mo, ml = oracle.merge_states(o[1:], l[1:])
    assert np.all(mo == 0) and np.all(np.isneginf(ml))


def test_merge_of_equal_states_adds_log_two():
    rng = np.random.default_rng(2)
    o1 = rng.standard_normal((4, 8))
    l1 = rng.standard_normal(4)
    mo, ml = oracle.merge_states(np.stack([o1, o1]), np.stack([l1, l1]))
    np.testing.assert_allclose(mo, o1, rtol=0, atol=1e-14)
    np.testing.assert_allclose(ml, l1 + math.log(2.0), rtol=0, atol=1e-14)


def test_merge_weights_are_exponentials_of_lse():
    # two states with lse 0 and ln 3: weights 1/4 and 3/4
    o = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    l = np.array([[0.0], [math.log(3.0)]])
    mo, ml = oracle.merge_states(o, l)
    np.testing.assert_allclose(mo[0], [0.25, 0.75], rtol=0, atol=1e-15)
    assert abs(ml[0] - math.log(4.0)) < 1e-15


# --------------------------------------------------------------------------
# worked example (hand-derived, see the fixture's notes)
# --------------------------------------------------------------------------

def test_worked_example_fixture():
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        ex = json.load(f)
    P, D = ex["page_size"], ex["head_dim"]
    w = W.make(1, 1, ex["num_qo_heads"], ex["num_kv_heads"], D, P, [ex["seq_len"]],
               dtype="f16", seed=0, pool_pages=ex["pool_pages"], scale=ex["scale"])
    w.page_table[0, :] = ex["page_table"]
    w.k.zero_()
    w.v.zero_()
    for t, (kr, vr) in enumerate(zip(ex["keys"], ex["values"])):
        page, slot = ex["page_table"][t // P], t % P
        w.k[page, 0, slot] = torch.tensor(kr, dtype=torch.float16)
        w.v[page, 0, slot] = torch.tensor(vr, dtype=torch.float16)
    for h, qr in enumerate(ex["queries"]):
        w.q[0, 0, h] = torch.tensor(qr, dtype=torch.float16)
    out, lse = oracle_run(w)
    e = math.e
    for h, exp_case in enumerate(ex["expected"]):
        # the fixture states the logits; weights are exp(z)/sum exp(z) in closed form
        z = exp_case["logits"]
        den = sum(e ** x for x in z)
        ref = [sum(e ** z[t] * ex["values"][t][c] for t in range(len(z))) / den for c in range(D)]
        np.testing.assert_allclose(out[0, 0, h], ref, rtol=0, atol=1e-15)
        np.testing.assert_allclose(out[0, 0, h], exp_case["out_decimal"], rtol=0, atol=1e-9)
        assert abs(lse[0, 0, h] - math.log(den)) < 1e-15
        assert abs(lse[0, 0, h] - exp_case["lse_decimal"]) < 1e-9
