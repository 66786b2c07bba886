"""Pins of the oracle's paged decode attention.

"Faster fuzzy minds" ("When scheduler does the work"; "Recurrent depth"):
decode runs one query per request over its cached KV, gathered through the
page table; the looped model is served as an ordinary deep transformer, so
each (layer, plane) bank is plain attention softmax(q K^T / sqrt(d)) V, with
GQA query-head groups sharing a kv head.

Pins: dense contiguous numpy attention on tiny inputs, closed forms (L = 1,
equal keys, q = 0, one dominant key), invariance under moving pages to other
physical slots, shared prefix pages versus private copies, and GQA equal to
MHA with the kv heads repeated.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as W
from test_oracle_paging import scatter_dense


def dense_attention(q, k, v, scale):
    """numpy fp64 softmax(q k^T * scale) v for one head: q [D], k/v [L][D]."""
    s = (k @ q) * scale
    m = s.max()
    w = np.exp(s - m)
    return (w[:, None] * v).sum(0) / w.sum(), m + math.log(w.sum())


def make_case(rng, seq_lens, Hq, Hkv, D, ps, extra_pages=3):
    B = len(seq_lens)
    Lmax = max(int(max(seq_lens)), 1)
    n = [-(-int(L) // ps) for L in seq_lens]
    P = sum(n) + extra_pages
    perm = rng.permutation(P)
    pt = np.full((B, max(max(n), 1)), -1, np.int32)
    c = 0
    for b in range(B):
        pt[b, : n[b]] = perm[c: c + n[b]]
        c += n[b]
    dk = W.bf16_normal(rng, (B, Lmax, Hkv, D))
    dv = W.bf16_normal(rng, (B, Lmax, Hkv, D))
    q = W.bf16_normal(rng, (B, Hq, D))
    sl = np.asarray(seq_lens, np.int32)
    kp = scatter_dense(dk, sl, pt, P, ps)
    vp = scatter_dense(dv, sl, pt, P, ps)
    return q, dk, dv, kp, vp, pt, sl


def f64(bits):
    return W.bf16_bits_to_float(bits).astype(np.float64)


@pytest.mark.parametrize("Hq,Hkv,D,ps", [(4, 2, 16, 4), (3, 3, 8, 16), (8, 1, 32, 1), (6, 2, 64, 16)])
def test_matches_dense_numpy_attention(Hq, Hkv, D, ps):
    rng = np.random.default_rng(Hq * 100 + D)
    seq_lens = [1, 5, 17, 40]
    q, dk, dv, kp, vp, pt, sl = make_case(rng, seq_lens, Hq, Hkv, D, ps)
    out, lse = oracle.decode_attn(q, kp, vp, pt, sl)
    G = Hq // Hkv
    scale = 1 / math.sqrt(D)
    for b, L in enumerate(seq_lens):
        for h in range(Hq):
            ref, ref_lse = dense_attention(f64(q[b, h]), f64(dk[b, :L, h // G]), f64(dv[b, :L, h // G]), scale)
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-13)
            assert lse[b, h] == pytest.approx(ref_lse, rel=1e-12, abs=1e-12)


def test_explicit_scale():
    rng = np.random.default_rng(21)
    q, dk, dv, kp, vp, pt, sl = make_case(rng, [9, 30], 2, 2, 16, 4)
    out, _ = oracle.decode_attn(q, kp, vp, pt, sl, scale=0.37)
    ref, _ = dense_attention(f64(q[1, 1]), f64(dk[1, :30, 1]), f64(dv[1, :30, 1]), 0.37)
    np.testing.assert_allclose(out[1, 1], ref, rtol=1e-12, atol=1e-13)
    out_d, _ = oracle.decode_attn(q, kp, vp, pt, sl)
    out_e, _ = oracle.decode_attn(q, kp, vp, pt, sl, scale=1 / 4.0)
    assert np.array_equal(out_d, out_e)


def test_single_token_returns_its_value_row():
    rng = np.random.default_rng(22)
    q, dk, dv, kp, vp, pt, sl = make_case(rng, [1, 1, 1], 4, 2, 32, 16)
    out, lse = oracle.decode_attn(q, kp, vp, pt, sl)
    for b in range(3):
        for h in range(4):
            assert np.array_equal(out[b, h], f64(dv[b, 0, h // 2]))
            assert lse[b, h] == pytest.approx(f64(q[b, h]) @ f64(dk[b, 0, h // 2]) / math.sqrt(32), abs=1e-12)


def test_equal_keys_and_zero_query_average_the_values():
    rng = np.random.default_rng(23)
    q, dk, dv, kp, vp, pt, sl = make_case(rng, [37, 64], 2, 1, 16, 8)
    kp[:] = kp[pt[0, 0], :, 0:1, :]                          # every key row identical
    out, lse = oracle.decode_attn(q, kp, vp, pt, sl)
    for b, L in enumerate([37, 64]):
        np.testing.assert_allclose(out[b, 0], f64(dv[b, :L, 0]).mean(0), rtol=0, atol=1e-13)
    q0 = np.zeros_like(q)
    q, dk, dv, kp, vp, pt, sl = make_case(rng, [50], 2, 1, 16, 8)
    out, lse = oracle.decode_attn(q0[:1], kp, vp, pt, sl)
    np.testing.assert_allclose(out[0, 1], f64(dv[0, :50, 0]).mean(0), rtol=0, atol=1e-13)
    assert lse[0, 0] == pytest.approx(math.log(50), abs=1e-13)


def test_one_dominant_key_selects_its_value():
    rng = np.random.default_rng(24)
    q, dk, dv, kp, vp, pt, sl = make_case(rng, [33], 1, 1, 16, 4)
    qv = f64(q[0, 0])
    big = W.float_to_bf16_bits(np.sign(qv) * 64.0)         # key aligned with q, huge score
    j = 19
    kp[pt[0, j // 4], 0, j % 4, :] = big
    out, _ = oracle.decode_attn(q, kp, vp, pt, sl)
    np.testing.assert_allclose(out[0, 0], f64(dv[0, j, 0]), atol=1e-12)


def test_empty_request_gives_zero_and_minus_inf():
    rng = np.random.default_rng(25)
    q, dk, dv, kp, vp, pt, sl = make_case(rng, [0, 7], 2, 2, 8, 4)
    out, lse = oracle.decode_attn(q, kp, vp, pt, sl)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_invariant_under_moving_pages():
    rng = np.random.default_rng(26)
    q, dk, dv, kp, vp, pt, sl = make_case(rng, [13, 29, 64], 4, 2, 16, 8)
    out, lse = oracle.decode_attn(q, kp, vp, pt, sl)
    P = kp.shape[0]
    new_of_old = rng.permutation(P)
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[new_of_old] = kp
    vp2[new_of_old] = vp
    pt2 = np.where(pt >= 0, new_of_old[np.maximum(pt, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.decode_attn(q, kp2, vp2, pt2, sl)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_shared_prefix_pages_equal_private_copies():
    rng = np.random.default_rng(27)
    ps, Hkv, D = 4, 2, 16
    prefix_pages = 5
    P = 40
    kp = W.bf16_normal(rng, (P, Hkv, ps, D))
    vp = W.bf16_normal(rng, (P, Hkv, ps, D))
    # shared: both requests point at pages 0..4 for their prefix, then private pages
    pt_shared = np.array([[0, 1, 2, 3, 4, 10, 11], [0, 1, 2, 3, 4, 20, -1]], np.int32)
    # private: request 1 gets its own copies of the prefix pages (30..34)
    kp[30:35] = kp[0:5]
    vp[30:35] = vp[0:5]
    pt_private = np.array([[0, 1, 2, 3, 4, 10, 11], [30, 31, 32, 33, 34, 20, -1]], np.int32)
    sl = np.array([27, 22], np.int32)
    q = W.bf16_normal(rng, (2, 4, D))
    a = oracle.decode_attn(q, kp, vp, pt_shared, sl)
    b = oracle.decode_attn(q, kp, vp, pt_private, sl)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(28)
    G, Hkv, D, ps = 4, 2, 16, 4
    q, dk, dv, kp, vp, pt, sl = make_case(rng, [11, 26], G * Hkv, Hkv, D, ps)
    out, lse = oracle.decode_attn(q, kp, vp, pt, sl)
    kp_rep = np.repeat(kp, G, axis=1)                 # kv head g -> heads g*G .. g*G+G-1
    vp_rep = np.repeat(vp, G, axis=1)
    out_m, lse_m = oracle.decode_attn(q, kp_rep, vp_rep, pt, sl)
    assert np.array_equal(out, out_m) and np.array_equal(lse, lse_m)


def test_banks_are_independent():
    rng = np.random.default_rng(29)
    q, dk, dv, kp, vp, pt, sl = make_case(rng, [10, 18], 2, 2, 8, 4)
    other = W.bf16_normal(rng, kp.shape)
    kp3 = np.stack([other, kp, other])
    vp3 = np.stack([other, vp, other])
    a = oracle.decode_attn(q, kp, vp, pt, sl)
    b = oracle.decode_attn(q, kp3, vp3, pt, sl, bank=1)
    assert np.array_equal(a[0], b[0])
