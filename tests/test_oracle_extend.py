"""Pins for the oracle's extend (span) attention with causal masking.

"Faster fuzzy minds", LOTUS: a block of positions is re-forwarded in place, each
pass one parallel extend-prefill over the block (its K/V overwritten in the same
slots).  The extend oracle is the pinned decode oracle applied to each new
token's causal prefix; these pins check the causal structure itself: future
keys do not matter, the last new token equals plain decode over the whole
sequence, and dense causal softmax attention on tiny inputs agrees.
"""
import numpy as np

import oracle
import workloads as W


def small_case(seed, lens, new, ps=16, Hq=4, Hkv=2, D=32):
    case = W.custom(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, ps=ps, seq_lens=lens, seed=seed)
    h = W.host_tensors(case)
    rng = np.random.default_rng(seed)
    q = W.bf16_normal(rng, (int(sum(new)), Hq, D))
    return case, h, q


def test_future_keys_do_not_matter():
    lens, new = [40, 75, 16], [8, 20, 16]
    case, h, q = small_case(1, lens, new)
    out, lse = oracle.extend_attn(q, h.k_pool, h.v_pool, case.page_table, case.seq_lens, new)
    req, lim = oracle.extend_rows(case.page_table, case.seq_lens, new)
    # scramble every key past one token's limit: that token's output is unchanged
    t = 5
    kp = h.k_pool.copy()
    b = int(req[t])
    for pos in range(int(lim[t]), lens[b]):
        page, off = divmod(pos, case.page_size)
        kp[case.page_table[b, page], :, off] ^= 0x1234
    out2, lse2 = oracle.extend_attn(q, kp, h.v_pool, case.page_table, case.seq_lens, new)
    assert np.array_equal(out2[t], out[t]) and np.array_equal(lse2[t], lse[t])
    assert not np.array_equal(out2[int(np.flatnonzero(req == b)[-1])], out[int(np.flatnonzero(req == b)[-1])])


def test_last_new_token_is_plain_decode():
    lens, new = [33, 129, 64], [1, 30, 64]
    case, h, q = small_case(2, lens, new)
    out, lse = oracle.extend_attn(q, h.k_pool, h.v_pool, case.page_table, case.seq_lens, new)
    last = np.cumsum(new) - 1
    dec, dlse = oracle.decode_attn(q[last], h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    assert np.array_equal(out[last], dec) and np.array_equal(lse[last], dlse)


def test_matches_dense_causal_softmax_attention():
    lens, new = [20, 37], [20, 9]                      # a whole-prompt prefill and an extend
    case, h, q = small_case(3, lens, new, ps=4, Hq=2, Hkv=1, D=8)
    out, lse = oracle.extend_attn(q, h.k_pool, h.v_pool, case.page_table, case.seq_lens, new)
    k_all, v_all = oracle.paged_gather(h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    f = lambda bits: (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)
    qi = 0
    for b, (L, n) in enumerate(zip(lens, new)):
        K = f(k_all[b, :L, 0])                          # [L][D]
        V = f(v_all[b, :L, 0])
        Q = f(q[qi:qi + n])                             # [n][Hq][D]
        S = np.einsum("nhd,ld->nhl", Q, K) / np.sqrt(8)
        mask = np.arange(L)[None, :] > (L - n + np.arange(n))[:, None]
        S = np.where(mask[:, None, :], -np.inf, S)
        P = np.exp(S - S.max(-1, keepdims=True))
        ref = np.einsum("nhl,ld->nhd", P / P.sum(-1, keepdims=True), V)
        assert np.allclose(out[qi:qi + n], ref, rtol=1e-12, atol=1e-12)
        qi += n
