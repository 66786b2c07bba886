"""Pins of the oracle's bank map, slot mapping, gather and KV append.

"Faster fuzzy minds", "When scheduler does the work": the KV is a flat pool
of fixed-size slots addressed through page_table[request, position], so a
sequence's KV need not be contiguous and two sequences may point at the same
slots.  "LOTUS": store_kv scatters each token's K/V to the slots it is handed;
passing the same slots again overwrites in place.  "Recurrent depth":
iteration t of layer l uses bank t*L + l.  vllm-rlt PR #152 (Summary, para 1)
with #147: prelude/coda layers write plane 0 only, recurrent layers every plane.

The pins build dense per-request K/V first and scatter them into the pool
with numpy fancy indexing (an independent route), then check that the
oracle's page-table walk brings back exactly the dense rows.
"""
import numpy as np
import pytest

import oracle
import workloads as W


def scatter_dense(dense, seq_lens, page_table, num_pages, ps):
    """Write dense [B][Lmax][Hkv][D] rows into a pool [P][Hkv][ps][D] through the page table."""
    B, Lmax, Hkv, D = dense.shape
    pool = np.zeros((num_pages, Hkv, ps, D), dense.dtype)
    for b in range(B):
        n = -(-int(seq_lens[b]) // ps)
        rows = np.zeros((n * ps, Hkv, D), dense.dtype)
        rows[: seq_lens[b]] = dense[b, : seq_lens[b]]
        pages = rows.reshape(n, ps, Hkv, D).transpose(0, 2, 1, 3)
        pages_in_use = page_table[b, :n]
        keep = np.arange(n * ps).reshape(n, ps) < seq_lens[b]
        for i, p in enumerate(pages_in_use):
            for o in range(ps):
                if keep[i, o]:
                    pool[p, :, o, :] = pages[i, :, o, :]
    return pool


def test_bank_map_fully_looped_is_t_times_L_plus_l():
    m, n = oracle.bank_map(np.ones(24, np.uint8), 4)
    assert n == 96
    for l in range(24):
        for t in range(4):
            assert m[l, t] == t * 24 + l


def test_bank_map_huginn_planes():
    rec = np.array([0, 0, 1, 1, 1, 1, 0, 0], np.uint8)
    m, n = oracle.bank_map(rec, 32)
    assert n == 8 + 31 * 4 == 132
    assert sorted(m[m >= 0].tolist()) == list(range(132))          # a bijection onto the banks
    assert np.all(m[:, 0] >= 0)                                      # plane 0 holds every layer
    assert np.all(m[[0, 1, 6, 7], 1:] == -1)                         # prelude/coda: plane 0 only
    assert np.all(m[2:6, :] >= 0)
    assert 32 * 8 / n == pytest.approx(256 / 132)
    # an unlooped model is a plain one: one plane, bank = layer
    m1, n1 = oracle.bank_map(np.zeros(5, np.uint8), 1)
    assert n1 == 5 and m1[:, 0].tolist() == list(range(5))


@pytest.mark.parametrize("ps", [1, 4, 16])
def test_gather_brings_back_dense_rows(ps):
    rng = np.random.default_rng(ps)
    seq_lens = np.array([1, ps, ps + 1, 3 * ps + 2, 0], np.int32)
    B, Hkv, D = len(seq_lens), 3, 8
    Lmax = int(seq_lens.max())
    n = [-(-int(L) // ps) for L in seq_lens]
    num_pages = sum(n) + 5
    perm = rng.permutation(num_pages)
    pt = np.full((B, max(n)), -1, np.int32)
    c = 0
    for b in range(B):
        pt[b, : n[b]] = perm[c: c + n[b]]
        c += n[b]
    dk = W.bf16_normal(rng, (B, Lmax, Hkv, D))
    dv = W.bf16_normal(rng, (B, Lmax, Hkv, D))
    kp = scatter_dense(dk, seq_lens, pt, num_pages, ps)
    vp = scatter_dense(dv, seq_lens, pt, num_pages, ps)
    gk, gv = oracle.paged_gather(kp, vp, pt, seq_lens)
    for b in range(B):
        L = seq_lens[b]
        assert np.array_equal(gk[b, :L], dk[b, :L])
        assert np.array_equal(gv[b, :L], dv[b, :L])
    # the slot of each position is the page the table names times ps plus the offset
    for b in range(B):
        for pos in range(seq_lens[b]):
            s = oracle.slot(pt, b, pos, ps)
            assert s // ps == pt[b, pos // ps] and s % ps == pos % ps


def test_gather_reads_shared_pages_for_every_request():
    case = W.config("huginn")
    ps = case.page_size
    assert case.unique_pages() < sum(case.pages_of(b) for b in range(case.batch))
    rng = np.random.default_rng(0)
    kp = W.bf16_normal(rng, (case.num_pages, 1, ps, 2))
    gk, _ = oracle.paged_gather(kp, kp, case.page_table, case.seq_lens)
    shared = int(np.floor(0.78 * case.pages_of(0)))
    for b in range(1, 4):
        s = min(shared, int(np.floor(0.78 * case.pages_of(b))))
        assert np.array_equal(gk[b, : s * ps], gk[0, : s * ps])


def test_append_writes_only_its_slots():
    rng = np.random.default_rng(9)
    P, Hkv, ps, D = 12, 2, 4, 8
    kp = W.bf16_normal(rng, (2, P, Hkv, ps, D))          # two banks
    vp = W.bf16_normal(rng, (2, P, Hkv, ps, D))
    k0, v0 = kp.copy(), vp.copy()
    loc = np.array([5, 46, -1, 0], np.int64)             # -1: no token this step
    kn = W.bf16_normal(rng, (4, Hkv, D))
    vn = W.bf16_normal(rng, (4, Hkv, D))
    oracle.kv_append(kp, vp, kn, vn, loc, bank=1)
    assert np.array_equal(kp[0], k0[0]) and np.array_equal(vp[0], v0[0])
    touched = np.zeros((P, ps), bool)
    for i, s in enumerate(loc):
        if s < 0:
            continue
        page, off = divmod(int(s), ps)
        touched[page, off] = True
        assert np.array_equal(kp[1, page, :, off, :], kn[i])
        assert np.array_equal(vp[1, page, :, off, :], vn[i])
    untouched = ~touched
    assert np.array_equal(kp[1].transpose(0, 2, 1, 3)[untouched], k0[1].transpose(0, 2, 1, 3)[untouched])
    assert np.array_equal(vp[1].transpose(0, 2, 1, 3)[untouched], v0[1].transpose(0, 2, 1, 3)[untouched])


def test_append_then_gather_sees_new_token_and_overwrite_in_place():
    case = W.config("tiny")
    h = W.host_tensors(case)
    kp, vp = h.k_pool.copy(), h.v_pool.copy()
    oracle.kv_append(kp, vp, h.k_new, h.v_new, case.new_slots)
    gk, gv = oracle.paged_gather(kp, vp, case.page_table, case.seq_lens)
    for b in range(case.batch):
        L = case.seq_lens[b]
        assert np.array_equal(gk[b, L - 1], h.k_new[b])
        assert np.array_equal(gv[b, L - 1], h.v_new[b])
    # LOTUS: the same slots again, new rows, overwrite in place
    rng = np.random.default_rng(11)
    k2 = W.bf16_normal(rng, h.k_new.shape)
    oracle.kv_append(kp, vp, k2, h.v_new, case.new_slots)
    gk2, _ = oracle.paged_gather(kp, vp, case.page_table, case.seq_lens)
    for b in range(case.batch):
        L = case.seq_lens[b]
        assert np.array_equal(gk2[b, L - 1], k2[b])
        assert np.array_equal(gk2[b, : L - 1], gk[b, : L - 1])
