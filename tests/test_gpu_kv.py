"""GPU parity of the KV append (store_kv) and the page-table gather: bit-exact.

"Faster fuzzy minds": store_kv scatters each token's K/V to the slots it is
handed (LOTUS overwrite-in-place = the same slots again); the pool is a flat
set of slots addressed through page_table[request, position].
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import bf16_dev, bits_host, i32_dev, i64_dev

pytestmark = pytest.mark.gpu


def device_pool(k_bits, v_bits, device):
    k = bf16_dev(k_bits, device)
    v = bf16_dev(v_bits, device)
    if k.dim() == 4:
        k, v = k[None].contiguous(), v[None].contiguous()
    return rlt.KVPool(k, v)


@pytest.mark.parametrize("name", ["tiny", "huginn"])
def test_append_matches_oracle_bit_exact(cuda_device, name):
    case = W.config(name)
    h = W.host_tensors(case)
    pool = device_pool(h.k_pool, h.v_pool, cuda_device)
    rlt.rlt_kv_append(pool, 0, bf16_dev(h.k_new, cuda_device), bf16_dev(h.v_new, cuda_device),
                      i64_dev(case.new_slots, cuda_device))
    kp, vp = h.k_pool.copy(), h.v_pool.copy()
    oracle.kv_append(kp, vp, h.k_new, h.v_new, case.new_slots)
    assert np.array_equal(bits_host(pool.k[0]), kp)
    assert np.array_equal(bits_host(pool.v[0]), vp)
    assert rlt.rlt_get_device_error() == 0


@pytest.mark.parametrize("ps", [1, 4, 16, 64])
@pytest.mark.parametrize("D", [64, 128])
def test_append_page_sizes_and_banks(cuda_device, ps, D):
    rng = np.random.default_rng(ps * D)
    banks, Hkv, N = 3, 3, 40
    P = 29 if ps >= 4 else 97                                     # at least 2N slots
    k0 = W.bf16_normal(rng, (banks, P, Hkv, ps, D))
    v0 = W.bf16_normal(rng, (banks, P, Hkv, ps, D))
    slots = rng.choice(P * ps, N, replace=False).astype(np.int64)
    slots[[3, 17]] = -1                                           # no token in these entries
    kn = W.bf16_normal(rng, (N, Hkv, D))
    vn = W.bf16_normal(rng, (N, Hkv, D))
    pool = device_pool(k0, v0, cuda_device)
    rlt.rlt_kv_append(pool, 2, bf16_dev(kn, cuda_device), bf16_dev(vn, cuda_device), i64_dev(slots, cuda_device))
    kp, vp = k0.copy(), v0.copy()
    oracle.kv_append(kp, vp, kn, vn, slots, bank=2)
    assert np.array_equal(bits_host(pool.k), kp) and np.array_equal(bits_host(pool.v), vp)
    # LOTUS: the same slots again overwrite in place
    kn2 = W.bf16_normal(rng, (N, Hkv, D))
    rlt.rlt_kv_append(pool, 2, bf16_dev(kn2, cuda_device), bf16_dev(vn, cuda_device), i64_dev(slots, cuda_device))
    oracle.kv_append(kp, vp, kn2, vn, slots, bank=2)
    assert np.array_equal(bits_host(pool.k), kp)


def test_append_out_of_range_slot_is_skipped_and_flagged(cuda_device):
    rng = np.random.default_rng(5)
    P, Hkv, ps, D = 8, 2, 16, 128
    k0 = W.bf16_normal(rng, (P, Hkv, ps, D))
    pool = device_pool(k0, k0, cuda_device)
    assert rlt.rlt_get_device_error() == 0
    slots = np.array([3, P * ps, 9], np.int64)                    # the middle one is past the pool
    kn = W.bf16_normal(rng, (3, Hkv, D))
    rlt.rlt_kv_append(pool, 0, bf16_dev(kn, cuda_device), bf16_dev(kn, cuda_device), i64_dev(slots, cuda_device))
    assert rlt.rlt_get_device_error() == rlt.DEVERR_BAD_SLOT
    kp = k0.copy()
    vp = k0.copy()
    oracle.kv_append(kp, vp, kn[[0, 2]], kn[[0, 2]], slots[[0, 2]])
    assert np.array_equal(bits_host(pool.k[0]), kp)
    assert rlt.rlt_get_device_error() == 0                        # reading cleared it


@pytest.mark.parametrize("name", ["tiny", "huginn", "longctx"])
def test_gather_matches_oracle_bit_exact(cuda_device, name):
    case = W.config(name)
    if name == "longctx":                       # keep the host pool small: 8 rows per page row
        case = W.custom(B=3, Hq=8, Hkv=2, D=128, ps=64, seq_lens=[1, 64 * 7 + 3, 2000], shared_frac=0.5)
    h = W.host_tensors(case)
    pool = device_pool(h.k_pool, h.v_pool, cuda_device)
    max_len = case.max_seq_len
    gk, gv = rlt.rlt_paged_gather(pool, 0, i32_dev(case.page_table, cuda_device),
                                  i32_dev(case.seq_lens, cuda_device), max_len)
    rk, rv = oracle.paged_gather(h.k_pool, h.v_pool, case.page_table, case.seq_lens, max_len=max_len)
    gk, gv = bits_host(gk), bits_host(gv)
    for b in range(case.batch):
        L = case.seq_lens[b]
        assert np.array_equal(gk[b, :L], rk[b, :L]) and np.array_equal(gv[b, :L], rv[b, :L])
    assert rlt.rlt_get_device_error() == 0


def test_gather_bad_page_is_skipped_and_flagged(cuda_device):
    case = W.config("tiny")
    h = W.host_tensors(case)
    pool = device_pool(h.k_pool, h.v_pool, cuda_device)
    b = int(np.argmax(case.seq_lens))                             # a request with >= 3 pages
    other = (b + 1) % case.batch
    pt = case.page_table.copy()
    pt[b, 2] = case.num_pages + 5
    gk, _ = rlt.rlt_paged_gather(pool, 0, i32_dev(pt, cuda_device), i32_dev(case.seq_lens, cuda_device),
                                 case.max_seq_len)
    assert rlt.rlt_get_device_error() == rlt.DEVERR_BAD_PAGE
    rk, _ = oracle.paged_gather(h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    gk = bits_host(gk)
    assert np.array_equal(gk[other, : case.seq_lens[other]], rk[other, : case.seq_lens[other]])
    assert np.array_equal(gk[b, :32], rk[b, :32])
