"""GPU parity of split-K paged GQA decode attention against the fp64 oracle.

"Faster fuzzy minds" ("When scheduler does the work", "Recurrent depth"):
one query per request attends over its cached tokens through the page table
of one (layer, plane) bank.  Bar: every bf16 output within 2e-2 absolute or
1e-2 relative of the oracle; lse within 1e-3.  Invariants that hold exactly on
the GPU (moving pages, shared vs private prefix pages) are checked bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import attn_close, bf16_dev, bits_host, i32_dev, i64_dev

pytestmark = pytest.mark.gpu


def dev_case(case, h, device):
    k = bf16_dev(h.k_pool, device)[None].contiguous()
    v = bf16_dev(h.v_pool, device)[None].contiguous()
    return (rlt.KVPool(k, v), bf16_dev(h.q, device), i32_dev(case.page_table, device),
            i32_dev(case.seq_lens, device))


def attend(pool, q, pt, sl, max_len, split_tokens=0, scale=0.0, bank=0):
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    out = rlt.rlt_paged_decode_attn(pool, bank, q, pt, sl, max_len, lse_out=lse, split_tokens=split_tokens,
                                     scale=scale)
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check(got, ref, lse=None, ref_lse=None):
    ok, mabs, mrel = attn_close(got, ref)
    assert ok, f"max abs {mabs:.3e} max rel {mrel:.3e}"
    if lse is not None:
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lse), fin)
        assert np.abs(lse[fin] - ref_lse[fin]).max(initial=0) <= 1e-3


def test_tiny_decode_step(cuda_device):
    # the whole step: append this step's token, then attend over all tokens
    case = W.config("tiny")
    h = W.host_tensors(case)
    pool, q, pt, sl = dev_case(case, h, cuda_device)
    rlt.rlt_kv_append(pool, 0, bf16_dev(h.k_new, cuda_device), bf16_dev(h.v_new, cuda_device),
                      i64_dev(case.new_slots, cuda_device))
    got, lse = attend(pool, q, pt, sl, case.max_seq_len)
    kp, vp = h.k_pool.copy(), h.v_pool.copy()
    oracle.kv_append(kp, vp, h.k_new, h.v_new, case.new_slots)
    ref, ref_lse = oracle.decode_attn(h.q, kp, vp, case.page_table, case.seq_lens)
    check(got, ref, lse, ref_lse)
    assert rlt.rlt_get_device_error() == 0


LENS = [1, 15, 16, 17, 63, 64, 65, 100, 255, 256, 257, 1000, 1531]


@pytest.mark.parametrize("G,D,ps", [(1, 128, 16), (2, 64, 16), (4, 128, 32), (8, 128, 64), (8, 64, 16),
                                    (1, 64, 128), (4, 64, 64), (2, 128, 16)])
@pytest.mark.parametrize("split_tokens", [0, 16, 64, 2048])
def test_shapes_ragged_lengths_and_splits(cuda_device, G, D, ps, split_tokens):
    Hkv = 2
    case = W.custom(B=len(LENS), Hq=G * Hkv, Hkv=Hkv, D=D, ps=ps, seq_lens=LENS, seed=G * 7 + D + ps)
    h = W.host_tensors(case)
    pool, q, pt, sl = dev_case(case, h, cuda_device)
    got, lse = attend(pool, q, pt, sl, case.max_seq_len, split_tokens=split_tokens)
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    check(got, ref, lse, ref_lse)
    assert rlt.rlt_get_device_error() == 0


def test_empty_and_single_token_requests(cuda_device):
    case = W.custom(B=5, Hq=4, Hkv=4, D=128, ps=16, seq_lens=[0, 1, 0, 2, 33])
    h = W.host_tensors(case)
    pool, q, pt, sl = dev_case(case, h, cuda_device)
    got, lse = attend(pool, q, pt, sl, 33, split_tokens=16)
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
    check(got, ref, lse, ref_lse)


def test_explicit_scale(cuda_device):
    case = W.custom(B=3, Hq=8, Hkv=2, D=64, ps=16, seq_lens=[40, 300, 7], seed=4)
    h = W.host_tensors(case)
    pool, q, pt, sl = dev_case(case, h, cuda_device)
    got, lse = attend(pool, q, pt, sl, 300, scale=0.3)
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens, scale=0.3)
    check(got, ref, lse, ref_lse)


def test_multi_bank_pool_reads_only_its_bank(cuda_device):
    case = W.custom(B=4, Hq=4, Hkv=4, D=128, ps=16, seq_lens=[70, 3, 129, 500], seed=8)
    h = W.host_tensors(case)
    other = W.bf16_normal(np.random.default_rng(1), h.k_pool.shape)
    k = bf16_dev(np.stack([other, other, h.k_pool]), cuda_device)
    v = bf16_dev(np.stack([other, h.v_pool, h.v_pool]), cuda_device)
    pool = rlt.KVPool(k, v)
    got, _ = attend(pool, bf16_dev(h.q, cuda_device), i32_dev(case.page_table, cuda_device),
                    i32_dev(case.seq_lens, cuda_device), 500, bank=2)
    ref, _ = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    check(got, ref)


def test_moving_pages_is_bit_exact(cuda_device):
    case = W.custom(B=6, Hq=16, Hkv=4, D=128, ps=16, seq_lens=[900, 17, 4000, 256, 1, 2500], seed=9)
    h = W.host_tensors(case)
    pool, q, pt, sl = dev_case(case, h, cuda_device)
    a, la = attend(pool, q, pt, sl, 4000)
    new_of_old = np.random.default_rng(3).permutation(case.num_pages)
    k2 = np.empty_like(h.k_pool)
    v2 = np.empty_like(h.v_pool)
    k2[new_of_old] = h.k_pool
    v2[new_of_old] = h.v_pool
    pt2 = np.where(case.page_table >= 0, new_of_old[np.maximum(case.page_table, 0)], -1).astype(np.int32)
    pool2 = rlt.KVPool(bf16_dev(k2, cuda_device)[None].contiguous(), bf16_dev(v2, cuda_device)[None].contiguous())
    b, lb = attend(pool2, q, i32_dev(pt2, cuda_device), sl, 4000)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_shared_prefix_pages_equal_private_copies_bit_exact(cuda_device):
    case = W.custom(B=4, Hq=8, Hkv=8, D=128, ps=16, seq_lens=[1200, 1100, 1300, 999], shared_frac=0.78, seed=10)
    h = W.host_tensors(case)
    pool, q, pt, sl = dev_case(case, h, cuda_device)
    a, la = attend(pool, q, pt, sl, 1300)
    # give every request private copies of the shared pages
    n = [case.pages_of(b) for b in range(case.batch)]
    total = sum(n)
    k2 = np.concatenate([h.k_pool, np.zeros((total,) + h.k_pool.shape[1:], np.uint16)])
    v2 = np.concatenate([h.v_pool, np.zeros((total,) + h.v_pool.shape[1:], np.uint16)])
    pt2 = case.page_table.copy()
    nxt = case.num_pages
    for b in range(case.batch):
        for i in range(n[b]):
            k2[nxt] = h.k_pool[pt2[b, i]]
            v2[nxt] = h.v_pool[pt2[b, i]]
            pt2[b, i] = nxt
            nxt += 1
    assert len(np.unique(pt2[pt2 >= 0])) == total
    pool2 = rlt.KVPool(bf16_dev(k2, cuda_device)[None].contiguous(), bf16_dev(v2, cuda_device)[None].contiguous())
    b_, lb = attend(pool2, q, i32_dev(pt2, cuda_device), sl, 1300)
    assert np.array_equal(a, b_) and np.array_equal(la, lb)


def test_gqa_equals_mha_with_repeated_kv_heads(cuda_device):
    G = 4
    case = W.custom(B=3, Hq=8, Hkv=2, D=128, ps=16, seq_lens=[333, 17, 1024], seed=12)
    h = W.host_tensors(case)
    pool, q, pt, sl = dev_case(case, h, cuda_device)
    a, _ = attend(pool, q, pt, sl, 1024)
    kr = np.repeat(h.k_pool, G, axis=1)
    vr = np.repeat(h.v_pool, G, axis=1)
    pool_m = rlt.KVPool(bf16_dev(kr, cuda_device)[None].contiguous(), bf16_dev(vr, cuda_device)[None].contiguous())
    b, _ = attend(pool_m, q, pt, sl, 1024)
    assert np.array_equal(a, b)


def test_split_count_independence(cuda_device):
    case = W.custom(B=5, Hq=8, Hkv=8, D=128, ps=16, seq_lens=[3000, 2048, 777, 16, 4096], seed=13)
    h = W.host_tensors(case)
    pool, q, pt, sl = dev_case(case, h, cuda_device)
    outs = [attend(pool, q, pt, sl, 4096, split_tokens=s) for s in (16, 128, 512, 2048)]
    for o, l in outs[1:]:
        assert np.abs(o - outs[0][0]).max() <= 2 ** -7 * np.abs(outs[0][0]).max() + 1e-6
        assert np.abs(l - outs[0][1]).max() <= 1e-4


def test_bad_page_is_skipped_and_flagged(cuda_device):
    case = W.custom(B=3, Hq=4, Hkv=4, D=128, ps=16, seq_lens=[100, 300, 64], seed=14)
    h = W.host_tensors(case)
    pool, q, _, sl = dev_case(case, h, cuda_device)
    assert rlt.rlt_get_device_error() == 0
    pt = case.page_table.copy()
    pt[1, 3] = case.num_pages + 100
    pt[2, 0] = -7
    got, _ = attend(pool, q, i32_dev(pt, cuda_device), sl, 300, split_tokens=64)
    assert rlt.rlt_get_device_error() & rlt.DEVERR_BAD_PAGE
    ref, _ = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    check(got[0], ref[0])                                 # other requests unaffected


def test_overlong_seq_len_is_clamped_and_flagged(cuda_device):
    case = W.custom(B=2, Hq=4, Hkv=4, D=128, ps=16, seq_lens=[50, 64], seed=15)
    h = W.host_tensors(case)
    pool, q, pt, _ = dev_case(case, h, cuda_device)
    sl = i32_dev(np.array([50, 10_000], np.int32), cuda_device)     # row 1 holds 4 pages only
    attend(pool, q, pt, sl, 64)
    assert rlt.rlt_get_device_error() & rlt.DEVERR_BAD_LEN


# ------------------------------------------------ full-size workloads, sampled

def full_size(name, device, rows):
    case = W.config(name)
    kd, vd = W.device_pool(case, 1, device)
    pool = rlt.KVPool(kd, vd)
    rng = np.random.default_rng(case.seed + 5)
    q_bits = W.bf16_normal(rng, (case.batch, case.num_q_heads, case.head_dim))
    q = bf16_dev(q_bits, device)
    pt = i32_dev(case.page_table, device)
    sl = i32_dev(case.seq_lens, device)
    got, lse = attend(pool, q, pt, sl, case.max_seq_len)       # the launch plan the bench times
    assert rlt.rlt_get_device_error() == 0
    kh, vh = bits_host(kd[0]), bits_host(vd[0])
    del kd, vd, pool
    ref, ref_lse = oracle.decode_attn_rows(q_bits, kh, vh, case.page_table, case.seq_lens, rows)
    check(got[rows], ref, lse[rows], ref_lse)


@pytest.mark.parametrize("name,rows", [
    ("ouro", [0, 17, 33, 63]),
    ("huginn", list(range(16))),
    ("gqa", None),
    ("longctx", [0, 5]),
])
def test_full_size_workloads_sampled(cuda_device, name, rows):
    # every sample includes the workload's longest request (the deepest split, the largest
    # combine fan-in) and its shortest
    L = W.config(name).seq_lens
    rows = set(rows) if rows is not None else {1, 128}
    rows |= {int(np.argmax(L)), int(np.argmin(L))}
    full_size(name, cuda_device, np.array(sorted(rows)))


def test_many_rows_warp_merge(cuda_device):
    # >= 2048 (request, query head) rows with a few splits each: the combine takes a warp per
    # row; ragged lengths with empty, one-split and several-split requests
    rng = np.random.default_rng(71)
    lens = rng.integers(1, 700, size=136)
    lens[[0, 5, 77]] = 0
    lens[[1, 9]] = [16, 33]
    case = W.custom(B=len(lens), Hq=16, Hkv=4, D=128, ps=16, seq_lens=lens.tolist(), seed=72)
    h = W.host_tensors(case)
    pool, q, pt, sl = dev_case(case, h, cuda_device)
    got, lse = attend(pool, q, pt, sl, case.max_seq_len, split_tokens=64)
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    assert np.all(got[lens == 0] == 0) and np.all(np.isneginf(lse[lens == 0]))
    check(got, ref, lse, ref_lse)
    assert rlt.rlt_get_device_error() == 0
