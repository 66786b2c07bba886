"""GPU parity of the append fused into decode attention.

"Faster fuzzy minds" ("When scheduler does the work"): in a decode step each
layer stores the new token's K/V in its slot (store_kv) and then attends over
every cached token, the new one included.  With k_new / v_new the attention
call does both: the split-K CTA reading the tile of position seq_lens[b] - 1
takes that row from k_new / v_new and writes it to the pool (for a private
tail on tensor cores, the producer lane copying that row writes it to the pool
just before its copy).  Checked against
the oracle's two steps (kv_append at the slot the page table gives position
L - 1, then decode attention over the updated pool): the pool bit for bit,
the output within the attention bar, lse within 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import attn_close, bf16_dev, bits_host, i32_dev

pytestmark = pytest.mark.gpu

# newest positions on row 0, row 15 and the rows between of a 16-token tile, one token,
# an empty request, and lengths spanning several splits
LENS = [1, 16, 17, 31, 0, 129, 500, 2048, 2049, 3001]


def oracle_step(case, h, kn, vn):
    """kv_append at each request's newest slot, then decode attention (both fp64 oracle)."""
    slots = np.array([oracle.slot(case.page_table, b, int(L) - 1, case.page_size) if L > 0 else -1
                      for b, L in enumerate(case.seq_lens)], np.int64)
    kp, vp = h.k_pool.copy(), h.v_pool.copy()
    oracle.kv_append(kp, vp, kn, vn, slots)
    ref, ref_lse = oracle.decode_attn(h.q, kp, vp, case.page_table, case.seq_lens)
    return kp, vp, ref, ref_lse


def new_rows(case, seed):
    rng = np.random.default_rng(seed)
    shape = (case.batch, case.num_kv_heads, case.head_dim)
    return W.bf16_normal(rng, shape), W.bf16_normal(rng, shape)


def check(got, ref, lse, ref_lse):
    ok, mabs, mrel = attn_close(got, ref)
    assert ok, f"max abs {mabs:.3e} max rel {mrel:.3e}"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.abs(lse[fin] - ref_lse[fin]).max(initial=0.0) <= 1e-3


@pytest.mark.parametrize("G,D,ps", [(1, 128, 16), (2, 64, 16), (4, 128, 32), (8, 128, 64), (1, 64, 128),
                                    (2, 128, 256)])
@pytest.mark.parametrize("split_tokens", [0, 16, 64, 2048])
def test_plain_fused_append(cuda_device, G, D, ps, split_tokens):
    Hkv = 2
    case = W.custom(B=len(LENS), Hq=G * Hkv, Hkv=Hkv, D=D, ps=ps, seq_lens=LENS, seed=G * 5 + D + ps)
    h = W.host_tensors(case)
    kn, vn = new_rows(case, 3 + G)
    k, v = bf16_dev(h.k_pool, cuda_device)[None].contiguous(), bf16_dev(h.v_pool, cuda_device)[None].contiguous()
    pool = rlt.KVPool(k, v)
    q = bf16_dev(h.q, cuda_device)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=cuda_device)
    out = rlt.rlt_paged_decode_attn(pool, 0, q, i32_dev(case.page_table, cuda_device),
                                    i32_dev(case.seq_lens, cuda_device), case.max_seq_len, lse_out=lse,
                                    split_tokens=split_tokens, k_new=bf16_dev(kn, cuda_device),
                                    v_new=bf16_dev(vn, cuda_device))
    assert rlt.rlt_get_device_error() == 0
    kp, vp, ref, ref_lse = oracle_step(case, h, kn, vn)
    assert np.array_equal(bits_host(k[0]), kp) and np.array_equal(bits_host(v[0]), vp)
    check(out.float().cpu().numpy(), ref, lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("tails", [False, True])
@pytest.mark.parametrize("G,ps", [(1, 16), (4, 16), (8, 16), (2, 64), (1, 256)])
def test_prefix_fused_append(cuda_device, tails, G, ps):
    # a shared prompt chain (tensor-core segments) and private rests; with private tails the
    # tensor-core kernel stores the new rows (its producer lanes, before their copies)
    Hkv = 2
    lens = [3000, 2900, 3100, 1500, 700, 2333, 2048, 257]
    case = W.custom(B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=128, ps=ps, seq_lens=lens, shared_frac=0.8, seed=30 + G + ps)
    h = W.host_tensors(case)
    kn, vn = new_rows(case, 40 + G)
    k, v = bf16_dev(h.k_pool, cuda_device)[None].contiguous(), bf16_dev(h.v_pool, cuda_device)[None].contiguous()
    pool = rlt.KVPool(k, v)
    q = bf16_dev(h.q, cuda_device)
    plan = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, 2, tails, G).to(cuda_device)
    assert plan.num_segments > 0
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=cuda_device)
    out = rlt.rlt_paged_decode_attn_prefix(pool, 0, q, i32_dev(case.page_table, cuda_device),
                                           i32_dev(case.seq_lens, cuda_device), case.max_seq_len, plan,
                                           lse_out=lse, k_new=bf16_dev(kn, cuda_device),
                                           v_new=bf16_dev(vn, cuda_device))
    assert rlt.rlt_get_device_error() == 0
    kp, vp, ref, ref_lse = oracle_step(case, h, kn, vn)
    assert np.array_equal(bits_host(k[0]), kp) and np.array_equal(bits_host(v[0]), vp)
    check(out.float().cpu().numpy(), ref, lse.cpu().numpy(), ref_lse)


def test_fused_equals_append_then_attention_bit_exact(cuda_device):
    # the same kernels with the row taken from k_new instead of the pool: identical bits
    case = W.custom(B=6, Hq=8, Hkv=2, D=128, ps=16, seq_lens=[900, 17, 4000, 256, 1, 2500], seed=12)
    h = W.host_tensors(case)
    kn, vn = new_rows(case, 13)
    pt, sl = i32_dev(case.page_table, cuda_device), i32_dev(case.seq_lens, cuda_device)
    q = bf16_dev(h.q, cuda_device)
    outs = []
    for fused in (False, True):
        k, v = bf16_dev(h.k_pool, cuda_device)[None].contiguous(), bf16_dev(h.v_pool, cuda_device)[None].contiguous()
        pool = rlt.KVPool(k, v)
        kd, vd = bf16_dev(kn, cuda_device), bf16_dev(vn, cuda_device)
        if fused:
            out = rlt.rlt_paged_decode_attn(pool, 0, q, pt, sl, case.max_seq_len, k_new=kd, v_new=vd)
        else:
            loc = torch.from_numpy(case.new_slots.copy()).to(cuda_device)
            rlt.rlt_kv_append(pool, 0, kd, vd, loc)
            out = rlt.rlt_paged_decode_attn(pool, 0, q, pt, sl, case.max_seq_len)
        outs.append((out.view(torch.int16).cpu(), bits_host(k[0]), bits_host(v[0])))
    assert rlt.rlt_get_device_error() == 0
    assert torch.equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1]) and np.array_equal(outs[0][2], outs[1][2])


@pytest.mark.parametrize("tails", [False, True])
def test_newest_token_inside_a_shared_prefix_is_flagged_not_written(cuda_device, tails):
    # requests 0 and 1 map the same two pages for 128 tokens: request 0's newest token
    # (position 127) lies in a tile the plan shares, so its slot is a shared page's; the
    # others' rows are written by the split-K kernel (or, with private tails, by the
    # tensor-core kernel)
    ps = 64
    case = W.custom(B=3, Hq=2, Hkv=2, D=128, ps=ps, seq_lens=[128, 600, 300], seed=17)
    pt = case.page_table.copy()
    pt[1, :2] = pt[0, :2]
    h = W.host_tensors(case)
    kn, vn = new_rows(case, 18)
    k, v = bf16_dev(h.k_pool, cuda_device)[None].contiguous(), bf16_dev(h.v_pool, cuda_device)[None].contiguous()
    pool = rlt.KVPool(k, v)
    plan = rlt.rlt_plan_prefix(pt, case.seq_lens, ps, 1, tails, 1).to(cuda_device)
    assert plan.num_segments > 0 and (plan.max_rest_len == 0) == tails
    rlt.rlt_get_device_error()
    rlt.rlt_paged_decode_attn_prefix(pool, 0, bf16_dev(h.q, cuda_device), i32_dev(pt, cuda_device),
                                     i32_dev(case.seq_lens, cuda_device), case.max_seq_len, plan,
                                     k_new=bf16_dev(kn, cuda_device), v_new=bf16_dev(vn, cuda_device))
    assert rlt.rlt_get_device_error() & rlt.DEVERR_BAD_SLOT
    kp, vp = h.k_pool.copy(), h.v_pool.copy()
    slots = np.array([-1] + [oracle.slot(pt, b, int(case.seq_lens[b]) - 1, ps) for b in (1, 2)], np.int64)
    oracle.kv_append(kp, vp, kn, vn, slots)                  # requests 1 and 2 appended, 0 not
    assert np.array_equal(bits_host(k[0]), kp) and np.array_equal(bits_host(v[0]), vp)


def test_clamped_length_gets_no_append(cuda_device):
    case = W.custom(B=2, Hq=4, Hkv=4, D=128, ps=16, seq_lens=[50, 64], seed=15)
    h = W.host_tensors(case)
    kn, vn = new_rows(case, 16)
    k, v = bf16_dev(h.k_pool, cuda_device)[None].contiguous(), bf16_dev(h.v_pool, cuda_device)[None].contiguous()
    pool = rlt.KVPool(k, v)
    sl = i32_dev(np.array([50, 10_000], np.int32), cuda_device)     # row 1 holds 4 pages only
    rlt.rlt_get_device_error()
    rlt.rlt_paged_decode_attn(pool, 0, bf16_dev(h.q, cuda_device), i32_dev(case.page_table, cuda_device), sl, 64,
                              k_new=bf16_dev(kn, cuda_device), v_new=bf16_dev(vn, cuda_device))
    assert rlt.rlt_get_device_error() & rlt.DEVERR_BAD_LEN
    kp, vp = h.k_pool.copy(), h.v_pool.copy()
    oracle.kv_append(kp, vp, kn, vn, np.array([case.new_slots[0], -1], np.int64))
    assert np.array_equal(bits_host(k[0]), kp) and np.array_equal(bits_host(v[0]), vp)


@pytest.mark.parametrize("name,rows", [("ouro", [0, 17, 33, 63]), ("huginn", list(range(16))), ("gqa", None),
                                       ("longctx", [0, 3, 7]), ("tiny", [0, 1, 2, 3])])
def test_full_size_fused_sampled(cuda_device, name, rows):
    # every workload at full size in the launch configuration bench.py times by default: the
    # append fused into the call, the shared-prefix plan with the bench's private-tails rule and
    # work-item size, split-K sized by the library
    import bench
    case = W.config(name)
    kd, vd = W.device_pool(case, 1, cuda_device)
    pool = rlt.KVPool(kd, vd)
    kh0, vh0 = bits_host(kd[0]), bits_host(vd[0])
    rng = np.random.default_rng(case.seed + 5)
    q_bits = W.bf16_normal(rng, (case.batch, case.num_q_heads, case.head_dim))
    kn, vn = new_rows(case, case.seed + 6)
    pt, sl = i32_dev(case.page_table, cuda_device), i32_dev(case.seq_lens, cuda_device)
    q = bf16_dev(q_bits, cuda_device)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=cuda_device)
    tails = case.group >= 8
    shared = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, 1, False, case.group)
    kw = dict(lse_out=lse, k_new=bf16_dev(kn, cuda_device), v_new=bf16_dev(vn, cuda_device))
    if shared.num_segments:
        sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
        chunk = bench.auto_chunk_tiles(rlt, case, tails, sms)
        plan = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, chunk, tails, case.group)
        out = rlt.rlt_paged_decode_attn_prefix(pool, 0, q, pt, sl, case.max_seq_len, plan.to(cuda_device), **kw)
    else:
        out = rlt.rlt_paged_decode_attn(pool, 0, q, pt, sl, case.max_seq_len, **kw)
    assert rlt.rlt_get_device_error() == 0
    kh, vh = bits_host(kd[0]), bits_host(vd[0])
    del kd, vd, pool
    oracle.kv_append(kh0, vh0, kn, vn, case.new_slots)
    assert np.array_equal(kh, kh0) and np.array_equal(vh, vh0)
    # the sample always holds the longest request (deepest split, largest combine fan-in) and the
    # shortest
    rows = set(rows) if rows is not None else {1, 128}
    rows = np.array(sorted(rows | {int(np.argmax(case.seq_lens)), int(np.argmin(case.seq_lens))}))
    ref, ref_lse = oracle.decode_attn_rows(q_bits, kh, vh, case.page_table, case.seq_lens, rows)
    check(out.float().cpu().numpy()[rows], ref, lse.cpu().numpy()[rows], ref_lse)
