"""GPU parity of causal extend (span) attention on tcgen05 against the fp64 oracle.

"Faster fuzzy minds", LOTUS: a block of positions is re-forwarded several times
in place, every pass attending over the whole block at once after its
K/V were written back to the same slots; packed prefill is the same call over a
whole prompt.  Bar: the attention tolerance (2e-2 abs or 1e-2 rel), lse within
1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import attn_close, bf16_dev, i32_dev, i64_dev

pytestmark = pytest.mark.gpu


def run_extend(case, h, q, new, device, chunk_tiles=2, max_ctas=0, k_pool=None, v_pool=None):
    kp = h.k_pool if k_pool is None else k_pool
    vp = h.v_pool if v_pool is None else v_pool
    pool = rlt.KVPool(bf16_dev(kp, device)[None].contiguous(), bf16_dev(vp, device)[None].contiguous())
    plan = rlt.rlt_plan_extend(case.seq_lens, new, case.page_size, chunk_tiles, case.group).to(device)
    qd = bf16_dev(q, device)
    lse = torch.empty(qd.shape[:2], dtype=torch.float32, device=device)
    out = rlt.rlt_paged_extend_attn(pool, 0, qd, i32_dev(case.page_table, device), plan, lse_out=lse,
                                    max_ctas=max_ctas)
    assert rlt.rlt_get_device_error() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check(got, ref, lse, ref_lse):
    ok, mabs, mrel = attn_close(got, ref)
    assert ok, f"max abs {mabs:.3e} max rel {mrel:.3e}"
    assert np.abs(lse - ref_lse).max() <= 1e-3


@pytest.mark.parametrize("G,ps,chunk_tiles,max_ctas", [(1, 16, 2, 0), (2, 32, 1, 3), (4, 64, 3, 0), (8, 16, 2, 1),
                                                       (8, 128, 1, 0), (1, 256, 2, 5)])
def test_extend_matches_oracle(cuda_device, G, ps, chunk_tiles, max_ctas):
    rng = np.random.default_rng(G * 7 + ps)
    lens = [300, 50, 1000, 128, 129, 7, 2000, 640]
    new = [40, 50, 0, 128, 1, 7, 300, 17]
    case = W.custom(B=len(lens), Hq=2 * G, Hkv=2, D=128, ps=ps, seq_lens=lens, seed=G + ps)
    h = W.host_tensors(case)
    q = W.bf16_normal(rng, (sum(new), 2 * G, 128))
    got, lse = run_extend(case, h, q, new, cuda_device, chunk_tiles, max_ctas)
    ref, ref_lse = oracle.extend_attn(q, h.k_pool, h.v_pool, case.page_table, case.seq_lens, new)
    check(got, ref, lse, ref_lse)


def test_whole_prompt_prefill_and_nan_padding(cuda_device):
    # every token new (packed prefill); page memory past each request's end holds NaN
    lens = [1, 64, 65, 333, 1024]
    case = W.custom(B=len(lens), Hq=8, Hkv=1, D=128, ps=64, seq_lens=lens, seed=11)
    h = W.host_tensors(case)
    kp, vp = h.k_pool.copy(), h.v_pool.copy()
    for b, L in enumerate(lens):
        n = -(-L // 64)
        last = case.page_table[b, n - 1]
        kp[last, :, L - (n - 1) * 64:, :] = 0x7FC0
        vp[last, :, L - (n - 1) * 64:, :] = 0x7FC0
    q = W.bf16_normal(np.random.default_rng(12), (sum(lens), 8, 128))
    got, lse = run_extend(case, h, q, lens, cuda_device, 1, k_pool=kp, v_pool=vp)
    ref, ref_lse = oracle.extend_attn(q, kp, vp, case.page_table, case.seq_lens, lens)
    assert np.all(np.isfinite(got))
    check(got, ref, lse, ref_lse)


def test_lotus_block_reforwarded_in_place(cuda_device):
    # a block of 48 latent positions after each prompt, re-forwarded 3 times: each pass
    # writes the block's K/V to the same slots (store_kv) and attends over prompt + block
    block, G = 48, 4
    prompts = [500, 1200, 77]
    lens = [p + block for p in prompts]
    case = W.custom(B=len(lens), Hq=4 * G, Hkv=4, D=128, ps=16, seq_lens=lens, seed=21)
    h = W.host_tensors(case)
    rng = np.random.default_rng(22)
    slots = np.concatenate([[oracle.slot(case.page_table, b, p, case.page_size) for p in range(prompts[b], lens[b])]
                            for b in range(len(lens))]).astype(np.int64)
    pool = rlt.KVPool(bf16_dev(h.k_pool, cuda_device)[None].contiguous(),
                      bf16_dev(h.v_pool, cuda_device)[None].contiguous())
    kp, vp = h.k_pool.copy(), h.v_pool.copy()
    plan = rlt.rlt_plan_extend(case.seq_lens, [block] * len(lens), case.page_size, 2, G).to(cuda_device)
    pt = i32_dev(case.page_table, cuda_device)
    for _ in range(3):
        kn = W.bf16_normal(rng, (len(slots), 4, 128))
        vn = W.bf16_normal(rng, (len(slots), 4, 128))
        q = W.bf16_normal(rng, (len(slots), 4 * G, 128))
        rlt.rlt_kv_append(pool, 0, bf16_dev(kn, cuda_device), bf16_dev(vn, cuda_device), i64_dev(slots, cuda_device))
        lse = torch.empty((len(slots), 4 * G), dtype=torch.float32, device=cuda_device)
        out = rlt.rlt_paged_extend_attn(pool, 0, bf16_dev(q, cuda_device), pt, plan, lse_out=lse)
        assert rlt.rlt_get_device_error() == 0
        oracle.kv_append(kp, vp, kn, vn, slots)
        ref, ref_lse = oracle.extend_attn(q, kp, vp, case.page_table, case.seq_lens, [block] * len(lens))
        check(out.float().cpu().numpy(), ref, lse.cpu().numpy(), ref_lse)
