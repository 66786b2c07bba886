"""GPU parity of shared-prefix (cascade) decode attention against the fp64 oracle.

The cascade path computes the same softmax(q K^T / sqrt(d)) V as plain paged
decode ("Faster fuzzy minds", "When scheduler does the work"); it only reads
each shared 128-token tile once per kv head, with tcgen05 tensor-core MMAs over
all members' queries.  Bar: the attention tolerance (2e-2 abs or 1e-2 rel)
against the oracle, lse within 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import attn_close, bf16_dev, bits_host, i32_dev

pytestmark = pytest.mark.gpu


def run_both(case, h, device, chunk_tiles=4, split_tokens=0, private_tails=False, max_ctas=0):
    pool = rlt.KVPool(bf16_dev(h.k_pool, device)[None].contiguous(), bf16_dev(h.v_pool, device)[None].contiguous())
    q = bf16_dev(h.q, device)
    pt = i32_dev(case.page_table, device)
    sl = i32_dev(case.seq_lens, device)
    plan = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, chunk_tiles,
                               private_tails, case.group).to(device)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=device)
    out = rlt.rlt_paged_decode_attn_prefix(pool, 0, q, pt, sl, case.max_seq_len, plan, lse_out=lse,
                                           split_tokens=split_tokens, max_ctas=max_ctas)
    lse_p = torch.empty_like(lse)
    plain = rlt.rlt_paged_decode_attn(pool, 0, q, pt, sl, case.max_seq_len, lse_out=lse_p)
    assert rlt.rlt_get_device_error() == 0
    return plan, out.float().cpu().numpy(), lse.cpu().numpy(), plain.float().cpu().numpy(), lse_p.cpu().numpy()


def check(got, ref, lse=None, ref_lse=None):
    ok, mabs, mrel = attn_close(got, ref)
    assert ok, f"max abs {mabs:.3e} max rel {mrel:.3e}"
    if lse is not None:
        assert np.abs(lse - ref_lse).max() <= 1e-3


def test_huginn_full_size(cuda_device):
    case = W.config("huginn")
    h = W.host_tensors(case)
    plan, got, lse, plain, _ = run_both(case, h, cuda_device)
    assert plan.num_segments > 0
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    check(got, ref, lse, ref_lse)
    check(plain, ref)


@pytest.mark.parametrize("G,ps,members", [(1, 16, 5), (2, 32, 9), (4, 64, 20), (8, 16, 8), (8, 128, 20),
                                           (1, 256, 3), (8, 64, 33)])
def test_groups_page_sizes_and_member_blocks(cuda_device, G, ps, members):
    # members x G query rows; more than 128 rows takes several member blocks
    Hkv = 2
    rng = np.random.default_rng(G * 100 + ps + members)
    lens = rng.integers(700, 2600, size=members)
    case = W.custom(B=members, Hq=G * Hkv, Hkv=Hkv, D=128, ps=ps, seq_lens=lens, shared_frac=0.8,
                    seed=G + ps + members)
    h = W.host_tensors(case)
    plan, got, lse, plain, plain_lse = run_both(case, h, cuda_device, chunk_tiles=2)
    assert plan.num_segments > 0
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    check(got, ref, lse, ref_lse)
    check(plain, ref, plain_lse, ref_lse)


@pytest.mark.parametrize("chunk_tiles,split_tokens", [(1, 16), (3, 0), (32, 2048)])
def test_chunk_and_split_settings(cuda_device, chunk_tiles, split_tokens):
    case = W.custom(B=6, Hq=16, Hkv=4, D=128, ps=16, seq_lens=[4000, 3900, 4100, 2500, 700, 3333],
                    shared_frac=0.9, seed=chunk_tiles)
    h = W.host_tensors(case)
    _, got, lse, _, _ = run_both(case, h, cuda_device, chunk_tiles, split_tokens)
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    check(got, ref, lse, ref_lse)


def test_no_sharing_falls_back_to_plain(cuda_device):
    case = W.custom(B=4, Hq=8, Hkv=8, D=128, ps=16, seq_lens=[500, 300, 1200, 17], seed=5)
    h = W.host_tensors(case)
    plan, got, _, plain, _ = run_both(case, h, cuda_device)
    assert plan.num_segments == 0
    assert np.array_equal(got, plain)


def test_shared_and_private_requests_mixed_with_empty(cuda_device):
    # requests 0..3 share, 4 and 5 are alone, 6 is empty
    rng = np.random.default_rng(9)
    ps = 16
    lens = [1500, 1700, 1600, 1555, 900, 2100, 0]
    P = 1500
    perm = iter(rng.permutation(P))
    pt = np.full((len(lens), -(-max(lens) // ps)), -1, np.int32)
    shared = [next(perm) for _ in range(64)]
    for r, L in enumerate(lens):
        n = -(-L // ps)
        k = min(64, n - 1) if r < 4 else 0
        pt[r, :k] = shared[:k]
        pt[r, k:n] = [next(perm) for _ in range(n - k)]
    case = W.PagedCase(name="mixed", num_layers=1, num_planes=1, recurrent=np.zeros(1, np.uint8), batch=len(lens),
                       num_q_heads=4, num_kv_heads=4, head_dim=128, page_size=ps, num_pages=P,
                       seq_lens=np.array(lens, np.int32), page_table=pt, new_slots=np.zeros(len(lens), np.int64))
    h = W.host_tensors(case)
    plan, got, lse, _, _ = run_both(case, h, cuda_device)
    assert plan.num_segments == 1 and plan.request_prefix[4, 0] == 0
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    assert np.all(got[6] == 0) and np.all(np.isneginf(lse[6]))
    check(got[:6], ref[:6], lse[:6], ref_lse[:6])


@pytest.mark.parametrize("chunk_tiles,tails", [(8, False), (6, True)])   # (6, private tails): the bench's launch
def test_longctx_full_size_sampled(cuda_device, chunk_tiles, tails):
    case = W.config("longctx")
    kd, vd = W.device_pool(case, 1, cuda_device)
    pool = rlt.KVPool(kd, vd)
    rng = np.random.default_rng(case.seed + 5)
    q_bits = W.bf16_normal(rng, (case.batch, case.num_q_heads, case.head_dim))
    q = bf16_dev(q_bits, cuda_device)
    pt = i32_dev(case.page_table, cuda_device)
    sl = i32_dev(case.seq_lens, cuda_device)
    plan = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, chunk_tiles, tails,
                               case.group).to(cuda_device)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=cuda_device)
    got = rlt.rlt_paged_decode_attn_prefix(pool, 0, q, pt, sl, case.max_seq_len, plan, lse_out=lse)
    got = got.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert rlt.rlt_get_device_error() == 0
    rows = np.array([0, 3, 7])
    ref, ref_lse = oracle.decode_attn_rows(q_bits, bits_host(kd[0]), bits_host(vd[0]), case.page_table,
                                           case.seq_lens, rows)
    check(got[rows], ref, lse[rows], ref_lse)


@pytest.mark.parametrize("G,ps,shared_frac", [(8, 64, 0.9), (8, 16, 0.0), (4, 16, 0.5), (2, 32, 0.8), (1, 128, 0.7)])
def test_private_tails_on_tensor_cores(cuda_device, G, ps, shared_frac):
    # every token through the tcgen05 kernel, ragged ends of all kinds (1, 63, 64, 65, 127, 129 ... tokens)
    lens = [1, 63, 64, 65, 127, 128, 129, 1000, 3001, 4096, 2222, 777]
    case = W.custom(B=len(lens), Hq=G * 2, Hkv=2, D=128, ps=ps, seq_lens=lens, shared_frac=shared_frac,
                    seed=G + ps)
    h = W.host_tensors(case)
    plan, got, lse, _, _ = run_both(case, h, cuda_device, chunk_tiles=2, private_tails=True)
    assert plan.max_rest_len == 0 and plan.num_segments >= len(lens)
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    check(got, ref, lse, ref_lse)


def test_private_tails_with_empty_and_nan_padding(cuda_device):
    # page memory past each request's end holds NaN: the masked tail must not leak it
    lens = [0, 5, 70, 200, 0, 1300]
    case = W.custom(B=len(lens), Hq=16, Hkv=2, D=128, ps=64, seq_lens=lens, seed=3)
    h = W.host_tensors(case)
    kp, vp = h.k_pool.copy(), h.v_pool.copy()
    for b, L in enumerate(lens):
        n = -(-L // 64)
        if n:
            last = case.page_table[b, n - 1]
            kp[last, :, L - (n - 1) * 64:, :] = 0x7FC0          # bf16 quiet NaN
            vp[last, :, L - (n - 1) * 64:, :] = 0x7FC0
    h = W.HostTensors(kp, vp, h.q, h.k_new, h.v_new)
    plan, got, lse, _, _ = run_both(case, h, cuda_device, private_tails=True)
    ref, ref_lse = oracle.decode_attn(h.q, kp, vp, case.page_table, case.seq_lens)
    assert np.all(got[0] == 0) and np.all(got[4] == 0)
    assert np.all(np.isfinite(got))
    check(got[[1, 2, 3, 5]], ref[[1, 2, 3, 5]], lse[[1, 2, 3, 5]], ref_lse[[1, 2, 3, 5]])


@pytest.mark.parametrize("max_ctas", [1, 2, 7])
@pytest.mark.parametrize("tails,chunk_tiles", [(False, 1), (True, 1), (True, 3)])
def test_persistent_ctas_with_many_runs(cuda_device, max_ctas, tails, chunk_tiles):
    # few CTAs: each walks many runs (kv heads, segments, member blocks, merged chunks) through one
    # pipeline, reusing its Q, O, S, P buffers and K/V rings across runs
    lens = [2900, 3100, 1500, 700, 2333, 129, 128, 4000, 3999]
    case = W.custom(B=len(lens), Hq=4, Hkv=2, D=128, ps=16, seq_lens=lens, shared_frac=0.8, seed=max_ctas)
    h = W.host_tensors(case)
    plan, got, lse, _, _ = run_both(case, h, cuda_device, chunk_tiles, private_tails=tails, max_ctas=max_ctas)
    assert plan.num_segments > 0
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    check(got, ref, lse, ref_lse)


def test_huginn_full_size_all_tensor_core_few_ctas(cuda_device):
    case = W.config("huginn")
    h = W.host_tensors(case)
    plan, got, lse, _, _ = run_both(case, h, cuda_device, 1, private_tails=True, max_ctas=5)
    assert plan.max_rest_len == 0
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    check(got, ref, lse, ref_lse)


@pytest.mark.parametrize("batch,tails", [(40, True), (70, True), (100, True)])
def test_many_segments(cuda_device, batch, tails):
    # more segments than one warp has lanes (one shared chain plus a private tail per request):
    # the scheduler's segment search reads the plan's rows 32 at a time, and a run's segment may
    # lie in any group of 32
    rng = np.random.default_rng(batch)
    lens = rng.integers(150, 700, size=batch)
    case = W.custom(B=batch, Hq=4, Hkv=2, D=128, ps=16, seq_lens=lens, shared_frac=0.6, seed=batch + tails)
    h = W.host_tensors(case)
    plan, got, lse, _, _ = run_both(case, h, cuda_device, 2, private_tails=tails, max_ctas=7)
    assert plan.num_segments > 32
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    check(got, ref, lse, ref_lse)
