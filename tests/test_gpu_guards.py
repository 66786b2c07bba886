"""Guard regions around every device buffer an entry point writes.

compute-sanitizer is not available on the GPU pool, so out-of-bounds writes are
caught the plain way: each output (and each workspace, sized exactly as the
library's size function says) sits between two 4 KiB guard regions filled with
a byte pattern, and after the call both guards must be unchanged.  The results
are also checked against the oracle, so a write that stayed in bounds but
landed in the wrong place still fails.  Cases use ragged lengths, many splits,
shared-prefix segments with and without private tails, and ragged channel
counts.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import NOISE_ABS, attn_close, bf16_dev, bits_host, i32_dev, i64_dev

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side; keeps the buffer 16-byte aligned
PATTERN = 0xA5


class Guarded:
    """nbytes of device memory between two guard regions."""

    def __init__(self, nbytes, device):
        self.n = int(nbytes)
        self.raw = torch.full((self.n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=device)

    def view(self, dtype, shape):
        return self.raw[GUARD: GUARD + self.n].view(dtype).view(shape)

    def bytes(self):
        return self.raw[GUARD: GUARD + self.n]

    def intact(self):
        return bool((self.raw[:GUARD] == PATTERN).all()) and bool((self.raw[GUARD + self.n:] == PATTERN).all())


def pool_of(h, device):
    k = Guarded(h.k_pool.size * 2, device)
    v = Guarded(h.v_pool.size * 2, device)
    kv = k.view(torch.int16, (1,) + h.k_pool.shape)
    vv = v.view(torch.int16, (1,) + h.v_pool.shape)
    kv.copy_(torch.from_numpy(h.k_pool.view(np.int16)).to(device)[None])
    vv.copy_(torch.from_numpy(h.v_pool.view(np.int16)).to(device)[None])
    return rlt.KVPool(kv.view(torch.bfloat16), vv.view(torch.bfloat16)), (k, v)


def ragged_case(G, D, seed, shared_frac=0.0):
    lens = [700, 33, 2000, 1, 1500, 129]
    return W.custom(B=len(lens), Hq=2 * G, Hkv=2, D=D, ps=16, seq_lens=lens, shared_frac=shared_frac, seed=seed)


@pytest.mark.parametrize("G,D,split_tokens", [(1, 128, 64), (4, 128, 0), (2, 64, 16), (8, 64, 128)])
def test_plain_decode_stays_in_its_buffers(cuda_device, G, D, split_tokens):
    case = ragged_case(G, D, seed=G * 10 + D)
    h = W.host_tensors(case)
    pool, pg = pool_of(h, cuda_device)
    B, Hq = case.batch, case.num_q_heads
    out = Guarded(B * Hq * D * 2, cuda_device)
    lse = Guarded(B * Hq * 4, cuda_device)
    ws_n = rlt.rlt_paged_decode_workspace_size(B, Hq, case.num_kv_heads, D, case.max_seq_len, split_tokens)
    ws = Guarded(max(ws_n, 16), cuda_device)
    rlt.rlt_paged_decode_attn(pool, 0, bf16_dev(h.q, cuda_device), i32_dev(case.page_table, cuda_device),
                              i32_dev(case.seq_lens, cuda_device), case.max_seq_len,
                              out=out.view(torch.bfloat16, (B, Hq, D)), lse_out=lse.view(torch.float32, (B, Hq)),
                              workspace=ws.bytes() if ws_n > 0 else None, split_tokens=split_tokens)
    torch.cuda.synchronize(cuda_device)
    assert rlt.rlt_get_device_error() == 0
    assert out.intact() and lse.intact() and ws.intact() and pg[0].intact() and pg[1].intact()
    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    ok, mabs, mrel = attn_close(out.view(torch.bfloat16, (B, Hq, D)).float().cpu().numpy(), ref)
    assert ok, f"max abs {mabs:.3e} max rel {mrel:.3e}"
    assert np.abs(lse.view(torch.float32, (B, Hq)).cpu().numpy() - ref_lse).max() <= 1e-3


@pytest.mark.parametrize("G,tails", [(1, False), (4, False), (8, True), (2, True)])
def test_shared_prefix_stays_in_its_buffers(cuda_device, G, tails):
    case = ragged_case(G, 128, seed=G + 3, shared_frac=0.8)
    h = W.host_tensors(case)
    pool, pg = pool_of(h, cuda_device)
    B, Hq = case.batch, case.num_q_heads
    plan = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, 2, tails, case.group).to(cuda_device)
    assert plan.num_segments > 0
    out = Guarded(B * Hq * 128 * 2, cuda_device)
    lse = Guarded(B * Hq * 4, cuda_device)
    ws = Guarded(rlt.rlt_paged_decode_prefix_workspace_size(B, Hq, case.num_kv_heads, 128, plan.max_rest_len,
                                                           plan.max_prefix_slots), cuda_device)
    rlt.rlt_paged_decode_attn_prefix(pool, 0, bf16_dev(h.q, cuda_device), i32_dev(case.page_table, cuda_device),
                                     i32_dev(case.seq_lens, cuda_device), case.max_seq_len, plan,
                                     out=out.view(torch.bfloat16, (B, Hq, 128)),
                                     lse_out=lse.view(torch.float32, (B, Hq)), workspace=ws.bytes())
    torch.cuda.synchronize(cuda_device)
    assert rlt.rlt_get_device_error() == 0
    assert out.intact() and lse.intact() and ws.intact() and pg[0].intact() and pg[1].intact()
    ref, _ = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    ok, mabs, mrel = attn_close(out.view(torch.bfloat16, (B, Hq, 128)).float().cpu().numpy(), ref)
    assert ok, f"max abs {mabs:.3e} max rel {mrel:.3e}"


def test_extend_stays_in_its_buffers(cuda_device):
    case = ragged_case(4, 128, seed=77)
    h = W.host_tensors(case)
    pool, pg = pool_of(h, cuda_device)
    new = np.minimum(case.seq_lens, [40, 33, 130, 1, 7, 129]).astype(np.int32)
    rows, Hq = int(new.sum()), case.num_q_heads
    rng = np.random.default_rng(5)
    q = W.bf16_normal(rng, (rows, Hq, 128))
    plan = rlt.rlt_plan_extend(case.seq_lens, new, case.page_size, 2, case.group).to(cuda_device)
    out = Guarded(rows * Hq * 128 * 2, cuda_device)
    lse = Guarded(rows * Hq * 4, cuda_device)
    ws = Guarded(int(rlt.load().rlt_paged_extend_workspace_size(rows, Hq, 128, max(plan.max_slots, 1))), cuda_device)
    rlt.rlt_paged_extend_attn(pool, 0, bf16_dev(q, cuda_device), i32_dev(case.page_table, cuda_device), plan,
                              out=out.view(torch.bfloat16, (rows, Hq, 128)),
                              lse_out=lse.view(torch.float32, (rows, Hq)), workspace=ws.bytes())
    torch.cuda.synchronize(cuda_device)
    assert rlt.rlt_get_device_error() == 0
    assert out.intact() and lse.intact() and ws.intact() and pg[0].intact() and pg[1].intact()
    ref, _ = oracle.extend_attn(q, h.k_pool, h.v_pool, case.page_table, case.seq_lens, new)
    ok, mabs, mrel = attn_close(out.view(torch.bfloat16, (rows, Hq, 128)).float().cpu().numpy(), ref)
    assert ok, f"max abs {mabs:.3e} max rel {mrel:.3e}"


def test_append_gather_and_noalloc_stay_in_their_buffers(cuda_device):
    case = ragged_case(2, 64, seed=19)
    h = W.host_tensors(case)
    pool, pg = pool_of(h, cuda_device)
    B, Hq, Hkv, D = case.batch, case.num_q_heads, case.num_kv_heads, case.head_dim
    kn = Guarded(B * Hkv * D * 2, cuda_device)
    vn = Guarded(B * Hkv * D * 2, cuda_device)
    kn.view(torch.int16, (B, Hkv, D)).copy_(torch.from_numpy(h.k_new.view(np.int16)).to(cuda_device))
    vn.view(torch.int16, (B, Hkv, D)).copy_(torch.from_numpy(h.v_new.view(np.int16)).to(cuda_device))
    rlt.rlt_kv_append(pool, 0, kn.view(torch.bfloat16, (B, Hkv, D)), vn.view(torch.bfloat16, (B, Hkv, D)),
                      i64_dev(case.new_slots, cuda_device))
    max_len = int(case.seq_lens.max())
    ko = Guarded(B * max_len * Hkv * D * 2, cuda_device)
    vo = Guarded(B * max_len * Hkv * D * 2, cuda_device)
    rlt.rlt_paged_gather(pool, 0, i32_dev(case.page_table, cuda_device), i32_dev(case.seq_lens, cuda_device),
                         max_len, k_out=ko.view(torch.bfloat16, (B, max_len, Hkv, D)),
                         v_out=vo.view(torch.bfloat16, (B, max_len, Hkv, D)))
    out = Guarded(B * Hq * D * 2, cuda_device)
    lse = Guarded(B * Hq * 4, cuda_device)
    rlt.rlt_paged_decode_attn_noalloc(pool, 0, bf16_dev(h.q, cuda_device), i32_dev(case.page_table, cuda_device),
                                      i32_dev(case.seq_lens, cuda_device), case.max_seq_len,
                                      out=out.view(torch.bfloat16, (B, Hq, D)),
                                      lse_out=lse.view(torch.float32, (B, Hq)), split_tokens=16)
    torch.cuda.synchronize(cuda_device)
    assert rlt.rlt_get_device_error() == 0
    for g in (kn, vn, ko, vo, out, lse) + pg:
        assert g.intact()
    kp, vp = h.k_pool.copy(), h.v_pool.copy()
    oracle.kv_append(kp, vp, h.k_new, h.v_new, case.new_slots)
    assert np.array_equal(bits_host(pool.k[0]), kp) and np.array_equal(bits_host(pool.v[0]), vp)
    kr, vr = oracle.paged_gather(kp, vp, case.page_table, case.seq_lens, max_len=max_len)
    kg = bits_host(ko.view(torch.bfloat16, (B, max_len, Hkv, D)))
    for b in range(B):
        n = int(case.seq_lens[b])
        assert np.array_equal(kg[b, :n], kr[b, :n])
    ref, _ = oracle.decode_attn(h.q, kp, vp, case.page_table, case.seq_lens)
    ok, mabs, mrel = attn_close(out.view(torch.bfloat16, (B, Hq, D)).float().cpu().numpy(), ref)
    assert ok, f"max abs {mabs:.3e} max rel {mrel:.3e}"


@pytest.mark.parametrize("rows,channels", [(37, 100), (5, 4096), (1, 3)])
def test_noise_and_publication_stay_in_their_buffers(cuda_device, rows, channels):
    nk = W.noise_keys(rows, channels, seed=rows)
    out = Guarded(rows * channels * 4, cuda_device)
    rlt.rlt_latent_noise_init(i64_dev(nk.seeds, cuda_device), i64_dev(nk.positions, cuda_device), channels, 0.02,
                              out=out.view(torch.float32, (rows, channels)))
    written = torch.randint(0, 500, (3, rows), dtype=torch.int32, device=cuda_device)
    pub = Guarded(rows * 4, cuda_device)
    rlt.rlt_publishable_prefix(written, 16, out=pub.view(torch.int32, (rows,)))
    torch.cuda.synchronize(cuda_device)
    assert out.intact() and pub.intact()
    ref = oracle.latent_noise_init(nk.seeds, nk.positions, channels, 0.02)
    assert np.abs(out.view(torch.float32, (rows, channels)).cpu().numpy() - ref).max() <= NOISE_ABS
    w = written.cpu().numpy()
    assert np.array_equal(pub.view(torch.int32, (rows,)).cpu().numpy(), w.min(axis=0) // 16 * 16)
