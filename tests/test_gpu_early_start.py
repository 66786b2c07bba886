"""Attention calls launched with RLT_ATTN_EARLY_START, chained as layers are.

With the flag a call's kernels are programmatic dependents of the kernel ahead of
them: they start while it still runs, read the page table, lengths, plan and the
bank's cached rows at once, and wait for it before reading q / k_new / v_new or
writing out, lse and the (shared) workspace.  Here call i+1's q, k_new and v_new
ARE call i's output buffer, written by call i's last kernel after it has let its
dependents start, and every call shares one workspace; before each run the
output buffers are filled with large garbage.  A read of q or of the new rows
before the wait, or a partial written while the previous combine still reads
the workspace, would show as a wrong output.  The expected values come from the
oracle run as the same chain (each output rounded to bf16 by the oracle's own
rounding and fed to the next call).  Checked eagerly (stream order) and as one
captured CUDA graph (programmatic graph edges, through the shared-prefix call's
fork and join too).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import attn_close, bf16_dev, bits_host, i32_dev

pytestmark = pytest.mark.gpu

N_CALLS = 4
LENS = [700, 1500, 33, 2047, 1, 900, 1200, 640]


def _setup(device, cascade, seed):
    # G = 1 (Hq = Hkv) so that one output [B][Hq][D] is also the next call's k_new / v_new
    case = W.custom(B=len(LENS), Hq=8, Hkv=8, D=128, ps=16, seq_lens=LENS, shared_frac=0.8 if cascade else 0.0,
                    seed=seed)
    hs = [W.host_tensors(case, seed=seed * 100 + i) for i in range(N_CALLS)]
    k = bf16_dev(np.stack([h.k_pool for h in hs]), device).contiguous()
    v = bf16_dev(np.stack([h.v_pool for h in hs]), device).contiguous()
    return case, hs, rlt.KVPool(k, v)


def _oracle_chain(case, hs):
    q, kn, vn = hs[0].q, hs[0].k_new, hs[0].v_new
    refs, lses, pools = [], [], []
    for i in range(N_CALLS):
        kp, vp = hs[i].k_pool.copy(), hs[i].v_pool.copy()
        oracle.kv_append(kp, vp, kn, vn, case.new_slots)
        ref, lse = oracle.decode_attn(q, kp, vp, case.page_table, case.seq_lens)
        refs.append(ref)
        lses.append(lse)
        pools.append((kp, vp))
        q = kn = vn = W.float_to_bf16_bits(ref.astype(np.float32))
    return refs, lses, pools


@pytest.mark.parametrize("cascade,split_tokens", [(False, 64), (False, 2048), (True, 0)])
def test_early_start_chain_matches_oracle(cuda_device, cascade, split_tokens):
    case, hs, pool = _setup(cuda_device, cascade, seed=31 + split_tokens)
    B, Hq, D = case.batch, case.num_q_heads, case.head_dim
    pt, sl = i32_dev(case.page_table, cuda_device), i32_dev(case.seq_lens, cuda_device)
    q0, kn0, vn0 = (bf16_dev(a, cuda_device) for a in (hs[0].q, hs[0].k_new, hs[0].v_new))
    outs = torch.empty((N_CALLS, B, Hq, D), dtype=torch.bfloat16, device=cuda_device)
    lses = torch.empty((N_CALLS, B, Hq), dtype=torch.float32, device=cuda_device)
    plan = None
    if cascade:
        plan = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, 2, False, case.group)
        assert plan.num_segments > 0 and plan.max_rest_len > 0      # tensor-core kernel + split-K rest
        plan.to(cuda_device)
        ws_bytes = rlt.rlt_paged_decode_prefix_workspace_size(B, Hq, case.num_kv_heads, D, plan.max_rest_len,
                                                              plan.max_prefix_slots, split_tokens)
    else:
        ws_bytes = rlt.rlt_paged_decode_workspace_size(B, Hq, case.num_kv_heads, D, case.max_seq_len, split_tokens)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=cuda_device)
    pool_k0, pool_v0 = pool.k.clone(), pool.v.clone()
    refs, ref_lses, ref_pools = _oracle_chain(case, hs)

    def chain(stream):
        for i in range(N_CALLS):
            src = outs[i - 1] if i > 0 else None
            q = src if src is not None else q0
            kn = src if src is not None else kn0
            vn = src if src is not None else vn0
            kw = dict(out=outs[i], lse_out=lses[i], workspace=ws, split_tokens=split_tokens, stream=stream,
                      k_new=kn, v_new=vn, early_start=True)
            if cascade:
                rlt.rlt_paged_decode_attn_prefix(pool, i, q, pt, sl, case.max_seq_len, plan, **kw)
            else:
                rlt.rlt_paged_decode_attn(pool, i, q, pt, sl, case.max_seq_len, **kw)

    def check():
        torch.cuda.synchronize(cuda_device)
        assert rlt.rlt_get_device_error() == 0
        got, got_lse = outs.float().cpu().numpy(), lses.cpu().numpy()
        for i in range(N_CALLS):
            ok, mabs, mrel = attn_close(got[i], refs[i])
            assert ok, (i, mabs, mrel)
            fin = np.isfinite(ref_lses[i])
            assert np.array_equal(np.isfinite(got_lse[i]), fin)
            assert np.abs(got_lse[i][fin] - ref_lses[i][fin]).max() <= 1e-3, i
        # the first call's append is bit-exact against the oracle; later calls store the rows
        # they were handed (the previous call's output) and touch nothing else
        kb, vb = bits_host(pool.k), bits_host(pool.v)
        assert np.array_equal(kb[0], ref_pools[0][0]) and np.array_equal(vb[0], ref_pools[0][1])
        flat = lambda a: a.reshape(-1, D)                       # noqa: E731  rows of one bank by slot*Hkv+h
        rows = np.array([int(s) // case.page_size * case.num_kv_heads * case.page_size + int(s) % case.page_size
                         for s in case.new_slots if s >= 0], np.int64)
        heads = np.arange(case.num_kv_heads, dtype=np.int64) * case.page_size
        new_rows = (rows[:, None] + heads[None, :]).reshape(-1)
        live = np.flatnonzero(case.new_slots >= 0)
        prev = bits_host(outs)
        for i in range(1, N_CALLS):
            for name, cur, orig in (("k", kb[i], hs[i].k_pool), ("v", vb[i], hs[i].v_pool)):
                c, o = flat(cur).copy(), flat(orig)
                assert np.array_equal(c[new_rows], prev[i - 1][live].reshape(-1, D)), (name, i)
                c[new_rows] = o[new_rows]
                assert np.array_equal(c, o), (name, i)

    def reset():
        pool.k.copy_(pool_k0)
        pool.v.copy_(pool_v0)
        outs.fill_(100.0)                        # garbage a too-early read would pick up
        lses.fill_(float("nan"))
        torch.cuda.synchronize(cuda_device)

    stream = torch.cuda.current_stream(cuda_device)
    for _ in range(2):                           # eager: programmatic dependents in stream order
        reset()
        chain(stream)
        check()

    side = torch.cuda.Stream(cuda_device)
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        chain(side)
    stream.wait_stream(side)
    for _ in range(3):                           # one captured graph: programmatic edges
        reset()
        graph.replay()
        check()
