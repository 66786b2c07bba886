"""The split-K kernel's bounded copy wait gives up, reports it, and leaves the device usable.

Every wait of the library's kernels has a time limit; a wait that runs out
records RLT_DEVERR_TIMEOUT, waits (bounded) for the copies its warp still has
in flight, and returns instead of spinning forever.  rlt_debug_fault_next_decode
makes that happen on purpose without any GPU fault: the next call's first tile
copy of one warp is never issued (the bytes its barrier expects never come) and
the wait limit is a few milliseconds.  Checked: the call returns at once, the
error word holds exactly the timeout bit, no byte outside the outputs,
workspace and pool changes, every row the dropped tile does not feed still
matches the oracle, and the next ordinary call on the same device matches the
oracle everywhere.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import attn_close, bf16_dev, i32_dev
from test_gpu_guards import Guarded, pool_of, ragged_case

pytestmark = pytest.mark.gpu


def test_copy_wait_runs_out_and_the_next_call_is_exact(cuda_device):
    G, D, split_tokens = 2, 128, 64
    case = ragged_case(G, D, seed=91)
    h = W.host_tensors(case)
    pool, pg = pool_of(h, cuda_device)
    B, Hq = case.batch, case.num_q_heads
    out = Guarded(B * Hq * D * 2, cuda_device)
    lse = Guarded(B * Hq * 4, cuda_device)
    ws_n = rlt.rlt_paged_decode_workspace_size(B, Hq, case.num_kv_heads, D, case.max_seq_len, split_tokens)
    ws = Guarded(ws_n, cuda_device)
    q, pt, sl = (bf16_dev(h.q, cuda_device), i32_dev(case.page_table, cuda_device),
                 i32_dev(case.seq_lens, cuda_device))

    def call():
        rlt.rlt_paged_decode_attn(pool, 0, q, pt, sl, case.max_seq_len, out=out.view(torch.bfloat16, (B, Hq, D)),
                                  lse_out=lse.view(torch.float32, (B, Hq)), workspace=ws.bytes(),
                                  split_tokens=split_tokens)

    ref, ref_lse = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    call()                                            # warm: attributes set, modules loaded
    torch.cuda.synchronize(cuda_device)
    assert rlt.rlt_get_device_error() == 0

    rlt.rlt_debug_fault_next_decode(2_000_000)        # 2 ms per wait
    t0 = time.perf_counter()
    call()
    torch.cuda.synchronize(cuda_device)
    elapsed = time.perf_counter() - t0
    assert rlt.rlt_get_device_error() == rlt.DEVERR_TIMEOUT
    assert elapsed < 0.5, elapsed                     # two 2 ms waits ran out, not the 1 s default
    assert out.intact() and lse.intact() and ws.intact() and pg[0].intact() and pg[1].intact()
    got = out.view(torch.bfloat16, (B, Hq, D)).float().cpu().numpy()
    got_lse = lse.view(torch.float32, (B, Hq)).cpu().numpy()
    assert np.isfinite(got).all()
    # request 0's query heads of kv head 0 lost the dropped tile; every other row is exact
    keep = np.ones((B, Hq), bool)
    keep[0, :G] = False
    ok, mabs, mrel = attn_close(got[keep], ref[keep])
    assert ok, (mabs, mrel)
    assert np.abs(got_lse[keep] - ref_lse[keep]).max() <= 1e-3
    # the fault did take effect: those rows' log-sum-exp misses the dropped tokens' weight
    assert np.abs(got_lse[0, :G] - ref_lse[0, :G]).min() > 1e-3

    call()                                            # the switch was one-shot: exact again
    torch.cuda.synchronize(cuda_device)
    assert rlt.rlt_get_device_error() == 0
    got = out.view(torch.bfloat16, (B, Hq, D)).float().cpu().numpy()
    ok, mabs, mrel = attn_close(got, ref)
    assert ok, (mabs, mrel)
    assert out.intact() and lse.intact() and ws.intact() and pg[0].intact() and pg[1].intact()
