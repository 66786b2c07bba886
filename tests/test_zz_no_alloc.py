"""rlt_paged_decode_attn_noalloc against rlt_paged_decode_attn, through the C ABI.

The no-allocation variant serves callers that cannot allocate device memory at
the point of the call (a host framework that owns every device allocation, or
a decode loop that must not risk a synchronising cudaMalloc): its split-K
partials live in a fixed array inside the library.  Two calls in a row, on
different inputs, must each give what the workspace-taking entry point gives
(the second call finds the first call's partials still in the array).  This
file is collected last so that a failure here stops a -x run only after every
other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import attn_close, bf16_dev, i32_dev

pytestmark = pytest.mark.gpu


def _inputs(seed, lens, device, Hq=16, Hkv=8, D=128, ps=16):
    case = W.custom(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, ps=ps, seq_lens=lens, seed=seed)
    h = W.host_tensors(case)
    pool = rlt.KVPool(bf16_dev(h.k_pool, device)[None].contiguous(), bf16_dev(h.v_pool, device)[None].contiguous())
    return case, pool, bf16_dev(h.q, device), i32_dev(case.page_table, device), i32_dev(case.seq_lens, device)


def _both(case, pool, q, pt, sl, split_tokens):
    ref_lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    ref = rlt.rlt_paged_decode_attn(pool, 0, q, pt, sl, case.max_seq_len, lse_out=ref_lse,
                                    split_tokens=split_tokens)
    out = torch.empty_like(q)
    lse = torch.empty_like(ref_lse)
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    rlt.rlt_paged_decode_attn_noalloc(pool, 0, q, pt, sl, case.max_seq_len, out=out, lse_out=lse,
                                      split_tokens=split_tokens)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before
    return ref.float().cpu().numpy(), ref_lse.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row(cuda_device):
    assert rlt.rlt_get_device_error() == 0
    # first call: long, ragged requests with many split-K partials in the scratch array
    args1 = _inputs(1, [4000, 17, 2500, 1, 640, 3333, 0, 1024], cuda_device)
    ref, ref_lse, got, lse = _both(*args1, split_tokens=64)
    assert rlt.rlt_paged_decode_workspace_size(8, 16, 8, 128, 4000, 64) > 0
    ok, mabs, mrel = attn_close(got, ref)
    assert ok, (mabs, mrel)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin) and np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-3
    # second call right after, other shapes and values, over the first call's leftovers
    args2 = _inputs(2, [300, 2900, 77, 1500], cuda_device, Hq=32, Hkv=8, D=64, ps=32)
    ref, ref_lse, got, lse = _both(*args2, split_tokens=0)
    ok, mabs, mrel = attn_close(got, ref)
    assert ok, (mabs, mrel)
    assert np.abs(lse - ref_lse).max() <= 1e-3
    assert rlt.rlt_get_device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_device):
    lib = rlt.load()
    pool = rlt.KVPool.empty(1, 4, 8, 16, 128, device=cuda_device)
    need = rlt.rlt_paged_decode_workspace_size(65535, 64, 8, 128, 1 << 20, 16)
    assert need > rlt.NOALLOC_SCRATCH_BYTES
    # aligned stand-ins for q, tables and out: the call is refused before any launch
    fake = ctypes.c_void_p(4096)
    status = lib.rlt_paged_decode_attn_noalloc(ctypes.byref(pool.struct), 0, fake, 64, fake, 1 << 16, fake, 65535,
                                               1 << 20, 0.0, fake, None, 16, None)
    assert status == 4                                   # RLT_ERR_WORKSPACE_TOO_SMALL, nothing launched
