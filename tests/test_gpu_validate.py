"""Debug mode RLT_VALIDATE=1: the compute calls check the batch's device arrays on the host
before launching.

"When scheduler does the work" ("Faster fuzzy minds"): the scheduler hands each token a slot
of the flat pool and requests sharing a prompt share its pages read-only.  In debug mode a
batch that breaks this (a page id outside the pool, a length past the page-table row, two
tokens written to one slot, a new token's slot on a page another request maps) fails the
call with a status and nothing is launched; a valid batch runs as without the mode.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import attn_close, bf16_dev, i32_dev, i64_dev

pytestmark = pytest.mark.gpu


@pytest.fixture
def validate(monkeypatch):
    monkeypatch.setenv("RLT_VALIDATE", "1")


def setup(case, device):
    h = W.host_tensors(case)
    pool = rlt.KVPool(bf16_dev(h.k_pool, device)[None].contiguous(), bf16_dev(h.v_pool, device)[None].contiguous())
    return h, pool, bf16_dev(h.q, device)


def test_valid_batch_runs_as_usual(cuda_device, validate):
    case = W.config("tiny")
    h, pool, q = setup(case, cuda_device)
    kn, vn = bf16_dev(h.k_new, cuda_device), bf16_dev(h.v_new, cuda_device)
    rlt.rlt_get_device_error()
    out = rlt.rlt_paged_decode_attn(pool, 0, q, i32_dev(case.page_table, cuda_device),
                                    i32_dev(case.seq_lens, cuda_device), case.max_seq_len, k_new=kn, v_new=vn)
    assert rlt.rlt_get_device_error() == 0
    kp, vp = h.k_pool.copy(), h.v_pool.copy()
    oracle.kv_append(kp, vp, h.k_new, h.v_new, case.new_slots)
    ref, _ = oracle.decode_attn(h.q, kp, vp, case.page_table, case.seq_lens)
    ok, mabs, mrel = attn_close(out.float().cpu().numpy(), ref)
    assert ok, f"max abs {mabs:.3e} max rel {mrel:.3e}"


def test_bad_page_fails_the_call_before_launch(cuda_device, validate):
    case = W.config("tiny")
    h, pool, q = setup(case, cuda_device)
    pt = case.page_table.copy()
    pt[1, 0] = case.num_pages + 3
    out = torch.full_like(q, 7.0)
    rlt.rlt_get_device_error()
    with pytest.raises(rlt.RltError) as e:
        rlt.rlt_paged_decode_attn(pool, 0, q, i32_dev(pt, cuda_device), i32_dev(case.seq_lens, cuda_device),
                                  case.max_seq_len, out=out)
    assert e.value.status == 2                                  # RLT_ERR_OUT_OF_RANGE
    torch.cuda.synchronize()
    assert rlt.rlt_get_device_error() == 0                      # nothing ran
    assert torch.all(out == 7.0)


def test_length_past_the_row_fails(cuda_device, validate):
    case = W.config("tiny")
    h, pool, q = setup(case, cuda_device)
    sl = case.seq_lens.copy()
    sl[2] = case.page_table.shape[1] * case.page_size + 1
    with pytest.raises(rlt.RltError):
        rlt.rlt_paged_decode_attn(pool, 0, q, i32_dev(case.page_table, cuda_device), i32_dev(sl, cuda_device),
                                  int(sl.max()))


def test_new_token_on_a_page_another_request_maps_fails(cuda_device, validate):
    # request 1 maps request 0's last page: request 0's fused append would write a shared page
    case = W.custom(B=3, Hq=4, Hkv=2, D=64, ps=16, seq_lens=[40, 90, 33], seed=5)
    h, pool, q = setup(case, cuda_device)
    pt = case.page_table.copy()
    pt[1, 0] = pt[0, (40 - 1) // 16]
    kn, vn = bf16_dev(h.k_new, cuda_device), bf16_dev(h.v_new, cuda_device)
    with pytest.raises(rlt.RltError):
        rlt.rlt_paged_decode_attn(pool, 0, q, i32_dev(pt, cuda_device), i32_dev(case.seq_lens, cuda_device),
                                  case.max_seq_len, k_new=kn, v_new=vn)
    # without the append the same tables are a valid (read-only) sharing
    rlt.rlt_paged_decode_attn(pool, 0, q, i32_dev(pt, cuda_device), i32_dev(case.seq_lens, cuda_device),
                              case.max_seq_len)


def test_append_slots_out_of_pool_or_repeated_fail(cuda_device, validate):
    case = W.config("tiny")
    h, pool, _ = setup(case, cuda_device)
    kn, vn = bf16_dev(h.k_new, cuda_device), bf16_dev(h.v_new, cuda_device)
    k0 = pool.k.clone()
    bad = case.new_slots.copy()
    bad[1] = case.num_pages * case.page_size
    with pytest.raises(rlt.RltError) as e:
        rlt.rlt_kv_append(pool, 0, kn, vn, i64_dev(bad, cuda_device))
    assert e.value.status == 2
    dup = case.new_slots.copy()
    dup[2] = dup[0]
    with pytest.raises(rlt.RltError) as e:
        rlt.rlt_kv_append(pool, 0, kn, vn, i64_dev(dup, cuda_device))
    assert e.value.status == 1                                  # RLT_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.equal(pool.k.view(torch.int16), k0.view(torch.int16))
    rlt.rlt_kv_append(pool, 0, kn, vn, i64_dev(case.new_slots, cuda_device))   # the valid batch goes through


def test_shared_prefix_call_is_checked(cuda_device, validate):
    case = W.custom(B=4, Hq=4, Hkv=4, D=128, ps=16, seq_lens=[900, 1000, 700, 1200], shared_frac=0.8, seed=9)
    h, pool, q = setup(case, cuda_device)
    plan = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, 2, False, case.group)
    assert plan.num_segments > 0
    plan.to(cuda_device)
    rlt.rlt_paged_decode_attn_prefix(pool, 0, q, i32_dev(case.page_table, cuda_device),
                                     i32_dev(case.seq_lens, cuda_device), case.max_seq_len, plan)
    pt = case.page_table.copy()
    pt[3, -1] = -5
    with pytest.raises(rlt.RltError):
        rlt.rlt_paged_decode_attn_prefix(pool, 0, q, i32_dev(pt, cuda_device), i32_dev(case.seq_lens, cuda_device),
                                         case.max_seq_len, plan)


def test_capture_skips_the_check(cuda_device, validate):
    # a capture cannot synchronise: the calls are recorded unchecked and replay normally
    case = W.config("tiny")
    h, pool, q = setup(case, cuda_device)
    pt, sl = i32_dev(case.page_table, cuda_device), i32_dev(case.seq_lens, cuda_device)
    out = torch.empty_like(q)
    rlt.rlt_paged_decode_attn(pool, 0, q, pt, sl, case.max_seq_len, out=out)     # first call outside
    torch.cuda.synchronize()
    ref = out.clone()
    side = torch.cuda.Stream(cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        rlt.rlt_paged_decode_attn(pool, 0, q, pt, sl, case.max_seq_len, out=out, stream=side)
    torch.cuda.current_stream(cuda_device).wait_stream(side)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
