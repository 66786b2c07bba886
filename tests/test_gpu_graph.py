"""The decode step as one CUDA-graph submission.

"Faster fuzzy minds" ("Recurrent depth — a deep model in a trench coat"): the
engine runs the looped model's decode step through its ordinary decode CUDA
graph; vllm-rlt PR #148 ("Fuse fixed-depth decode loops into one submission")
submits a fixed-depth loop's decode work together.  Every compute entry point
of the library is stream-capturable: captured once, a step of append +
attention over several layer-plane banks (+ noise) replays with the arrays'
current contents.  Checked: replay equals the eager calls bit for bit, and a
replay after the inputs' contents changed matches the oracle on the new inputs.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import NOISE_ABS, attn_close, bf16_dev, bits_host, i32_dev, i64_dev

pytestmark = pytest.mark.gpu


def capture(fn, device):
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        fn(side)
    torch.cuda.current_stream(device).wait_stream(side)
    return graph


@pytest.mark.parametrize("fused", [False, True])
def test_plain_step_replays_and_follows_new_inputs(cuda_device, fused):
    # fused: the append rides in the attention call (k_new / v_new), at position seq_lens[b] - 1
    case = W.config("tiny")
    banks = 3
    h = W.host_tensors(case)
    rng = np.random.default_rng(11)
    k = bf16_dev(np.stack([h.k_pool] * banks), cuda_device).contiguous()
    v = bf16_dev(np.stack([h.v_pool] * banks), cuda_device).contiguous()
    pool = rlt.KVPool(k, v)
    qs = [W.bf16_normal(rng, h.q.shape) for _ in range(banks)]
    kn = [W.bf16_normal(rng, h.k_new.shape) for _ in range(banks)]
    vn = [W.bf16_normal(rng, h.v_new.shape) for _ in range(banks)]
    q = bf16_dev(np.stack(qs), cuda_device)
    k_new = bf16_dev(np.stack(kn), cuda_device)
    v_new = bf16_dev(np.stack(vn), cuda_device)
    loc = i64_dev(case.new_slots, cuda_device)
    pt = i32_dev(case.page_table, cuda_device)
    sl = i32_dev(case.seq_lens, cuda_device)
    max_len = case.max_seq_len
    B, Hq, D = case.batch, case.num_q_heads, case.head_dim
    out = torch.empty((banks, B, Hq, D), dtype=torch.bfloat16, device=cuda_device)
    lse = torch.empty((banks, B, Hq), dtype=torch.float32, device=cuda_device)
    ws = torch.empty(max(rlt.rlt_paged_decode_workspace_size(B, Hq, case.num_kv_heads, D, max_len, 32), 16),
                     dtype=torch.uint8, device=cuda_device)

    def step(stream):
        for b in range(banks):
            if not fused:
                rlt.rlt_kv_append(pool, b, k_new[b], v_new[b], loc, stream=stream)
            extra = {"k_new": k_new[b], "v_new": v_new[b]} if fused else {}
            rlt.rlt_paged_decode_attn(pool, b, q[b], pt, sl, max_len, out=out[b], lse_out=lse[b],
                                      workspace=ws, split_tokens=32, stream=stream, **extra)

    # eager reference of the same step (appends overwrite the same slots: idempotent)
    step(torch.cuda.current_stream(cuda_device))
    torch.cuda.synchronize(cuda_device)
    eager, eager_lse = out.clone(), lse.clone()
    graph = capture(step, cuda_device)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize(cuda_device)
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert torch.equal(lse, eager_lse)
    assert rlt.rlt_get_device_error() == 0

    # new contents in the same buffers: other queries and new tokens, shorter lengths
    qs2 = [W.bf16_normal(rng, h.q.shape) for _ in range(banks)]
    kn2 = [W.bf16_normal(rng, h.k_new.shape) for _ in range(banks)]
    vn2 = [W.bf16_normal(rng, h.v_new.shape) for _ in range(banks)]
    q.copy_(bf16_dev(np.stack(qs2), cuda_device))
    k_new.copy_(bf16_dev(np.stack(kn2), cuda_device))
    v_new.copy_(bf16_dev(np.stack(vn2), cuda_device))
    lens2 = np.maximum(case.seq_lens - rng.integers(0, 40, size=B), 1).astype(np.int32)
    lens2[0] = 0                                   # an empty request too
    slots2 = np.array([case.page_table[b, (L - 1) // case.page_size] * case.page_size + (L - 1) % case.page_size
                       if L > 0 else -1 for b, L in enumerate(lens2)], np.int64)
    sl.copy_(i32_dev(lens2, cuda_device))
    loc.copy_(i64_dev(slots2, cuda_device))
    graph.replay()
    torch.cuda.synchronize(cuda_device)
    assert rlt.rlt_get_device_error() == 0
    for b in range(banks):
        kp, vp = h.k_pool.copy(), h.v_pool.copy()
        oracle.kv_append(kp, vp, kn[b], vn[b], case.new_slots)      # the first step's writes stay
        oracle.kv_append(kp, vp, kn2[b], vn2[b], slots2)
        assert np.array_equal(bits_host(k[b]), kp) and np.array_equal(bits_host(v[b]), vp)
        ref, ref_lse = oracle.decode_attn(qs2[b], kp, vp, case.page_table, lens2)
        got = out[b].float().cpu().numpy()
        ok, mabs, mrel = attn_close(got, ref)
        assert ok, f"bank {b}: max abs {mabs:.3e} max rel {mrel:.3e}"
        assert np.all(got[0] == 0) and np.all(np.isneginf(lse[b, 0].cpu().numpy()))
        fin = np.isfinite(ref_lse)
        assert np.abs(lse[b].cpu().numpy()[fin] - ref_lse[fin]).max() <= 1e-3


def test_cascade_step_with_noise_replays_bit_exact(cuda_device):
    # shared prefix -> tensor-core segments + split-K rest (forked onto a side stream and joined),
    # plus the new tokens' latent noise
    case = W.custom(B=6, Hq=16, Hkv=2, D=128, ps=16, seq_lens=[3000, 2900, 3100, 1500, 700, 2333],
                    shared_frac=0.8, seed=21)
    h = W.host_tensors(case)
    pool = rlt.KVPool(bf16_dev(h.k_pool, cuda_device)[None].contiguous(),
                      bf16_dev(h.v_pool, cuda_device)[None].contiguous())
    q = bf16_dev(h.q, cuda_device)
    pt = i32_dev(case.page_table, cuda_device)
    sl = i32_dev(case.seq_lens, cuda_device)
    nk = W.noise_keys(6 * 512, 256, seed=4)
    seeds_h, pos_h = nk.seeds, nk.positions
    seeds, pos = i64_dev(seeds_h, cuda_device), i64_dev(pos_h, cuda_device)
    noise = torch.empty((6 * 512, 256), dtype=torch.float32, device=cuda_device)
    results = {}
    for tails in (False, True):
        plan = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, 2, tails, case.group)
        plan.to(cuda_device)
        assert plan.num_segments > 0
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=cuda_device)

        def step(stream):
            rlt.rlt_latent_noise_init(seeds, pos, 256, 0.02, out=noise, stream=stream)
            rlt.rlt_paged_decode_attn_prefix(pool, 0, q, pt, sl, case.max_seq_len, plan, out=out, lse_out=lse,
                                             stream=stream)

        step(torch.cuda.current_stream(cuda_device))
        torch.cuda.synchronize(cuda_device)
        eager, eager_lse, eager_noise = out.clone(), lse.clone(), noise.clone()
        graph = capture(step, cuda_device)
        out.zero_()
        noise.zero_()
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize(cuda_device)
        assert rlt.rlt_get_device_error() == 0
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
        assert torch.equal(lse, eager_lse)
        assert torch.equal(noise, eager_noise)
        results[tails] = out.float().cpu().numpy()
    ref, _ = oracle.decode_attn(h.q, h.k_pool, h.v_pool, case.page_table, case.seq_lens)
    for got in results.values():
        ok, mabs, mrel = attn_close(got, ref)
        assert ok, f"max abs {mabs:.3e} max rel {mrel:.3e}"
    ref_noise = oracle.latent_noise_init(seeds_h, pos_h, 256, 0.02)
    assert np.abs(noise.cpu().numpy() - ref_noise).max() <= NOISE_ABS
