"""GPU parity of the fused RoPE append and of the prefix-publication coverage.

"Faster fuzzy minds" ("Recurrent depth"): a token keeps one RoPE position
across all T of its banks.  vllm-rlt PR #152 (Summary): publication needs a
written prefix in every layer each plane holds.  Bar: V rows and untouched
slots bit-exact; rotated keys within one bf16 ulp of the fp64 oracle (the
kernel rotates in fp32), with such ulp flips rare; counters and publishable
lengths bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import bf16_dev, bits_host, i64_dev

pytestmark = pytest.mark.gpu


def ulp_diff(a, b):
    """|a - b| in units of bf16 patterns (same-sign values)."""
    a = a.astype(np.int32)
    b = b.astype(np.int32)
    sa = np.where(a & 0x8000, -(a & 0x7FFF), a & 0x7FFF)
    sb = np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.abs(sa - sb)


def random_case(rng, P, Hkv, ps, D, n, banks=1):
    k = W.bf16_normal(rng, (banks, P, Hkv, ps, D))
    v = W.bf16_normal(rng, (banks, P, Hkv, ps, D))
    kn = W.bf16_normal(rng, (n, Hkv, D))
    vn = W.bf16_normal(rng, (n, Hkv, D))
    slots = rng.choice(P * ps, size=n, replace=False).astype(np.int64)
    slots[rng.random(n) < 0.1] = -1
    pos = rng.integers(0, 131072, size=n).astype(np.int64)
    pos[:3] = [0, 1, 131071][: min(3, n)]
    return k, v, kn, vn, slots, pos


@pytest.mark.parametrize("D,rot_dim,base", [(128, 128, 10000.0), (128, 64, 500000.0), (64, 64, 10000.0),
                                            (128, 2, 10000.0)])
def test_append_rope_matches_oracle(cuda_device, D, rot_dim, base):
    rng = np.random.default_rng(D + rot_dim)
    P, Hkv, ps, n = 40, 4, 16, 300
    k, v, kn, vn, slots, pos = random_case(rng, P, Hkv, ps, D, n)
    pool = rlt.KVPool(bf16_dev(k, cuda_device), bf16_dev(v, cuda_device))
    rlt.rlt_kv_append_rope(pool, 0, bf16_dev(kn, cuda_device), bf16_dev(vn, cuda_device), i64_dev(pos, cuda_device),
                           i64_dev(slots, cuda_device), rot_dim, base)
    assert rlt.rlt_get_device_error() == 0
    kr, vr = k[0].copy(), v[0].copy()
    oracle.kv_append_rope(kr, vr, kn, vn, pos, slots, rot_dim, base)
    kg, vg = bits_host(pool.k[0]), bits_host(pool.v[0])
    assert np.array_equal(vg, vr)
    d = ulp_diff(kg, kr)
    assert d.max() <= 1
    assert (d > 0).mean() < 0.01
    # everything outside the appended rows is untouched
    mask = np.ones(kg.shape, bool)
    for s in slots[slots >= 0]:
        mask[s // ps, :, s % ps] = False
    assert np.array_equal(kg[mask], k[0][mask])


def test_one_position_for_every_plane(cuda_device):
    # the same token appended to the banks of 4 planes at its sequence position: identical keys
    rng = np.random.default_rng(7)
    P, Hkv, ps, D, n = 20, 2, 16, 128, 64
    k, v, kn, vn, slots, pos = random_case(rng, P, Hkv, ps, D, n, banks=4)
    pool = rlt.KVPool(bf16_dev(k, cuda_device), bf16_dev(v, cuda_device))
    knd, vnd = bf16_dev(kn, cuda_device), bf16_dev(vn, cuda_device)
    pd, sd = i64_dev(pos, cuda_device), i64_dev(slots, cuda_device)
    for bank in range(4):
        rlt.rlt_kv_append_rope(pool, bank, knd, vnd, pd, sd, D, 10000.0)
    kg = bits_host(pool.k)
    live = slots[slots >= 0]
    rows = [kg[b][live // ps, :, live % ps] for b in range(4)]
    for b in range(1, 4):
        assert np.array_equal(rows[b], rows[0])


def test_written_counters_and_publishable_prefix(cuda_device):
    # a partially looped stack: layers 0 and 3 on plane 0 only, layers 1-2 looped over 3 planes
    recurrent = [0, 1, 1, 0]
    T, B, ps = 3, 6, 16
    bmap, nbanks = rlt.rlt_bank_map(recurrent, T)
    assert nbanks == 8
    rng = np.random.default_rng(8)
    P, Hkv, D = 64, 2, 64
    pool = rlt.KVPool.empty(nbanks, P, Hkv, ps, D, device=cuda_device)
    written = torch.zeros((nbanks, B), dtype=torch.int32, device=cuda_device)
    w_ref = np.zeros((nbanks, B), np.int32)
    lens = rng.integers(20, 200, size=B)
    slot_base = 0
    for bank in range(nbanks):
        # each bank receives a prefill chunk of every request, of a length that varies by bank
        req, pos, loc = [], [], []
        for b in range(B):
            L = int(max(lens[b] - rng.integers(0, 30), 0))
            req += [b] * L
            pos += list(range(L))
        n = len(req)
        loc = (np.arange(n) % (P * ps)).astype(np.int64)
        loc[rng.random(n) < 0.05] = -1
        kn = W.bf16_normal(rng, (n, Hkv, D))
        req_a, pos_a = np.array(req, np.int32), np.array(pos, np.int64)
        rlt.rlt_kv_append_rope(pool, bank, bf16_dev(kn, cuda_device), bf16_dev(kn, cuda_device),
                               i64_dev(pos_a, cuda_device), i64_dev(loc, cuda_device), D, 10000.0,
                               request=torch.from_numpy(req_a).to(cuda_device), written=written)
        oracle.mark_written(w_ref, bank, req_a, pos_a, loc)
    assert rlt.rlt_get_device_error() == 0
    assert np.array_equal(written.cpu().numpy(), w_ref)
    got = rlt.rlt_publishable_prefix(written, ps).cpu().numpy()
    assert np.array_equal(got, oracle.publishable_prefix(bmap, w_ref, ps))
    assert np.all(got > 0)


def test_bad_request_and_slot_are_flagged(cuda_device):
    pool = rlt.KVPool.empty(1, 4, 1, 16, 64, device=cuda_device)
    kn = torch.zeros((2, 1, 64), dtype=torch.bfloat16, device=cuda_device)
    written = torch.zeros((1, 2), dtype=torch.int32, device=cuda_device)
    pos = torch.tensor([5, 6], dtype=torch.int64, device=cuda_device)
    rlt.rlt_kv_append_rope(pool, 0, kn, kn, pos, torch.tensor([1, 2], dtype=torch.int64, device=cuda_device), 64,
                           1e4, request=torch.tensor([0, 7], dtype=torch.int32, device=cuda_device), written=written)
    assert rlt.rlt_get_device_error() == rlt.DEVERR_BAD_SLOT
    assert written.cpu().tolist() == [[6, 0]]
    rlt.rlt_kv_append_rope(pool, 0, kn, kn, pos, torch.tensor([1, 64], dtype=torch.int64, device=cuda_device), 64,
                           1e4)
    assert rlt.rlt_get_device_error() == rlt.DEVERR_BAD_SLOT
    with pytest.raises(rlt.RltError):
        rlt.rlt_kv_append_rope(pool, 0, kn, kn, pos, pos, 63, 1e4)          # odd rot_dim
