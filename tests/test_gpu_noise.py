"""GPU parity of the position-keyed latent noise (vllm-rlt PR #152, Summary para 2).

Bar: the 24-bit uniforms bit-exact against the oracle's hash; fp32 values within
1e-6 absolute of the oracle's fp64 truncated-normal inverse CDF.
"""
import numpy as np
import pytest

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from helpers import NOISE_ABS, i64_dev

pytestmark = pytest.mark.gpu


def run(seeds, positions, channels, sigma, device):
    s = i64_dev(np.asarray(seeds, np.uint64), device)
    p = i64_dev(positions, device)
    h = rlt.rlt_noise_hash24(s, p, channels)
    x = rlt.rlt_latent_noise_init(s, p, channels, sigma)
    return h.cpu().numpy().view(np.uint32), x.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "huginn"])
def test_workload_noise_matches_oracle(cuda_device, name):
    nz = W.config(name).noise
    h, x = run(nz.seeds, nz.positions, nz.channels, nz.initializer_range, cuda_device)
    assert np.array_equal(h, oracle.noise_hash24(nz.seeds, nz.positions, nz.channels))
    ref = oracle.latent_noise_init(nz.seeds, nz.positions, nz.channels, nz.initializer_range)
    assert np.abs(x - ref).max() <= NOISE_ABS
    assert rlt.rlt_get_device_error() == 0


def test_bulk_noise_full_size_sampled(cuda_device):
    # 2^24 draws in one launch (64 seeds x 64 positions x 4096 channels); the
    # hash is checked on every value, the inverse CDF on a sample of rows
    nz = W.config("longctx").noise
    assert nz.rows * nz.channels == 1 << 24
    h, x = run(nz.seeds, nz.positions, nz.channels, nz.initializer_range, cuda_device)
    assert np.array_equal(h, oracle.noise_hash24(nz.seeds, nz.positions, nz.channels))
    rows = np.random.default_rng(0).choice(nz.rows, 24, replace=False)
    ref = oracle.latent_noise_init(nz.seeds[rows], nz.positions[rows], nz.channels, nz.initializer_range)
    assert np.abs(x[rows] - ref).max() <= NOISE_ABS
    # tails: the extreme cells of the grid, wherever they occur
    lo, hi = h == h.min(), h == h.max()
    assert np.abs(x[lo] - oracle.noise_value(int(h.min()), 0.02)).max() <= NOISE_ABS
    assert np.abs(x[hi] - oracle.noise_value(int(h.max()), 0.02)).max() <= NOISE_ABS
    assert np.abs(x).max() < 3 * 0.02


@pytest.mark.parametrize("channels", [1, 3, 5, 8, 13, 64, 100])
def test_ragged_channel_counts(cuda_device, channels):
    nz = W.noise_keys(37, channels, seed=channels)
    h, x = run(nz.seeds, nz.positions, channels, 0.05, cuda_device)
    assert np.array_equal(h, oracle.noise_hash24(nz.seeds, nz.positions, channels))
    ref = oracle.latent_noise_init(nz.seeds, nz.positions, channels, 0.05)
    assert np.abs(x - ref).max() <= 2.5 * NOISE_ABS    # sigma 0.05: 2.5x the 0.02 scale


def test_batch_independence_on_gpu(cuda_device):
    nz = W.noise_keys(64, 256, seed=3)
    h_all, x_all = run(nz.seeds, nz.positions, 256, 0.02, cuda_device)
    perm = np.random.default_rng(1).permutation(64)
    h_p, x_p = run(nz.seeds[perm], nz.positions[perm], 256, 0.02, cuda_device)
    assert np.array_equal(h_p, h_all[perm]) and np.array_equal(x_p, x_all[perm])
    h_one, x_one = run(nz.seeds[7:8], nz.positions[7:8], 256, 0.02, cuda_device)
    assert np.array_equal(h_one[0], h_all[7]) and np.array_equal(x_one[0], x_all[7])


def test_extreme_keys(cuda_device):
    seeds = np.array([0, 2**64 - 1, 2**63, 1], np.uint64)
    pos = np.array([0, 2**62, -1, 2**31], np.int64)
    h, x = run(seeds, pos, 16, 0.02, cuda_device)
    assert np.array_equal(h, oracle.noise_hash24(seeds, pos, 16))
    assert np.abs(x - oracle.latent_noise_init(seeds, pos, 16, 0.02)).max() <= NOISE_ABS


def test_empty_is_a_no_op(cuda_device):
    import torch
    s = torch.zeros(0, dtype=torch.int64, device=cuda_device)
    out = rlt.rlt_latent_noise_init(s, s, 64, 0.02)
    assert out.shape == (0, 64)
