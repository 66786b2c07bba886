"""Pins of the oracle's position-keyed latent noise against things other than itself.

vllm-rlt PR #152 (Summary, para 2; Tests): the latent state a token starts
from depends only on (request seed, position, channel), hashed by SplitMix64
steps down to 24 uniform bits and mapped by the inverse CDF of a normal with
std = initializer_range, cut off at +-3 sigma.  The PR's CPU suite is said to
check that the draws do not depend on the batch, follow seed and position, do
not alias seed and channel, and have the cut-off normal's moments and tail
mass; those checks, the published SplitMix64 outputs and library/closed-form
values of the truncated normal pin the oracle here.
"""
import math
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle

GAMMA = 0x9E3779B97F4A7C15
M64 = 2**64 - 1
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64.txt")
SIGMA = 0.02
TWO24 = 1 << 24


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                s, i, v = line.split()
                rows.append((int(s), int(i), int(v)))
    return rows


def test_splitmix64_published_outputs():
    # Output i of a SplitMix64 generator seeded with s mixes the state s + (i+1)*gamma;
    # one stage folds its key into the state and adds gamma before mixing, so
    # stage(0, s + i*gamma) is output i.
    rows = _golden()
    assert len(rows) >= 8
    for s, i, v in rows:
        assert oracle.mix64((s + (i + 1) * GAMMA) & M64) == v
        assert oracle.stage(0, (s + i * GAMMA) & M64) == v


def test_stage_is_keyed_by_xor_into_state():
    # stage(h, x) depends on h and x only through h ^ x (a state folded with a key)
    rng = np.random.default_rng(1)
    for _ in range(50):
        h, x, y = (int(v) for v in rng.integers(0, 2**64, size=3, dtype=np.uint64))
        assert oracle.stage(h, x) == oracle.stage(h ^ y, x ^ y)


def test_key_chains_seed_then_position_then_channel():
    rng = np.random.default_rng(2)
    for _ in range(50):
        s = int(rng.integers(0, 2**64, dtype=np.uint64))
        p = int(rng.integers(0, 1 << 40))
        c = int(rng.integers(0, 8192))
        h = oracle.stage(oracle.stage(oracle.stage(0, s), p), c)
        assert oracle.noise_key(s, p, c) == h
        # the first stage of the chain is a SplitMix64 generator seeded with the seed
        assert oracle.stage(0, s) == oracle.mix64((s + GAMMA) & M64)


def test_hash24_is_top_24_bits_of_key():
    seeds = np.array([0, 1, 2**64 - 1, 12345], np.uint64)
    pos = np.array([0, 7, 2**40, 3], np.int64)
    h = oracle.noise_hash24(seeds, pos, 5)
    for r in range(4):
        for c in range(5):
            assert int(h[r, c]) == oracle.noise_key(int(seeds[r]), int(pos[r]), c) >> 40
    assert h.max() < TWO24


def test_batch_independence_and_chunking():
    # same (seed, pos, ch) -> same bits, whatever else shares the call and in whatever order
    keys_s = np.array([5, 5, 9, 1 << 63, 5], np.uint64)
    keys_p = np.array([0, 1, 1, 77, 0], np.int64)
    full = oracle.noise_hash24(keys_s, keys_p, 33)
    for r in range(5):
        alone = oracle.noise_hash24(keys_s[r:r + 1], keys_p[r:r + 1], 33)
        assert np.array_equal(alone[0], full[r])
    perm = np.array([3, 0, 4, 2, 1])
    assert np.array_equal(oracle.noise_hash24(keys_s[perm], keys_p[perm], 33), full[perm])
    assert np.array_equal(full[0], full[4])
    # prefill in chunks of 2 and of 8 tokens gives what one pass gives
    seeds = np.full(24, 42, np.uint64)
    pos = np.arange(24, dtype=np.int64)
    one = oracle.latent_noise_init(seeds, pos, 16, SIGMA)
    for chunk in (2, 8):
        parts = [oracle.latent_noise_init(seeds[i:i + chunk], pos[i:i + chunk], 16, SIGMA)
                 for i in range(0, 24, chunk)]
        assert np.array_equal(np.concatenate(parts), one)


def test_prefix_cache_hit_draws_same_suffix_noise():
    # a cached run prefills only positions k.. of the prompt; its noise equals the cold run's
    seeds = np.full(40, 7, np.uint64)
    pos = np.arange(40, dtype=np.int64)
    cold = oracle.noise_hash24(seeds, pos, 64)
    warm = oracle.noise_hash24(seeds[25:], pos[25:], 64)
    assert np.array_equal(cold[25:], warm)


def test_seed_position_channel_keying():
    rng = np.random.default_rng(3)
    n = 20000
    s = rng.integers(0, 2**64, size=n, dtype=np.uint64)
    p = rng.integers(0, 1 << 20, size=n).astype(np.int64)
    base = oracle.noise_hash24(s, p, 2)
    # change one component at a time: each changes h24 except for ~2^-24 coincidences
    other_seed = oracle.noise_hash24(s ^ np.uint64(1), p, 2)
    other_pos = oracle.noise_hash24(s, p + 1, 2)
    assert (other_seed[:, 0] == base[:, 0]).sum() <= 2
    assert (other_pos[:, 0] == base[:, 0]).sum() <= 2
    assert (base[:, 1] == base[:, 0]).sum() <= 2


def test_no_seed_channel_aliasing():
    # (s+1, c-1) must not reproduce (s, c), and swapping seed and channel gives a new value
    rng = np.random.default_rng(4)
    n = 4000
    s = rng.integers(1, 1 << 12, size=n)
    c = rng.integers(1, 1 << 12, size=n)
    p = rng.integers(0, 1 << 16, size=n)
    a = np.array([oracle.noise_key(int(s[i]), int(p[i]), int(c[i])) >> 40 for i in range(n)], np.float64)
    b = np.array([oracle.noise_key(int(s[i]) + 1, int(p[i]), int(c[i]) - 1) >> 40 for i in range(n)], np.float64)
    w = np.array([oracle.noise_key(int(c[i]), int(p[i]), int(s[i])) >> 40 for i in range(n)], np.float64)
    assert (a == b).sum() <= 1
    assert (a == w)[s != c].sum() <= 1
    r = np.corrcoef(a, b)[0, 1]
    assert abs(r) < 5 / math.sqrt(n)


def test_h24_is_uniform():
    seeds = np.repeat(np.arange(64, dtype=np.uint64), 64)
    pos = np.tile(np.arange(64, dtype=np.int64), 64)
    h = oracle.noise_hash24(seeds, pos, 64).ravel()          # 2^18 draws
    counts = np.bincount(h >> 16, minlength=256)                 # top 8 bits
    chi2 = ((counts - h.size / 256) ** 2 / (h.size / 256)).sum()
    assert chi2 < stats.chi2.ppf(1 - 1e-6, 255)
    assert abs(h.mean() / TWO24 - 0.5) < 5 * math.sqrt(1 / 12 / h.size)


# ---------------------------------------------------------- inverse CDF map

def _library_value(h24):
    """scipy's ndtri/ndtr form of the truncated-normal inverse CDF at the cell midpoint."""
    u = (np.asarray(h24, np.float64) + 0.5) / TWO24
    lo, hi = special.ndtr(-3.0), special.ndtr(3.0)
    return SIGMA * special.ndtri(lo + u * (hi - lo))


def _erfinv_value(h24):
    """The same quantity as sigma*sqrt(2)*erfinv((2u-1) erf(3/sqrt 2)), via scipy.special.erfinv."""
    u = (np.asarray(h24, np.float64) + 0.5) / TWO24
    return SIGMA * math.sqrt(2.0) * special.erfinv((2 * u - 1) * special.erf(3 / math.sqrt(2.0)))


def test_inverse_cdf_matches_library_routines():
    rng = np.random.default_rng(5)
    h = np.concatenate([[0, 1, 2, 1000, (1 << 23) - 1, 1 << 23, (1 << 23) + 1,
                         TWO24 - 1001, TWO24 - 2, TWO24 - 1],
                        rng.integers(0, TWO24, 3000)]).astype(np.uint32)
    got = oracle.noise_values(h, SIGMA)
    np.testing.assert_allclose(got, _library_value(h), rtol=0, atol=1e-14)
    np.testing.assert_allclose(got, _erfinv_value(h), rtol=0, atol=1e-13)


def test_inverse_cdf_special_points():
    # u = 1/2 +- half a cell straddles 0; the map is odd about the middle of the grid
    assert abs(oracle.noise_value(1 << 23, SIGMA)) < 1e-8
    assert oracle.noise_value((1 << 23) - 1, SIGMA) < 0 < oracle.noise_value(1 << 23, SIGMA)
    rng = np.random.default_rng(6)
    for h in rng.integers(0, TWO24, 200):
        a = oracle.noise_value(int(h), SIGMA)
        b = oracle.noise_value(TWO24 - 1 - int(h), SIGMA)
        assert abs(a + b) < 1e-15
    # extremes stay inside the +-3 sigma truncation, and only just
    top = oracle.noise_value(TWO24 - 1, SIGMA)
    assert 2.9 * SIGMA < top < 3 * SIGMA
    # linear in sigma
    assert abs(oracle.noise_value(12345, 1.0) * 0.02 - oracle.noise_value(12345, 0.02)) < 1e-16


def test_inverse_cdf_monotone_on_grid_samples():
    h = np.sort(np.random.default_rng(7).choice(TWO24, 4000, replace=False)).astype(np.uint32)
    x = oracle.noise_values(h, SIGMA)
    assert np.all(np.diff(x) > 0)


@pytest.mark.parametrize("t", [1.0, 2.0, 2.5])
def test_tail_boundaries(t):
    # the cell where x crosses -t sigma: the fraction of cells below is
    # (Phi(-t) - Phi(-3)) / (Phi(3) - Phi(-3)), the truncated normal's CDF at -t
    frac = (stats.norm.cdf(-t) - stats.norm.cdf(-3)) / (stats.norm.cdf(3) - stats.norm.cdf(-3))
    k = int(math.floor(frac * TWO24 - 0.5))   # last cell whose midpoint lies below
    assert oracle.noise_value(k, SIGMA) < -t * SIGMA <= oracle.noise_value(k + 1, SIGMA)
    assert -oracle.noise_value(TWO24 - 1 - k, SIGMA) < -t * SIGMA


def test_truncated_normal_moments_by_quadrature():
    # midpoint rule over 2^16 equal strata of the 2^24 cells: the grid's moments
    # approach the truncated normal's closed forms
    n = 1 << 16
    stride = TWO24 // n
    h = (np.arange(n, dtype=np.int64) * stride + stride // 2).astype(np.uint32)
    z = oracle.noise_values(h, 1.0)
    a = 3.0
    Z = stats.norm.cdf(a) - stats.norm.cdf(-a)
    var = 1 - 2 * a * stats.norm.pdf(a) / Z
    m4 = 3 - (2 * a**3 + 6 * a) * stats.norm.pdf(a) / Z
    assert abs(z.mean()) < 1e-6
    assert abs((z**2).mean() - var) < 2e-5
    assert abs((z**4).mean() - m4) < 2e-4
    for t in (1.0, 2.0, 2.5):
        tail = (stats.norm.sf(t) - stats.norm.sf(a)) * 2 / Z
        assert abs((np.abs(z) > t).mean() - tail) < 2 / n
    assert abs(math.sqrt(var) - 0.98657839) < 1e-8      # std of N(0,1) truncated at +-3


def test_noise_sample_moments_through_the_hash():
    # 2^16 keyed draws: the whole pipeline (hash -> 24-bit uniform -> inverse CDF)
    rows = 256
    seeds = np.arange(rows, dtype=np.uint64) * np.uint64(0x1000193)
    pos = np.arange(rows, dtype=np.int64) * 3
    x = oracle.latent_noise_init(seeds, pos, 256, SIGMA).ravel() / SIGMA
    a = 3.0
    Z = stats.norm.cdf(a) - stats.norm.cdf(-a)
    var = 1 - 2 * a * stats.norm.pdf(a) / Z
    m4 = 3 - (2 * a**3 + 6 * a) * stats.norm.pdf(a) / Z
    n = x.size
    assert abs(x.mean()) < 5 * math.sqrt(var / n)
    assert abs((x**2).mean() - var) < 5 * math.sqrt((m4 - var**2) / n)
    p1 = (stats.norm.sf(1) - stats.norm.sf(a)) * 2 / Z
    assert abs((np.abs(x) > 1).mean() - p1) < 5 * math.sqrt(p1 * (1 - p1) / n)
    assert np.abs(x).max() < 3.0
