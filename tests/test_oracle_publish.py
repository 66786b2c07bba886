"""Pins for the oracle's written-prefix counters and prefix-publication coverage.

vllm-rlt PR #152 (Summary; Tests): publication used to require a contiguous
written prefix in every layer of every plane, which a partially looped model
(Huginn: prelude and coda layers on plane 0 only) never has; coverage is now
checked per plane over the layers that plane holds, fully looped models are
unchanged, and "publication covers only the layers each plane holds".  Checked
by brute force over all (layer, plane) pairs on small cases.
"""
import numpy as np

import oracle


def brute_publishable(recurrent, num_planes, written_by_layer_plane, page_size):
    """Min written length over the (layer, plane) pairs the model holds, in whole pages."""
    L = len(recurrent)
    out = []
    for b in range(written_by_layer_plane.shape[2]):
        lens = [written_by_layer_plane[l, t, b] for l in range(L) for t in range(num_planes)
                if t == 0 or recurrent[l]]
        out.append(min(lens) // page_size * page_size if lens else 0)
    return np.array(out, np.int32)


def test_huginn_publishes_once_every_held_bank_has_written():
    recurrent = [0, 0, 1, 1, 1, 1, 0, 0]                  # 2 prelude, 4 recurrent, 2 coda
    T, B, ps = 32, 5, 16
    bmap, nbanks = oracle.bank_map(recurrent, T)
    assert nbanks == 132
    rng = np.random.default_rng(0)
    full = rng.integers(0, 3000, size=B)
    per_lp = np.zeros((8, T, B), np.int32)
    written = np.zeros((nbanks, B), np.int32)
    for l in range(8):
        for t in range(T):
            if bmap[l, t] >= 0:
                lens = np.maximum(full - rng.integers(0, 40, size=B), 0)
                per_lp[l, t] = lens
                written[bmap[l, t]] = lens
    got = oracle.publishable_prefix(bmap, written, ps)
    assert np.array_equal(got, brute_publishable(recurrent, T, per_lp, ps))
    assert np.all(got > 0)
    # the rule before the fix asked every layer of every plane; prelude and coda layers
    # never write deeper planes, so nothing would ever publish
    old = [min(per_lp[l, t, b] for l in range(8) for t in range(T)) for b in range(B)]
    assert all(v == 0 for v in old)


def test_fully_looped_model_needs_every_bank():
    recurrent = [1] * 6
    T, B, ps = 4, 3, 64
    bmap, nbanks = oracle.bank_map(recurrent, T)
    written = np.full((nbanks, B), 1000, np.int32)
    assert np.array_equal(oracle.publishable_prefix(bmap, written, ps), [960] * B)
    written[bmap[5, 3], 1] = 300                          # one layer-plane behind for request 1
    assert np.array_equal(oracle.publishable_prefix(bmap, written, ps), [960, 256, 960])
    written[bmap[0, 0], 2] = 0
    assert oracle.publishable_prefix(bmap, written, ps)[2] == 0


def test_no_bank_publishes_nothing():
    bmap = np.full((2, 2), -1, np.int32)
    assert np.array_equal(oracle.publishable_prefix(bmap, np.zeros((0, 3), np.int32), 16), [0, 0, 0])


def test_mark_written_advances_to_the_furthest_appended_position():
    written = np.zeros((3, 4), np.int32)
    # a prefill chunk of request 2 (positions 0..99) and decode tokens of requests 0 and 1
    req = np.array([2] * 100 + [0, 1], np.int32)
    pos = np.array(list(range(100)) + [7, 41], np.int64)
    loc = np.arange(102, dtype=np.int64)
    loc[50] = -1                                         # a skipped slot leaves no mark by itself
    oracle.mark_written(written, 1, req, pos, loc)
    assert written[1].tolist() == [8, 42, 100, 0]
    assert np.all(written[0] == 0) and np.all(written[2] == 0)
    oracle.mark_written(written, 1, np.array([2], np.int32), np.array([10]), np.array([5]))
    assert written[1, 2] == 100                          # never moves back
