"""Pins of the sampler oracle: numpy's Philox, double-precision exp, exact special
cases of top-k, and the empirical distribution of draws (chi-square)."""
import math

import numpy as np
import pytest
from scipy import stats

from kv_cached_generation_gpt_b300 import synthetic as syn
from oracle import sampler as S

MASK = (1 << 64) - 1


@pytest.mark.parametrize("seed,row,step", [(0, 0, 0), (1337, 3, 1), (2**64 - 1, 63, 512), (42, 7, 2**40)])
def test_philox_matches_numpy_bit_generator(seed, row, step):
    # numpy's Philox increments its 256-bit counter before producing a block, so start one below.
    c = step - 1
    ctr = np.array([c & MASK] + ([0, 0, 0] if c >= 0 else [MASK, MASK, MASK]), dtype=np.uint64)
    g = np.random.Philox(counter=ctr, key=np.array([seed, row], dtype=np.uint64))
    want = [int(x) for x in g.random_raw(4)]
    assert S.philox4x64_10((step, 0, 0, 0), (seed, row)) == want


def test_gexp_within_two_ulp_of_exp():
    x = np.unique(np.concatenate([
        np.linspace(-64, 0, 400_001, dtype=np.float32),
        -np.abs(np.random.default_rng(1).standard_normal(200_000).astype(np.float32)) * 4,
    ]))
    got = S.gexp(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(got - ref) / ulp) <= 2.0
    assert S.gexp(np.float32(0.0)) == 1.0
    assert S.gexp(np.float32(-np.inf)) == 0.0
    assert S.gexp(np.float32(-64.5)) == 0.0
    assert np.all(np.diff(got) >= 0)  # monotone on the sorted sweep


def test_top_k_one_is_argmax():
    logits = syn.make_logits(4, 300, seed=3)
    for step in range(20):
        got = S.sample(logits, 0.7, 1, seed=step, step=step)
        assert np.array_equal(got, np.argmax(logits, axis=1))


def test_top_k_at_least_vocab_is_no_mask():
    logits = syn.make_logits(3, 65, seed=4)
    for step in range(10):
        a = S.sample(logits, 0.8, 200, seed=9, step=step)
        b = S.sample(logits, 0.8, None, seed=9, step=step)
        c = S.sample(logits, 0.8, 65, seed=9, step=step)
        assert np.array_equal(a, b) and np.array_equal(a, c)


def test_top_k_keeps_ties_with_kth_value():
    s = np.array([0.5, 2.0, 1.0, 1.0, 1.0, -3.0, 1.0], np.float32)
    keep = S.survivors(s, 2)
    # 2nd largest is 1.0; every 1.0 survives, so 5 survivors for k = 2
    assert keep.tolist() == [False, True, True, True, True, False, True]
    assert S.topk_threshold(s, 2) == np.float32(1.0)
    assert S.survivors(s, 1).sum() == 1


def test_masked_entries_never_drawn():
    logits = syn.make_logits(2, 1000, seed=5, std=0.1)  # flat: masked ones would be likely
    for step in range(200):
        tok = S.sample(logits, 1.0, 50, seed=1, step=step)
        for b in range(2):
            s = S.scaled_logits(logits[b], 1.0)
            assert s[tok[b]] >= S.topk_threshold(s, 50)


def test_greedy_temperature_zero_lowest_index_on_ties():
    logits = np.array([[1.0, 3.0, 3.0, 2.0]], np.float32)
    assert S.sample(logits, 0.0, None, seed=0, step=0)[0] == 1


def test_pick_boundaries():
    w = np.array([0, 5, 0, 3, 2, 0], np.uint64)  # W = 10
    assert S.pick(w, 0) == 1  # target 0
    assert S.pick(w, MASK) == 4  # target W-1 = 9
    # target = floor(r W / 2^64): every integer target in [0, W) maps to the interval holding it
    for target in range(10):
        r = -(-(target << 64) // 10)  # smallest r with floor(r*10/2^64) == target
        want = 1 if target < 5 else (3 if target < 8 else 4)
        assert S.pick(w, r) == want


def test_integer_weights_exact_and_bounded():
    s = np.array([0.0, -1.0, -30.0, -64.0, -100.0], np.float32)
    w = S.integer_weights(s, np.ones(5, bool))
    assert w[0] == 2**40
    assert w[1] == math.floor(float(S.gexp(np.float32(-1.0))) * 2**40)
    assert w[2] == 0 and w[3] == 0 and w[4] == 0  # e^-30 < 2^-40


def test_draws_follow_softmax_chi_square():
    logits = np.array([[0.3, -1.2, 2.0, 0.0, 1.1, -0.4, 0.9, 1.7]], np.float32)
    T, k = 0.9, 5
    n = 40_000
    counts = np.zeros(8)
    for step in range(n):
        counts[S.sample(logits, T, k, seed=2024, step=step)[0]] += 1
    s = logits[0].astype(np.float64) / T
    keep = s >= np.sort(s)[::-1][k - 1]
    p = np.where(keep, np.exp(s - s.max()), 0.0)
    p /= p.sum()
    assert counts[~keep].sum() == 0
    chi2, pval = stats.chisquare(counts[keep], n * p[keep])
    assert pval > 1e-4, (chi2, pval)


def test_rows_use_independent_streams():
    logits = np.zeros((2, 64), np.float32)  # uniform over 64
    a = np.array([S.sample(logits, 1.0, None, seed=77, step=t) for t in range(300)])
    assert np.mean(a[:, 0] == a[:, 1]) < 0.1
    # same row, same seed and step -> same draw
    assert S.sample(logits, 1.0, None, 77, 5)[0] == S.sample(logits, 1.0, None, 77, 5)[0]
