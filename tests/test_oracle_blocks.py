"""Pins of the oracle's building blocks against library routines and closed forms.

The oracle computes with numpy/scipy; every pin here comes from somewhere else:
torch's own layer_norm / gelu / scaled_dot_product_attention (fp64, CPU), exact
special cases, or invariants of the definitions.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import gpt as og

RNG = np.random.default_rng(7)


def _t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


@pytest.mark.parametrize("with_bias", [False, True])
def test_layer_norm_matches_torch(with_bias):
    x = RNG.standard_normal((5, 7, 96)) * 3 + 1.5
    w = 1 + 0.1 * RNG.standard_normal(96)
    b = 0.2 * RNG.standard_normal(96) if with_bias else None
    got = og.layer_norm(x, w, b)
    ref = F.layer_norm(_t(x), (96,), _t(w), None if b is None else _t(b), eps=1e-5).numpy()
    assert np.max(np.abs(got - ref)) < 1e-12


def test_layer_norm_invariants():
    x = RNG.standard_normal((4, 256)) * 5 + 3
    y = og.layer_norm(x, np.ones(256), None)
    assert np.max(np.abs(y.mean(-1))) < 1e-12
    # biased variance with eps: var(y) = var / (var + eps)
    var = x.var(-1)
    assert np.allclose(y.var(-1), var / (var + 1e-5), rtol=1e-12, atol=0)
    # a constant row normalises to zero (x - mu = 0 exactly), then beta is added
    c = np.full((1, 64), 2.5)
    beta = RNG.standard_normal(64)
    assert np.array_equal(og.layer_norm(c, np.ones(64), beta), beta[None, :])


def test_gelu_matches_torch_and_limits():
    z = np.concatenate([np.linspace(-8, 8, 4001), RNG.standard_normal(1000) * 3])
    ref = F.gelu(_t(z), approximate="none").numpy()
    assert np.max(np.abs(og.gelu(z) - ref)) < 1e-14
    assert og.gelu(np.array([0.0]))[0] == 0.0
    assert og.gelu(np.array([40.0]))[0] == 40.0
    assert og.gelu(np.array([-40.0]))[0] == 0.0
    # the tanh approximation differs from the exact form by ~1e-4: the pin tells them apart
    tanh_form = F.gelu(_t(z), approximate="tanh").numpy()
    assert np.max(np.abs(og.gelu(z) - tanh_form)) > 1e-5


@pytest.mark.parametrize("T", [1, 5, 33])
def test_attention_matches_sdpa_causal(T):
    q, k, v = (RNG.standard_normal((2, 3, T, 16)) for _ in range(3))
    got = og.attention(q, k, v, q_pos0=0)
    ref = F.scaled_dot_product_attention(_t(q), _t(k), _t(v), is_causal=True).numpy()
    assert np.max(np.abs(got - ref)) < 1e-12


def test_attention_offset_mask_matches_sdpa_with_explicit_mask():
    # 3 new queries after a cache of 6 keys: query i sits at position 6+i.
    c, Tq = 6, 3
    q = RNG.standard_normal((1, 2, Tq, 8))
    k, v = (RNG.standard_normal((1, 2, c + Tq, 8)) for _ in range(2))
    allowed = np.arange(c + Tq)[None, :] <= (c + np.arange(Tq))[:, None]
    ref = F.scaled_dot_product_attention(_t(q), _t(k), _t(v), attn_mask=torch.from_numpy(allowed)).numpy()
    assert np.max(np.abs(og.attention(q, k, v, q_pos0=c) - ref)) < 1e-12


def test_attention_special_cases():
    # one key: softmax over one entry is 1, so y = v exactly
    q, k, v = (RNG.standard_normal((2, 2, 1, 8)) for _ in range(3))
    assert np.array_equal(og.attention(q, k, v, 0), v)
    # equal keys: uniform weights over the visible prefix, so y_i = mean(v_0..v_i)
    T = 9
    q = RNG.standard_normal((1, 1, T, 8))
    k = np.repeat(RNG.standard_normal((1, 1, 1, 8)), T, axis=2)
    v = RNG.standard_normal((1, 1, T, 8))
    prefix_mean = np.cumsum(v, axis=2) / np.arange(1, T + 1)[None, None, :, None]
    assert np.max(np.abs(og.attention(q, k, v, 0) - prefix_mean)) < 1e-13
    # softmax rows sum to one: with v = 1 every output is 1
    q, k = (RNG.standard_normal((2, 3, 17, 8)) * 4 for _ in range(2))
    ones = np.ones((2, 3, 17, 8))
    assert np.max(np.abs(og.attention(q, k, ones, 0) - 1.0)) < 1e-12
    # first query sees only the first key, whatever the rest hold
    v = RNG.standard_normal((2, 3, 17, 8))
    assert np.max(np.abs(og.attention(q, k, v, 0)[:, :, 0] - v[:, :, 0])) < 1e-15


def test_scale_is_inverse_sqrt_head_size():
    # two keys, one query: weight ratio is exp((q.k0 - q.k1)/sqrt(hs))
    hs = 64
    q = RNG.standard_normal((1, 1, 1, hs))
    k = RNG.standard_normal((1, 1, 2, hs))
    v = np.zeros((1, 1, 2, hs))
    v[..., 0, 0] = 1.0
    v[..., 1, 1] = 1.0
    y = og.attention(q, k, v, q_pos0=1)[0, 0, 0]
    d = float(q[0, 0, 0] @ (k[0, 0, 0] - k[0, 0, 1])) / math.sqrt(hs)
    assert abs(y[0] / y[1] - math.exp(d)) < 1e-12 * math.exp(abs(d))
