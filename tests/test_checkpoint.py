"""HF GPT-2 layout <-> nanoGPT names: the Conv1D transpose, the causal-mask buffers, the tied
lm_head and bias=False exports ("原生 nanoGPT 模型服务首选", §1 正确性; "nanoGPT 架构分析", §4.1;
"第 4 章 模型构建", §4.5).  CPU only: the conversion is host-side and runs once at load.

The HF side is pinned by its own definition, not by the reverse conversion: an HF Conv1D
computes y = x W + b with W stored (in, out), so the reference forward below is written
directly on the HF tensors with that rule and compared with the oracle on the converted ones.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from kv_cached_generation_gpt_b300 import checkpoint as ck
from kv_cached_generation_gpt_b300 import synthetic as syn
from oracle import gpt as og

SHAPES = [syn.ModelShape(2, 2, 64, 24, 97, True, "f32"), syn.ModelShape(2, 4, 128, 32, 65, False, "f32")]


def _hf_forward(sd, n_head, idx):
    """GPT-2 on HF-layout tensors in fp64: every projection is a Conv1D, y = x @ W + b."""
    t = {ck._strip(k): torch.from_numpy(np.asarray(v, np.float64)) for k, v in sd.items()}
    wte = t["wte.weight"]
    C = wte.shape[1]
    idx = torch.from_numpy(idx.astype(np.int64))
    B, T = idx.shape
    L = len({k.split(".")[1] for k in t if k.startswith("h.")})
    conv = lambda x, w, b: x @ w + b  # noqa: E731  (Conv1D)
    x = wte[idx] + t["wpe.weight"][:T]
    for l in range(L):
        g = lambda n: t[f"h.{l}.{n}"]  # noqa: E731
        h = F.layer_norm(x, (C,), g("ln_1.weight"), g("ln_1.bias"), 1e-5)
        q, k, v = conv(h, g("attn.c_attn.weight"), g("attn.c_attn.bias")).split(C, dim=2)
        q, k, v = (z.view(B, T, n_head, C // n_head).transpose(1, 2) for z in (q, k, v))
        y = F.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(1, 2).reshape(B, T, C)
        x = x + conv(y, g("attn.c_proj.weight"), g("attn.c_proj.bias"))
        h = F.layer_norm(x, (C,), g("ln_2.weight"), g("ln_2.bias"), 1e-5)
        x = x + conv(F.gelu(conv(h, g("mlp.c_fc.weight"), g("mlp.c_fc.bias"))), g("mlp.c_proj.weight"),
                     g("mlp.c_proj.bias"))
    x = F.layer_norm(x, (C,), t["ln_f.weight"], t["ln_f.bias"], 1e-5)
    return (x @ t["lm_head.weight"].T).numpy()


def _oracle(config, sd, idx):
    cfg = og.Config(config["n_layer"], config["n_head"], config["n_embd"], config["block_size"],
                    config["vocab_size"], config["bias"])
    return og.forward_full(cfg, og.weights_from_state_dict(cfg, sd), idx)


@pytest.mark.parametrize("shape", SHAPES)
def test_hf_checkpoint_converts_to_the_nanogpt_model(shape):
    sd = syn.make_weights(shape, seed=3, bias_std=0.05 if shape.bias else None, random_gamma=True)
    hf = ck.to_hf_state_dict(sd, shape.n_layer)
    # the HF layout: Conv1D (in, out), causal-mask buffers, a tied lm_head, biases always present
    assert hf["transformer.h.0.attn.c_attn.weight"].shape == (shape.n_embd, 3 * shape.n_embd)
    assert hf["transformer.h.1.mlp.c_proj.weight"].shape == (4 * shape.n_embd, shape.n_embd)
    assert "transformer.h.0.attn.bias" in hf and "lm_head.weight" in hf
    assert "transformer.h.0.ln_1.bias" in hf
    config, back = ck.from_hf_state_dict(hf, n_head=shape.n_head, drop_zero_bias=True)
    assert config == dict(n_layer=shape.n_layer, n_head=shape.n_head, n_embd=shape.n_embd,
                          block_size=shape.block_size, vocab_size=shape.vocab_size, bias=shape.bias)
    assert sorted(back) == sorted(sd)
    for k in sd:
        assert np.array_equal(back[k], sd[k]), k
    idx = syn.make_tokens(2, 11, shape.vocab_size, seed=4)
    got = _oracle(config, back, idx)
    ref = _hf_forward(hf, shape.n_head, idx)
    assert np.max(np.abs(got - ref)) < 1e-10


def test_every_conv1d_weight_is_transposed_and_nothing_else():
    """For each projection, x W_hf (the Conv1D rule) equals x W^T (nn.Linear's rule) on the
    converted weight; LayerNorm and embedding tensors come through unchanged."""
    shape = SHAPES[0]
    rng = np.random.default_rng(0)
    hf = ck.to_hf_state_dict(syn.make_weights(shape, seed=5, bias_std=0.02), shape.n_layer)
    _, sd = ck.from_hf_state_dict(hf, n_head=shape.n_head)
    for l in range(shape.n_layer):
        for name in ck.CONV1D_SUFFIXES:
            w_hf = hf[f"transformer.h.{l}.{name}"]
            x = rng.standard_normal((3, w_hf.shape[0]))
            assert np.allclose(x @ w_hf, x @ sd[f"transformer.h.{l}.{name}"].T, rtol=0, atol=1e-12)
        assert np.array_equal(hf[f"transformer.h.{l}.ln_2.weight"], sd[f"transformer.h.{l}.ln_2.weight"])
    assert np.array_equal(hf["transformer.wte.weight"], sd["transformer.wte.weight"])


def test_a_missed_transpose_is_caught_or_visible():
    """The hazard the pages name: c_attn given in nn.Linear layout is rejected by its shape; the
    square c_proj given untransposed passes the shape check but changes the logits."""
    shape = SHAPES[0]
    sd = syn.make_weights(shape, seed=7, bias_std=0.02)
    hf = ck.to_hf_state_dict(sd, shape.n_layer)
    bad = dict(hf)
    bad["transformer.h.0.attn.c_attn.weight"] = sd["transformer.h.0.attn.c_attn.weight"]
    with pytest.raises(ValueError):
        ck.from_hf_state_dict(bad, n_head=shape.n_head)
    bad = dict(hf)
    bad["transformer.h.1.attn.c_proj.weight"] = sd["transformer.h.1.attn.c_proj.weight"]
    config, conv = ck.from_hf_state_dict(bad, n_head=shape.n_head)
    idx = syn.make_tokens(1, 9, shape.vocab_size, seed=8)
    assert np.max(np.abs(_oracle(config, conv, idx) - _hf_forward(hf, shape.n_head, idx))) > 1e-6


def test_bias_false_model_exported_with_zero_biases():
    """HF has no bias switch, so a bias=False model is exported with zero biases; converting
    back with drop_zero_bias restores bias=False, and without it the zeros give bit-identical
    logits (bias=None == bias=zeros)."""
    shape = SHAPES[1]
    sd = syn.make_weights(shape, seed=9, random_gamma=True)
    hf = ck.to_hf_state_dict(sd, shape.n_layer)
    assert not np.any(hf["transformer.h.0.attn.c_attn.bias"])
    c1, nb = ck.from_hf_state_dict(hf, n_head=shape.n_head, drop_zero_bias=True)
    c2, zb = ck.from_hf_state_dict(hf, n_head=shape.n_head)
    assert c1["bias"] is False and c2["bias"] is True
    idx = syn.make_tokens(2, 13, shape.vocab_size, seed=10)
    assert np.array_equal(_oracle(c1, nb, idx), _oracle(c2, zb, idx))


def test_rejects_untied_head_unknown_keys_and_missing_layers():
    shape = SHAPES[0]
    hf = ck.to_hf_state_dict(syn.make_weights(shape, seed=1, bias_std=0.02), shape.n_layer)
    untied = dict(hf)
    untied["lm_head.weight"] = hf["lm_head.weight"] + 1.0
    with pytest.raises(ValueError):
        ck.from_hf_state_dict(untied)
    extra = dict(hf)
    extra["transformer.h.0.attn.rotary"] = np.zeros(4, np.float32)
    with pytest.raises(ValueError):
        ck.from_hf_state_dict(extra)
    gap = {k: v for k, v in hf.items() if not k.startswith("transformer.h.0.")}
    with pytest.raises(ValueError):
        ck.from_hf_state_dict(gap)
    # without the "transformer." prefix, and with torch tensors, the result is the same
    bare = {k[len("transformer."):] if k.startswith("transformer.") else k: torch.from_numpy(v)
            for k, v in hf.items()}
    c_a, a = ck.from_hf_state_dict(hf, n_head=2)
    c_b, b = ck.from_hf_state_dict(bare, n_head=2)
    assert c_a == c_b and all(np.array_equal(a[k], b[k]) for k in a)
