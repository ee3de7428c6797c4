"""Pins of the oracle's whole-model forward: invariants the pages fix, a closed form,
the pages' parameter counts, and torch's own modules run in fp64 (a library pin)."""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from kv_cached_generation_gpt_b300 import synthetic as syn
from oracle import gpt as og

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "param_counts.json")


def _cfg(shape):
    return og.Config(shape.n_layer, shape.n_head, shape.n_embd, shape.block_size, shape.vocab_size, shape.bias)


def _model(shape, seed=11, bias_std=None, random_gamma=False):
    sd = syn.make_weights(shape, seed=seed, bias_std=bias_std, random_gamma=random_gamma)
    return _cfg(shape), og.weights_from_state_dict(_cfg(shape), sd), sd


TOY = syn.ModelShape(2, 2, 32, 24, 50, False, "f32")
TOY_BIAS = syn.ModelShape(2, 4, 64, 24, 97, True, "f32")


# ------------------------------------------------------------- library pin: torch modules, fp64


def _torch_forward(shape, sd, idx):
    """nanoGPT's forward written with torch.nn.functional (fp64): F.embedding, F.layer_norm,
    F.linear with nn.Linear's (out, in) weights, scaled_dot_product_attention(is_causal=True),
    F.gelu(approximate='none'), and the lm_head as F.linear with the wte matrix."""
    C, nh = shape.n_embd, shape.n_head
    t = {k: torch.from_numpy(v.astype(np.float64)) for k, v in sd.items()}
    idx = torch.from_numpy(idx.astype(np.int64))
    B, T = idx.shape
    x = F.embedding(idx, t["transformer.wte.weight"]) + t["transformer.wpe.weight"][:T]
    for l in range(shape.n_layer):
        g = lambda n: t.get(f"transformer.h.{l}.{n}")
        h = F.layer_norm(x, (C,), g("ln_1.weight"), g("ln_1.bias"), 1e-5)
        q, k, v = F.linear(h, g("attn.c_attn.weight"), g("attn.c_attn.bias")).split(C, dim=2)
        q, k, v = (z.view(B, T, nh, C // nh).transpose(1, 2) for z in (q, k, v))
        y = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        y = y.transpose(1, 2).contiguous().view(B, T, C)
        x = x + F.linear(y, g("attn.c_proj.weight"), g("attn.c_proj.bias"))
        h = F.layer_norm(x, (C,), g("ln_2.weight"), g("ln_2.bias"), 1e-5)
        h = F.gelu(F.linear(h, g("mlp.c_fc.weight"), g("mlp.c_fc.bias")), approximate="none")
        x = x + F.linear(h, g("mlp.c_proj.weight"), g("mlp.c_proj.bias"))
    x = F.layer_norm(x, (C,), t["transformer.ln_f.weight"], t.get("transformer.ln_f.bias"), 1e-5)
    return F.linear(x, t["transformer.wte.weight"]).numpy()


@pytest.mark.parametrize("shape,bias_std", [(TOY, None), (TOY_BIAS, 0.05), (syn.TINY, None)])
def test_forward_matches_torch_modules(shape, bias_std):
    cfg, w, sd = _model(shape, bias_std=bias_std, random_gamma=True)
    idx = syn.make_tokens(2, min(17, shape.block_size), shape.vocab_size, seed=5)
    got = og.forward_full(cfg, w, idx)
    ref = _torch_forward(shape, sd, idx)
    assert got.shape == ref.shape
    assert np.max(np.abs(got - ref)) < 1e-10


# ------------------------------------------------------------- invariants the pages fix


def test_kv_cache_equals_full_recompute():
    """Cached decode gives the no-cache last-position logits (the KV-cache sketch)."""
    cfg, w, _ = _model(TOY_BIAS, bias_std=0.05, random_gamma=True)
    idx = syn.make_tokens(3, 20, cfg.vocab_size, seed=9)
    full = og.forward_full(cfg, w, idx)
    logits, cache = og.prefill(cfg, w, idx[:, :7])
    assert np.max(np.abs(logits - full[:, 6])) < 1e-12
    for t in range(7, 20):
        logits, cache = og.decode(cfg, w, cache, idx[:, t])
        assert np.max(np.abs(logits - full[:, t])) < 1e-11
    assert cache[0][0].shape == (3, cfg.n_head, 20, cfg.head_size)
    # a multi-token append onto a cache (offset causal mask) equals the full pass too
    logits, cache = og.prefill(cfg, w, idx[:, :5])
    chunk, _ = og.forward(cfg, w, idx[:, 5:12], cache, all_positions=True)
    assert np.max(np.abs(chunk - full[:, 5:12])) < 1e-11


def test_causal_mask_future_tokens_do_not_change_past_logits():
    cfg, w, _ = _model(TOY, random_gamma=True)
    idx = syn.make_tokens(1, 16, cfg.vocab_size, seed=3)
    base = og.forward_full(cfg, w, idx)
    for i in (0, 4, 14):
        pert = idx.copy()
        pert[:, i + 1:] = (pert[:, i + 1:] + 17) % cfg.vocab_size
        out = og.forward_full(cfg, w, pert)
        assert np.array_equal(out[:, :i + 1], base[:, :i + 1])
        if i + 1 < 16:
            assert not np.array_equal(out[:, i + 1:], base[:, i + 1:])


def test_bias_none_equals_bias_zeros():
    """LayerNorm/Linear with bias=None is the same computation as bias = zeros."""
    shape_nb = TOY
    cfg, w, sd = _model(shape_nb, random_gamma=True)
    shape_b = dataclasses.replace(shape_nb, bias=True)
    sd_zero = dict(sd)
    C = shape_nb.n_embd
    for l in range(shape_nb.n_layer):
        for name, n in (("ln_1.bias", C), ("attn.c_attn.bias", 3 * C), ("attn.c_proj.bias", C),
                        ("ln_2.bias", C), ("mlp.c_fc.bias", 4 * C), ("mlp.c_proj.bias", C)):
            sd_zero[f"transformer.h.{l}.{name}"] = np.zeros(n, np.float32)
    sd_zero["transformer.ln_f.bias"] = np.zeros(C, np.float32)
    w0 = og.weights_from_state_dict(_cfg(shape_b), sd_zero)
    assert w0.layers[0].c_attn_b is not None and w.layers[0].c_attn_b is None
    idx = syn.make_tokens(2, 11, cfg.vocab_size, seed=4)
    assert np.array_equal(og.forward_full(cfg, w, idx), og.forward_full(_cfg(shape_b), w0, idx))


def test_zero_layers_closed_form():
    """L = 0: logits = LN_f(wte[id] + wpe[pos]) wte^T, with the tied matrix."""
    shape = syn.ModelShape(0, 2, 32, 16, 40, True, "f32")
    cfg, w, _ = _model(shape, bias_std=0.1, random_gamma=True)
    idx = syn.make_tokens(1, 9, 40, seed=2)
    h = w.wte[idx[0]] + w.wpe[:9]
    mu = h.mean(-1, keepdims=True)
    sd = np.sqrt(((h - mu) ** 2).mean(-1, keepdims=True) + 1e-5)
    want = ((h - mu) / sd * w.ln_f_w + w.ln_f_b) @ w.wte.T
    assert np.max(np.abs(og.forward_full(cfg, w, idx)[0] - want)) < 1e-12


def test_lm_head_is_tied_to_wte():
    """Scaling one wte row changes that token's logit linearly (the same matrix is the head)."""
    shape = syn.ModelShape(1, 2, 32, 16, 40, False, "f32")
    cfg, w, _ = _model(shape)
    idx = np.array([[1, 2, 3]], np.int32)  # token 7 is not an input, so only its logit moves
    base = og.forward_full(cfg, w, idx)
    w.wte[7] *= 2.0
    after = og.forward_full(cfg, w, idx)
    assert np.max(np.abs(after[..., 7] - 2.0 * base[..., 7])) < 1e-12
    others = np.delete(np.arange(40), 7)
    assert np.array_equal(after[..., others], base[..., others])


def test_teacher_forced_greedy_is_self_consistent():
    cfg, w, _ = _model(syn.TINY)
    prompt = syn.make_tokens(1, 16, 65)
    fed, logits = og.teacher_forced(cfg, w, prompt, n_steps=6)
    assert logits.shape == (7, 1, 65)
    for i in range(6):
        assert fed[0, i] == np.argmax(logits[i, 0])
    full = og.forward_full(cfg, w, np.concatenate([prompt, fed], axis=1))
    assert np.max(np.abs(full[0, 15:] - logits[:, 0])) < 1e-11


def test_context_overflow_and_bad_tokens_raise():
    cfg, w, _ = _model(TOY)
    with pytest.raises(ValueError):
        og.prefill(cfg, w, np.zeros((1, cfg.block_size + 1), np.int32))
    with pytest.raises(ValueError):
        og.prefill(cfg, w, np.full((1, 3), cfg.vocab_size, np.int32))


# ------------------------------------------------------------- parameter counts printed by the pages


def _count_arrays(shape):
    sd = syn.make_weights(shape, seed=1)
    return sum(a.size for a in sd.values())


def test_param_count_formula_matches_weight_arrays():
    for shape in (TOY, TOY_BIAS, syn.TINY, syn.CHAR):
        assert og.param_count(_cfg(shape)) == _count_arrays(shape)
    assert og.param_count(_cfg(syn.GPT2_124M)) == 124_373_760
    assert og.param_count(_cfg(syn.GPT2_350M_BIAS)) == 354_823_168


def test_param_counts_printed_by_pages():
    cases = json.load(open(GOLDEN))["cases"]
    c0 = cases[0]
    lead = 12 * c0["n_layer"] * c0["n_embd"] ** 2 + c0["vocab_size"] * c0["n_embd"]
    assert round(lead / 1e6) == c0["printed_millions"]
    c1 = cases[1]
    assert math.floor(c1["n_embd"] * c1["vocab_size"] / 1e6) == c1["printed_millions"]
    c2 = cases[2]
    tied = og.Config(c2["n_layer"], 6, c2["n_embd"], c2["block_size"], c2["vocab_size"], False)
    untied_extra = c2["vocab_size"] * c2["n_embd"]  # a separate lm_head matrix
    assert math.floor(untied_extra / 1e6) == c2["printed_saving_millions"]
    # the exact count sits within the formula's leading terms plus the small LN/position terms
    assert 0 < og.param_count(tied) - lead < 0.01 * lead
    c3 = cases[3]
    cfg = og.Config(c3["n_layer"], 12, c3["n_embd"], c3["block_size"], c3["vocab_size"], c3["bias"])
    assert math.floor(og.param_count(cfg) / 1e6) == c3["printed_millions"]


def test_generate_top_k_one_is_greedy_and_cache_bounds():
    cfg, w, _ = _model(syn.TINY)
    prompt = syn.make_tokens(2, 16, 65, seed=12)
    out = og.generate(cfg, w, prompt, max_new_tokens=8, temperature=0.8, top_k=1, seed=3)
    fed, logits = og.teacher_forced(cfg, w, np.ascontiguousarray(prompt[:1]), n_steps=7)
    assert np.array_equal(out[:1, 16:16 + 7], fed)
    assert out[0, -1] == np.argmax(logits[-1, 0])
    g = og.generate(cfg, w, prompt, max_new_tokens=8, temperature=0.0, top_k=None, seed=3)
    assert np.array_equal(g, out)
    # prompt + new tokens may fill block_size exactly (the last token is never fed back)
    og.generate(cfg, w, prompt[:, :4], max_new_tokens=cfg.block_size - 3, temperature=1.0, top_k=5, seed=1)
    with pytest.raises(ValueError):
        og.generate(cfg, w, prompt[:, :4], max_new_tokens=cfg.block_size - 2, temperature=1.0, top_k=5, seed=1)


def test_generate_cropped_is_the_cached_generate_until_the_crop():
    # no crop needed: the pages' generate() without a cache and the cached one draw the same
    cfg, w, _ = _model(TOY_BIAS, bias_std=0.05)
    prompt = syn.make_tokens(2, 5, TOY_BIAS.vocab_size, seed=8)
    n = cfg.block_size - 5 + 1  # the last draw sees exactly block_size tokens
    a = og.generate(cfg, w, prompt, n, temperature=0.9, top_k=10, seed=4)
    b = og.generate_cropped(cfg, w, prompt, n, temperature=0.9, top_k=10, seed=4)
    assert np.array_equal(a, b)


def test_generate_cropped_conditions_each_draw_on_the_last_block_size_tokens():
    # brute force: past the crop, draw j equals the sampler applied to the plain forward of the
    # last block_size tokens with positions restarting at 0; and a prompt longer than
    # block_size behaves as its last block_size tokens
    from oracle import sampler as osm

    cfg, w, _ = _model(TOY, seed=3)
    bs = cfg.block_size
    prompt = syn.make_tokens(2, bs - 3, TOY.vocab_size, seed=6)
    out = og.generate_cropped(cfg, w, prompt, 9, temperature=1.0, top_k=None, seed=2)
    for j in range(9):
        ctx = out[:, :prompt.shape[1] + j][:, -bs:]
        logits = og.forward_full(cfg, w, ctx)[:, -1, :]
        assert np.array_equal(out[:, prompt.shape[1] + j], osm.sample(logits.astype(np.float32), 1.0, None, 2, j))
    long_prompt = syn.make_tokens(2, bs + 7, TOY.vocab_size, seed=9)
    a = og.generate_cropped(cfg, w, long_prompt, 3, temperature=0.0, top_k=None, seed=0)
    b = og.generate_cropped(cfg, w, long_prompt[:, 7:], 3, temperature=0.0, top_k=None, seed=0)
    assert np.array_equal(a[:, -3:], b[:, -3:])
