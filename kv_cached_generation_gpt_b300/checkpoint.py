"""GPT-2 checkpoints in the HuggingFace layout <-> nanoGPT state_dict names (host side, once).

Load-time format conversion only: nothing here runs per token, and the model's arithmetic
stays in the library's kernels.  No download: the caller brings the tensors.

Why it is needed ("原生 nanoGPT 模型服务首选", §1 正确性; "nanoGPT 架构分析", §4.1 Pretrained
权重加载; "第 4 章 模型构建", §4.5 GPT2LMHeadModel 内部长什么样): HuggingFace's GPT2LMHeadModel
keeps every projection as a Conv1D whose weight is stored (in_features, out_features), while
nanoGPT (and this library's gpt_create) takes nn.Linear weights (out_features, in_features) --
the fused c_attn included, q | k | v blocks along the output features.  A transpose missed or
applied twice does not crash: it silently corrupts the output.  HF's layout also always has
biases (a bias=False model gets zero biases there), registers the causal mask as a buffer
(`attn.bias`, `attn.masked_bias`) that is not a parameter, and may store the tied lm_head as
its own `lm_head.weight`, equal to wte.
"""
from __future__ import annotations

import re

import numpy as np

# Projections stored as Conv1D (in, out) in the HF layout; nn.Linear (out, in) in nanoGPT's.
CONV1D_SUFFIXES = ("attn.c_attn.weight", "attn.c_proj.weight", "mlp.c_fc.weight", "mlp.c_proj.weight")
# Non-parameter buffers of the HF attention module (the causal mask and its fill value).
HF_BUFFERS = ("attn.bias", "attn.masked_bias")
LAYER_PARAMS = ("ln_1.weight", "ln_1.bias", "attn.c_attn.weight", "attn.c_attn.bias", "attn.c_proj.weight",
                "attn.c_proj.bias", "ln_2.weight", "ln_2.bias", "mlp.c_fc.weight", "mlp.c_fc.bias",
                "mlp.c_proj.weight", "mlp.c_proj.bias")

_LAYER_KEY = re.compile(r"^h\.(\d+)\.(.+)$")


def _numpy(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t
    # torch tensors (any device / dtype): widen to fp32 on the host; the caller picks the
    # model's storage type afterwards
    return t.detach().float().cpu().numpy()


def _strip(key: str) -> str:
    return key[len("transformer."):] if key.startswith("transformer.") else key


def from_hf_state_dict(sd: dict, n_head: int | None = None, drop_zero_bias: bool = False):
    """Convert a GPT-2 state_dict in the HuggingFace layout to nanoGPT names and layout.

    sd: HF keys with or without the "transformer." prefix (`wte.weight`, `wpe.weight`,
    `h.{l}.ln_1.weight`, `h.{l}.attn.c_attn.weight` (C, 3C), ..., `ln_f.weight`, optionally
    `lm_head.weight`), values numpy arrays or torch tensors.
    n_head: heads per layer (the tensors do not fix it); default n_embd // 64, GPT-2's head size.
    drop_zero_bias: when every bias and LayerNorm beta is exactly zero, return a bias=False model
    (the reverse of the zero-filled slots an HF export of a bias=False model carries).

    Returns (config, state_dict): config a dict of gpt_create's fields (n_layer, n_head, n_embd,
    block_size, vocab_size, bias); state_dict with nanoGPT keys (`transformer.h.{l}.attn.c_attn.weight`
    (3C, C), ...) as contiguous fp32 numpy arrays.  Raises ValueError on a missing key, an
    unexpected one, a shape that does not fit GPT-2, or an lm_head that is not tied to wte."""
    src = {}
    for k, v in sd.items():
        k = _strip(k)
        if any(k.endswith("." + b) for b in HF_BUFFERS) and _LAYER_KEY.match(k):
            continue
        src[k] = _numpy(v)
    for k in ("wte.weight", "wpe.weight", "ln_f.weight"):
        if k not in src:
            raise ValueError(f"missing {k}")
    wte = src.pop("wte.weight")
    V, C = wte.shape
    wpe = src.pop("wpe.weight")
    if wpe.ndim != 2 or wpe.shape[1] != C:
        raise ValueError(f"wpe shape {wpe.shape} does not match n_embd {C}")
    head = src.pop("lm_head.weight", None)
    if head is not None and (head.shape != wte.shape or not np.array_equal(head, wte)):
        raise ValueError("lm_head.weight is not tied to wte.weight")
    layers = sorted({int(m.group(1)) for m in map(_LAYER_KEY.match, src) if m})
    L = len(layers)
    if layers != list(range(L)):
        raise ValueError(f"layer indices {layers} are not 0..{L - 1}")
    out = {"transformer.wte.weight": np.ascontiguousarray(wte), "transformer.wpe.weight": np.ascontiguousarray(wpe),
           "transformer.ln_f.weight": src.pop("ln_f.weight")}
    if "ln_f.bias" in src:
        out["transformer.ln_f.bias"] = src.pop("ln_f.bias")
    expect = {"ln_1.weight": (C,), "ln_1.bias": (C,), "attn.c_attn.weight": (C, 3 * C), "attn.c_attn.bias": (3 * C,),
              "attn.c_proj.weight": (C, C), "attn.c_proj.bias": (C,), "ln_2.weight": (C,), "ln_2.bias": (C,),
              "mlp.c_fc.weight": (C, 4 * C), "mlp.c_fc.bias": (4 * C,), "mlp.c_proj.weight": (4 * C, C),
              "mlp.c_proj.bias": (C,)}
    for l in range(L):
        for name in LAYER_PARAMS:
            key = f"h.{l}.{name}"
            if key not in src:
                if name.endswith(".bias"):
                    continue
                raise ValueError(f"missing {key}")
            t = src.pop(key)
            if t.shape != expect[name]:
                raise ValueError(f"{key}: shape {t.shape}, expected {expect[name]} (HF Conv1D layout)")
            if name in CONV1D_SUFFIXES:
                t = t.T  # Conv1D (in, out) -> nn.Linear (out, in)
            out[f"transformer.h.{l}.{name}"] = np.ascontiguousarray(t)
    if src:
        raise ValueError(f"unexpected keys: {sorted(src)[:5]}")
    bias_keys = [k for k in out if k.endswith(".bias")]
    n_bias_expected = 6 * L + 1  # per layer ln_1, c_attn, c_proj, ln_2, c_fc, mlp c_proj; ln_f
    if not bias_keys:
        has_bias = False
    elif len(bias_keys) == n_bias_expected:
        has_bias = True
        if drop_zero_bias and all(not np.any(out[k]) for k in bias_keys):
            for k in bias_keys:
                del out[k]
            has_bias = False
    else:
        raise ValueError(f"{len(bias_keys)} bias tensors: expected all {n_bias_expected} or none")
    if n_head is None:
        n_head = C // 64
    if n_head < 1 or C % n_head:
        raise ValueError(f"n_embd {C} is not a multiple of n_head {n_head}")
    config = dict(n_layer=L, n_head=n_head, n_embd=C, block_size=wpe.shape[0], vocab_size=V, bias=has_bias)
    return config, out


def to_hf_state_dict(sd: dict, n_layer: int, prefix: str = "transformer.", tied_head: bool = True) -> dict:
    """The reverse: nanoGPT-named (out, in) weights to the HF layout (Conv1D (in, out)).  A
    bias=False model gets the zero biases and LayerNorm betas the HF module always has (the
    exact zeros of "原生 nanoGPT 模型服务首选", §1: bias=None and bias=zeros agree), and the
    lm_head is written as a copy of wte when tied_head is set."""
    get = lambda k: _numpy(sd[k])  # noqa: E731
    wte = get("transformer.wte.weight")
    C = wte.shape[1]
    out = {prefix + "wte.weight": wte.copy(), prefix + "wpe.weight": get("transformer.wpe.weight").copy(),
           prefix + "ln_f.weight": get("transformer.ln_f.weight").copy(),
           prefix + "ln_f.bias": (get("transformer.ln_f.bias").copy() if "transformer.ln_f.bias" in sd
                                  else np.zeros(C, np.float32))}
    zeros = {"ln_1.bias": C, "attn.c_attn.bias": 3 * C, "attn.c_proj.bias": C, "ln_2.bias": C, "mlp.c_fc.bias": 4 * C,
             "mlp.c_proj.bias": C}
    for l in range(n_layer):
        for name in LAYER_PARAMS:
            key = f"transformer.h.{l}.{name}"
            if key in sd:
                t = get(key)
                t = np.ascontiguousarray(t.T) if name in CONV1D_SUFFIXES else t.copy()
            else:
                t = np.zeros(zeros[name], np.float32)
            out[f"{prefix}h.{l}.{name}"] = t
        # the causal-mask buffer an HF module registers (ignored by the conversion back)
        out[f"{prefix}h.{l}.attn.bias"] = np.tril(np.ones((1, 1, 4, 4), np.float32))
    if tied_head:
        out["lm_head.weight"] = wte.copy()
    return out
