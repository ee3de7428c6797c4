"""fp64 CPU oracle of nanoGPT's GPT-2 decoder, with and without a KV cache.

TEST INFRASTRUCTURE: imported only by tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py.  Nothing here is shared with the CUDA path.

Every tensor is float64; the matmul is numpy's (a library primitive).  Nothing
is blocked, fused or reordered beyond what the definitions below state.  For
bf16 models the caller hands in the bf16-rounded weight values widened to
float64, so weight quantisation is not counted as error; activations are never
rounded here.

Pages restated (title, site, section):
  [serving] "原生 nanoGPT 模型服务首选" (lzwjava.github.io):
            §1 "正确性" -- LayerNorm(ndim, bias) with eps 1e-5 and bias=None allowed;
            §2 "采样一致性" -- generate();
            §"一个值得做的改进" -- the KV-cache sketch (cat past K/V along time,
            is_causal only without a past).
  [sdk]     "极速上手nanoGPT：从模型加载到文本生成的全流程SDK开发指南" (deepseek.csdn.net):
            §"GPTConfig类"; §"注意力机制" (scaled_dot_product_attention(is_causal=True)
            and the manual masked-softmax path, shapes (B, nh, T, hs)).
  [arch]    "nanoGPT 架构分析" (wangbinyq.github.io), §4.1 "GPT 模型 (model.py)":
            pre-LN residual blocks, 4x MLP, weight tying, last-position lm_head.
  [ch4]     "第 4 章 模型构建" (aiknowledge.cn), §4.5: wte + wpe (learned absolute
            positions), lower-triangular causal mask, lm_head Linear(n_embd, vocab,
            bias=False) sharing wte.
  [guide]   "LLM研究框架选择指南：从nanoGPT到nanochat的实战分析" (intelliparadigm.com),
            §2.1 Block: x = x + attn(ln_1(x)); x = x + mlp(ln_2(x)), MLP with nn.GELU().

Readings where the pages leave a step open:
  * GELU is the exact erf form (nn.GELU()'s default; no approximation is named).
  * LayerNorm variance is the biased one (F.layer_norm's definition).
  * c_attn's output splits into q | k | v blocks of n_embd columns; head h owns
    columns [h*hs, (h+1)*hs) of each block; heads are re-concatenated in order
    before c_proj.
  * A token appended to a cache of length c sits at position c; a query at
    position p sees keys 0..p (the offset form of the causal mask, which is the
    sketch's "no mask" for a single new token and the plain causal mask for an
    empty cache).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
from scipy.special import erf

LN_EPS = 1e-5  # [serving] §1: F.layer_norm(..., 1e-5)


@dataclasses.dataclass(frozen=True)
class Config:
    """[sdk] §"GPTConfig类": block_size, vocab_size, n_layer, n_head, n_embd, bias."""

    n_layer: int
    n_head: int
    n_embd: int
    block_size: int
    vocab_size: int
    bias: bool

    @property
    def head_size(self) -> int:
        return self.n_embd // self.n_head


@dataclasses.dataclass
class Layer:
    ln_1_w: np.ndarray
    ln_1_b: np.ndarray | None
    c_attn_w: np.ndarray  # (3C, C), nn.Linear (out, in) layout
    c_attn_b: np.ndarray | None
    attn_proj_w: np.ndarray  # (C, C)
    attn_proj_b: np.ndarray | None
    ln_2_w: np.ndarray
    ln_2_b: np.ndarray | None
    c_fc_w: np.ndarray  # (4C, C)
    c_fc_b: np.ndarray | None
    mlp_proj_w: np.ndarray  # (C, 4C)
    mlp_proj_b: np.ndarray | None


@dataclasses.dataclass
class Weights:
    wte: np.ndarray  # (V, C); also the lm_head weight ([arch] §4.1 weight tying)
    wpe: np.ndarray  # (block_size, C)
    layers: list[Layer]
    ln_f_w: np.ndarray
    ln_f_b: np.ndarray | None


def weights_from_state_dict(cfg: Config, sd: dict) -> Weights:
    """Build fp64 weights from nanoGPT state_dict names (missing biases -> None)."""

    def get(name):
        a = sd.get(name)
        return None if a is None else np.asarray(a, dtype=np.float64)

    layers = []
    for l in range(cfg.n_layer):
        p = f"transformer.h.{l}."
        layers.append(Layer(
            get(p + "ln_1.weight"), get(p + "ln_1.bias"),
            get(p + "attn.c_attn.weight"), get(p + "attn.c_attn.bias"),
            get(p + "attn.c_proj.weight"), get(p + "attn.c_proj.bias"),
            get(p + "ln_2.weight"), get(p + "ln_2.bias"),
            get(p + "mlp.c_fc.weight"), get(p + "mlp.c_fc.bias"),
            get(p + "mlp.c_proj.weight"), get(p + "mlp.c_proj.bias"),
        ))
    return Weights(get("transformer.wte.weight"), get("transformer.wpe.weight"), layers,
                   get("transformer.ln_f.weight"), get("transformer.ln_f.bias"))


# ---------------------------------------------------------------- building blocks


def layer_norm(x: np.ndarray, weight: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    """[serving] §1: F.layer_norm over the last axis, eps 1e-5, biased variance.

    A missing bias (bias=False) adds nothing."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    y = (x - mu) / np.sqrt(var + LN_EPS) * weight
    if bias is not None:
        y = y + bias
    return y


def gelu(z: np.ndarray) -> np.ndarray:
    """[guide] §2.1, [arch] §4.1: nn.GELU(), exact form 0.5 z (1 + erf(z / sqrt 2))."""
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def linear(x: np.ndarray, weight: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    """nn.Linear: y = x W^T (+ b), W stored (out_features, in_features)."""
    y = x @ weight.T
    if bias is not None:
        y = y + bias
    return y


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos0: int) -> np.ndarray:
    """[sdk] §"注意力机制", manual path, with [ch4] §4.5's lower-triangular mask.

    q: (B, nh, Tq, hs) at absolute positions q_pos0 .. q_pos0+Tq-1;
    k, v: (B, nh, Tk, hs) at positions 0 .. Tk-1.  Query i sees key j iff
    j <= q_pos0 + i.  Scores are (q k^T) / sqrt(hs); masked entries are -inf
    before the softmax over keys; the result is softmax @ v."""
    hs = q.shape[-1]
    att = (q @ np.swapaxes(k, -1, -2)) * (1.0 / math.sqrt(hs))
    tq, tk = q.shape[-2], k.shape[-2]
    qpos = q_pos0 + np.arange(tq)[:, None]
    kpos = np.arange(tk)[None, :]
    att = np.where(kpos <= qpos, att, -np.inf)
    att = att - att.max(axis=-1, keepdims=True)
    p = np.exp(att)
    p = p / p.sum(axis=-1, keepdims=True)
    return p @ v


def causal_self_attention(cfg: Config, lw: Layer, x: np.ndarray, past=None):
    """[serving] §"一个值得做的改进" + [sdk] §"注意力机制".

    x: (B, T, C).  c_attn gives q|k|v (split at n_embd), each viewed (B, nh, T, hs).
    With a past (pk, pv) of length c, k and v are concatenated after it along time.
    Returns (y after c_proj, present=(k, v))."""
    B, T, C = x.shape
    nh, hs = cfg.n_head, cfg.head_size
    qkv = linear(x, lw.c_attn_w, lw.c_attn_b)
    q, k, v = qkv[..., :C], qkv[..., C:2 * C], qkv[..., 2 * C:]

    def heads(t):
        return t.reshape(B, T, nh, hs).transpose(0, 2, 1, 3)

    q, k, v = heads(q), heads(k), heads(v)
    c = 0
    if past is not None:
        pk, pv = past
        c = pk.shape[2]
        k = np.concatenate([pk, k], axis=2)
        v = np.concatenate([pv, v], axis=2)
    y = attention(q, k, v, q_pos0=c)
    y = y.transpose(0, 2, 1, 3).reshape(B, T, C)
    return linear(y, lw.attn_proj_w, lw.attn_proj_b), (k, v)


def mlp(lw: Layer, x: np.ndarray) -> np.ndarray:
    """[arch] §4.1 / [guide] §2.1: Linear(C, 4C) -> GELU -> Linear(4C, C)."""
    return linear(gelu(linear(x, lw.c_fc_w, lw.c_fc_b)), lw.mlp_proj_w, lw.mlp_proj_b)


def block(cfg: Config, lw: Layer, x: np.ndarray, past=None):
    """[guide] §2.1 / [arch] §4.1 pre-LN block: x += attn(ln_1(x)); x += mlp(ln_2(x))."""
    a, present = causal_self_attention(cfg, lw, layer_norm(x, lw.ln_1_w, lw.ln_1_b), past)
    x = x + a
    x = x + mlp(lw, layer_norm(x, lw.ln_2_w, lw.ln_2_b))
    return x, present


# ---------------------------------------------------------------- model


def forward(cfg: Config, w: Weights, idx: np.ndarray, past=None, all_positions: bool = False):
    """One forward pass over new tokens ``idx`` (B, T), after an optional cache ``past``.

    Embedding ([ch4] §4.5): x = wte[id] + wpe[pos], pos = c .. c+T-1 where c is the
    cache length.  Then the blocks, ln_f, and the tied lm_head (x wte^T, no bias).
    Inference evaluates the lm_head on the last position only ([arch] §4.1
    "生成优化"); ``all_positions=True`` returns logits for every position.

    Returns (logits, presents): logits (B, V) or (B, T, V); presents a list of
    (k, v) per layer, each (B, nh, c+T, hs)."""
    idx = np.asarray(idx)
    B, T = idx.shape
    c = 0 if past is None else past[0][0].shape[2]
    if T < 1 or c + T > cfg.block_size:
        raise ValueError("context overflow: cache %d + new %d > block_size %d" % (c, T, cfg.block_size))
    if idx.min() < 0 or idx.max() >= cfg.vocab_size:
        raise ValueError("token id out of range")
    x = w.wte[idx] + w.wpe[c:c + T][None, :, :]
    presents = []
    for l, lw in enumerate(w.layers):
        x, present = block(cfg, lw, x, None if past is None else past[l])
        presents.append(present)
    x = layer_norm(x, w.ln_f_w, w.ln_f_b)
    if all_positions:
        return x @ w.wte.T, presents
    return x[:, -1, :] @ w.wte.T, presents


def forward_full(cfg: Config, w: Weights, idx: np.ndarray) -> np.ndarray:
    """No-cache forward: logits at every position, (B, T, V)."""
    return forward(cfg, w, idx, None, all_positions=True)[0]


def prefill(cfg: Config, w: Weights, idx: np.ndarray):
    """Prompt pass from an empty cache: (last-position logits (B, V), cache)."""
    return forward(cfg, w, idx, None)


def decode(cfg: Config, w: Weights, cache, tokens: np.ndarray):
    """One KV-cached step: tokens (B,) at position len(cache) -> (logits (B, V), cache)."""
    return forward(cfg, w, np.asarray(tokens).reshape(-1, 1), cache)


def greedy(logits: np.ndarray) -> np.ndarray:
    """argmax over the vocabulary, lowest index on ties (torch.argmax's convention)."""
    return np.argmax(logits, axis=-1).astype(np.int32)


def teacher_forced(cfg: Config, w: Weights, prompt: np.ndarray, forced: np.ndarray | None = None,
                   n_steps: int | None = None):
    """Prefill ``prompt`` (B, P), then decode.

    If ``forced`` (B, N) is given, decode step i feeds forced[:, i]; otherwise it feeds
    the oracle's own greedy token of the previous logits (N = n_steps).
    Returns (fed tokens (B, N), logits (N+1, B, V)): logits[0] from the prefill,
    logits[i+1] from decode step i."""
    logits, cache = prefill(cfg, w, prompt)
    out = [logits]
    n = forced.shape[1] if forced is not None else int(n_steps)
    fed = np.zeros((prompt.shape[0], n), np.int32)
    for i in range(n):
        tok = forced[:, i] if forced is not None else greedy(out[-1])
        fed[:, i] = tok
        logits, cache = decode(cfg, w, cache, tok)
        out.append(logits)
    return fed, np.stack(out)


def param_count(cfg: Config) -> int:
    """Exact number of stored parameters with lm_head tied to wte.

    V*C (wte, counted once) + block*C (wpe) + per layer 12 C^2 + 2C (weights + the two
    LayerNorm gammas) + C (ln_f gamma); with bias: + per layer 11C + C."""
    C, L = cfg.n_embd, cfg.n_layer
    n = cfg.vocab_size * C + cfg.block_size * C + L * (12 * C * C + 2 * C) + C
    if cfg.bias:
        n += L * 11 * C + C
    return n


def generate(cfg: Config, w: Weights, idx: np.ndarray, max_new_tokens: int, temperature: float,
             top_k: int | None, seed: int):
    """[serving] §2 generate() with a KV cache instead of recomputing the prefix.

    Draw j (j = 0 .. max_new_tokens-1) samples from the logits after the prompt (j=0)
    or after feeding new token j-1, with the sampler's step index j.  The cache never
    crops: idx.shape[1] + max_new_tokens - 1 must fit in block_size.  Logits are
    handed to the sampler as fp32, the precision of the library's logits buffer.
    Returns (B, T + max_new_tokens) int32."""
    from oracle import sampler

    idx = np.asarray(idx, dtype=np.int32)
    B, T = idx.shape
    if T + max_new_tokens - 1 > cfg.block_size:
        raise ValueError("context overflow")
    out = [idx]
    logits, cache = prefill(cfg, w, idx)
    for j in range(max_new_tokens):
        tok = sampler.sample(logits.astype(np.float32), temperature, top_k, seed, j)
        out.append(tok[:, None])
        if j + 1 < max_new_tokens:
            logits, cache = decode(cfg, w, cache, tok)
    return np.concatenate(out, axis=1)


def generate_cropped(cfg: Config, w: Weights, idx: np.ndarray, max_new_tokens: int, temperature: float,
                     top_k: int | None, seed: int):
    """[serving] §2 generate() exactly as printed, no cache: before every draw the context is
    cropped to its last block_size tokens (positions restart at 0 in the window), run through
    the whole model, and the last position's logits are sampled (draw index j = the step).
    Agrees with generate() wherever no crop is needed.  Returns (B, T + max_new_tokens) int32."""
    from oracle import sampler

    idx = np.asarray(idx, dtype=np.int32)
    for j in range(max_new_tokens):
        cond = idx if idx.shape[1] <= cfg.block_size else idx[:, -cfg.block_size:]
        logits = forward(cfg, w, cond)[0]
        tok = sampler.sample(logits.astype(np.float32), temperature, top_k, seed, j)
        idx = np.concatenate([idx, tok[:, None].astype(np.int32)], axis=1)
    return idx
