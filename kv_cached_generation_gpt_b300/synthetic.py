"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws random numbers and names shapes.  It holds none of the
model's arithmetic: no layer norm, no matmul, no attention, no sampling.

Weights follow GPT-2's random initialisation as nanoGPT describes it
("nanoGPT 架构分析", wangbinyq.github.io, §4.1 "特殊残差初始化"): every Linear and
embedding weight N(0, 0.02), the two residual projections (attn.c_proj and
mlp.c_proj) N(0, 0.02/sqrt(2*n_layer)), LayerNorm gamma = 1 and beta = 0
("原生 nanoGPT 模型服务首选", §1 LayerNorm(ndim, bias)).  When ``bias_std`` is
given, every Linear bias and LayerNorm beta is N(0, bias_std) instead of zero.
Weight names are nanoGPT's state_dict names; the lm_head has no entry because
it is tied to ``transformer.wte.weight``.

Token ids are uniform in [0, token_hi).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

WEIGHT_SEED = 1337
TOKEN_SEED = 1338


@dataclasses.dataclass(frozen=True)
class ModelShape:
    n_layer: int
    n_head: int
    n_embd: int
    block_size: int
    vocab_size: int
    bias: bool
    dtype: str  # "f32" or "bf16": the storage type the GPU path is given

    @property
    def head_size(self) -> int:
        return self.n_embd // self.n_head


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    model: ModelShape
    batch: int
    prompt: int
    decode_steps: int
    temperature: float  # 0 means greedy argmax
    top_k: int  # <= 0 means no top-k masking
    token_hi: int  # prompt ids are drawn from [0, token_hi)
    bias_std: float | None = None


TINY = ModelShape(4, 4, 128, 64, 65, False, "f32")
CHAR = ModelShape(6, 6, 384, 256, 65, False, "bf16")
GPT2_124M = ModelShape(12, 12, 768, 1024, 50304, False, "bf16")
GPT2_350M_BIAS = ModelShape(24, 16, 1024, 1024, 50257, True, "bf16")

WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_b1_p16_d32", TINY, 1, 16, 32, 0.0, 0, 65),
        Workload("char_b1_p1_d255", CHAR, 1, 1, 255, 0.8, 200, 65),
        Workload("gpt2_124m_b1_p128_d896", GPT2_124M, 1, 128, 896, 0.0, 200, 50257),
        Workload("gpt2_124m_b64_p512_d512", GPT2_124M, 64, 512, 512, 1.0, 50, 50257),
        Workload("gpt2_350m_b8_p768_d256", GPT2_350M_BIAS, 8, 768, 256, 0.0, 0, 50257, 0.02),
    ]
}

LAYER_KEYS = (
    "ln_1.weight", "ln_1.bias",
    "attn.c_attn.weight", "attn.c_attn.bias",
    "attn.c_proj.weight", "attn.c_proj.bias",
    "ln_2.weight", "ln_2.bias",
    "mlp.c_fc.weight", "mlp.c_fc.bias",
    "mlp.c_proj.weight", "mlp.c_proj.bias",
)


def layer_key(layer: int, name: str) -> str:
    return f"transformer.h.{layer}.{name}"


def make_weights(shape: ModelShape, seed: int = WEIGHT_SEED, bias_std: float | None = None,
                 random_gamma: bool = False) -> dict[str, np.ndarray]:
    """Return fp32 weights keyed by nanoGPT state_dict name (biases absent when bias=False).

    ``random_gamma`` draws LayerNorm gammas as 1 + N(0, 0.1) (used by unit tests only, so
    that a dropped gamma is visible)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    C, L, V = shape.n_embd, shape.n_layer, shape.vocab_size
    proj_std = 0.02 / math.sqrt(2 * max(L, 1))

    def normal(shp, std):
        return (rng.standard_normal(shp, dtype=np.float32) * np.float32(std)).astype(np.float32)

    def gamma():
        if random_gamma:
            return (1.0 + rng.standard_normal(C, dtype=np.float32) * np.float32(0.1)).astype(np.float32)
        return np.ones(C, np.float32)

    def beta(n):
        if bias_std is None:
            return np.zeros(n, np.float32)
        return normal(n, bias_std)

    w: dict[str, np.ndarray] = {}
    w["transformer.wte.weight"] = normal((V, C), 0.02)
    w["transformer.wpe.weight"] = normal((shape.block_size, C), 0.02)
    for l in range(L):
        w[layer_key(l, "ln_1.weight")] = gamma()
        w[layer_key(l, "attn.c_attn.weight")] = normal((3 * C, C), 0.02)
        w[layer_key(l, "attn.c_proj.weight")] = normal((C, C), proj_std)
        w[layer_key(l, "ln_2.weight")] = gamma()
        w[layer_key(l, "mlp.c_fc.weight")] = normal((4 * C, C), 0.02)
        w[layer_key(l, "mlp.c_proj.weight")] = normal((C, 4 * C), proj_std)
        if shape.bias:
            w[layer_key(l, "ln_1.bias")] = beta(C)
            w[layer_key(l, "attn.c_attn.bias")] = beta(3 * C)
            w[layer_key(l, "attn.c_proj.bias")] = beta(C)
            w[layer_key(l, "ln_2.bias")] = beta(C)
            w[layer_key(l, "mlp.c_fc.bias")] = beta(4 * C)
            w[layer_key(l, "mlp.c_proj.bias")] = beta(C)
    w["transformer.ln_f.weight"] = gamma()
    if shape.bias:
        w["transformer.ln_f.bias"] = beta(C)
    return w


def make_tokens(batch: int, length: int, token_hi: int, seed: int = TOKEN_SEED) -> np.ndarray:
    """Uniform token ids in [0, token_hi), int32, shape (batch, length)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(0, token_hi, size=(batch, length), dtype=np.int64).astype(np.int32)


def make_logits(batch: int, vocab: int, seed: int, std: float = 1.0) -> np.ndarray:
    """Random fp32 logits (for sampler tests)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return (rng.standard_normal((batch, vocab), dtype=np.float32) * np.float32(std)).astype(np.float32)


def to_bf16_values(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even) and return them widened to fp32.

    Storage-format conversion done by torch: both sides then see the same bf16 values."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


def storage_values(shape: ModelShape, weights: dict[str, np.ndarray]) -> dict[str, np.ndarray]:
    """The values the GPU path stores: bf16-rounded for bf16 models, as-is for f32 models."""
    if shape.dtype == "f32":
        return dict(weights)
    return {k: to_bf16_values(v) for k, v in weights.items()}
