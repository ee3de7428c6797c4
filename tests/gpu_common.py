"""Shared helpers of the GPU parity tests: seeded inputs on both sides, model handles."""
from __future__ import annotations

import numpy as np
import torch

from kv_cached_generation_gpt_b300 import gpt as G
from kv_cached_generation_gpt_b300 import synthetic as syn
from oracle import gpt as og


def torch_dtype(shape: syn.ModelShape) -> torch.dtype:
    return torch.float32 if shape.dtype == "f32" else torch.bfloat16


def device_state_dict(shape: syn.ModelShape, sd: dict[str, np.ndarray]) -> dict[str, torch.Tensor]:
    dt = torch_dtype(shape)
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(dt).cuda() for k, v in sd.items()}


def oracle_model(shape: syn.ModelShape, sd: dict[str, np.ndarray]):
    cfg = og.Config(shape.n_layer, shape.n_head, shape.n_embd, shape.block_size, shape.vocab_size, shape.bias)
    return cfg, og.weights_from_state_dict(cfg, syn.storage_values(shape, sd))


def make_gpu_model(shape: syn.ModelShape, sd: dict[str, np.ndarray], max_batch: int, page_size: int = 0,
                   n_pages: int = 0) -> G.GPT:
    return G.GPT(shape.n_layer, shape.n_head, shape.n_embd, shape.block_size, shape.vocab_size, shape.bias,
                 torch_dtype(shape), max_batch, device_state_dict(shape, sd), page_size, n_pages)


def gpu_teacher_forced(model: G.GPT, prompt: np.ndarray, forced: np.ndarray, rows=None) -> np.ndarray:
    """Prefill the prompt, then feed forced[:, i] for each decode step.  Returns fp32 logits
    (N+1, len(rows), V) for the selected rows (all rows by default)."""
    tok = torch.from_numpy(np.ascontiguousarray(prompt, dtype=np.int32)).cuda()
    sel = slice(None) if rows is None else torch.tensor(rows, device="cuda")
    out = [model.prefill(tok)[sel].clone()]
    for i in range(forced.shape[1]):
        t = torch.from_numpy(np.ascontiguousarray(forced[:, i], dtype=np.int32)).cuda()
        out.append(model.decode_step(t)[sel].clone())
    status = model.sync_status()
    assert status == G.GPT_OK, G.lib().gpt_strerror(status)
    return torch.stack(out).cpu().numpy()


def argmax_agreement(gpu: np.ndarray, ref: np.ndarray) -> float:
    return float(np.mean(np.argmax(gpu, axis=-1) == np.argmax(ref, axis=-1)))
