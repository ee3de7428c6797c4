"""ctypes binding of libgpt_b300.so with the names of include/gpt.h.

Argument marshalling only: torch CUDA tensors in, device pointers and the current
stream handed to the library, status codes turned into exceptions.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.  If the library
is not built, or a call fails, this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgpt_b300.so")

GPT_OK = 0
GPT_EINVAL = -1
GPT_ECONTEXT = -2
GPT_ECUDA = -3
GPT_ENOMEM = -4
GPT_ETOKEN = -5
GPT_ETIMEOUT = -6
GPT_EPOSITION = -7
GPT_EUNSUPPORTED = -8
GPT_ESTATE = -9
GPT_ETOOBIG = -10

GPT_DTYPE_F32 = 0
GPT_DTYPE_BF16 = 1

EXPORTED = (
    "gpt_create", "gpt_create_paged", "gpt_destroy", "gpt_prefill", "gpt_prefill_ragged", "gpt_extend", "gpt_decode_step", "gpt_generate", "gpt_last_timing",
    "gpt_cache_length", "gpt_kernel_launches", "gpt_sync_status", "gpt_strerror", "gpt_last_error_detail", "gpt_linear_bf16",
    "gpt_layernorm", "gpt_attention_prefill", "gpt_attention_decode", "gpt_sample", "gpt_op_status",
    "gpt_attention_decode_noalloc", "gpt_linear_decode_bf16", "gpt_layernorm_linear_decode_bf16", "gpt_profile_gemms", "gpt_gemm_timing",
    "gpt_debug_bounded_wait", "gpt_debug_fail_allocation",
)

c_int32, c_void_p, c_float, c_uint64, c_int64 = ctypes.c_int32, ctypes.c_void_p, ctypes.c_float, ctypes.c_uint64, ctypes.c_int64


class gpt_config_t(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in
                ("n_layer", "n_head", "n_embd", "block_size", "vocab_size", "bias", "dtype", "max_batch")]


LAYER_FIELDS = ("ln_1_w", "ln_1_b", "c_attn_w", "c_attn_b", "attn_proj_w", "attn_proj_b",
                "ln_2_w", "ln_2_b", "c_fc_w", "c_fc_b", "mlp_proj_w", "mlp_proj_b")
# state_dict suffix of each field (nanoGPT names)
LAYER_KEYS = ("ln_1.weight", "ln_1.bias", "attn.c_attn.weight", "attn.c_attn.bias", "attn.c_proj.weight",
              "attn.c_proj.bias", "ln_2.weight", "ln_2.bias", "mlp.c_fc.weight", "mlp.c_fc.bias",
              "mlp.c_proj.weight", "mlp.c_proj.bias")


class gpt_layer_weights_t(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in LAYER_FIELDS]


class gpt_weights_t(ctypes.Structure):
    _fields_ = [("wte", c_void_p), ("wpe", c_void_p), ("ln_f_w", c_void_p), ("ln_f_b", c_void_p),
                ("layers", ctypes.POINTER(gpt_layer_weights_t))]


class GptError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        detail = lib().gpt_last_error_detail().decode()
        msg = f"{where}: {lib().gpt_strerror(code).decode()} ({code})"
        super().__init__(msg + (f" [{detail}]" if detail and code in (GPT_ECUDA, GPT_ENOMEM, GPT_EUNSUPPORTED, GPT_ETOOBIG) else ""))


_lib = None


def lib() -> ctypes.CDLL:
    """Load libgpt_b300.so (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; build it with `python -m kv_cached_generation_gpt_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        sig = {
            "gpt_create": (ctypes.c_int, [P(gpt_config_t), P(gpt_weights_t), c_void_p, P(c_void_p)]),
            "gpt_create_paged": (ctypes.c_int, [P(gpt_config_t), P(gpt_weights_t), c_void_p, c_int32, c_int32,
                                                P(c_void_p)]),
            "gpt_destroy": (None, [c_void_p]),
            "gpt_prefill": (ctypes.c_int, [c_void_p, c_void_p, c_int32, c_int32, c_void_p]),
            "gpt_decode_step": (ctypes.c_int, [c_void_p, c_void_p, c_void_p]),
            "gpt_extend": (ctypes.c_int, [c_void_p, c_void_p, c_int32, c_void_p]),
            "gpt_prefill_ragged": (ctypes.c_int, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_void_p]),
            "gpt_generate": (ctypes.c_int, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_float, c_int32,
                                            c_uint64, c_void_p]),
            "gpt_last_timing": (ctypes.c_int, [c_void_p, P(c_float), P(c_float)]),
            "gpt_cache_length": (c_int32, [c_void_p]),
            "gpt_profile_gemms": (ctypes.c_int, [c_void_p, c_int32]),
            "gpt_gemm_timing": (ctypes.c_int, [c_void_p, P(c_float), P(ctypes.c_double)]),
            "gpt_kernel_launches": (c_int64, [c_void_p]),
            "gpt_sync_status": (ctypes.c_int, [c_void_p]),
            "gpt_strerror": (ctypes.c_char_p, [ctypes.c_int]),
            "gpt_last_error_detail": (ctypes.c_char_p, []),
            "gpt_linear_bf16": (ctypes.c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                               c_int32, c_int32, c_int32, c_void_p]),
            "gpt_linear_decode_bf16": (ctypes.c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32,
                                                      c_int32, c_int32, c_void_p]),
            "gpt_layernorm_linear_decode_bf16": (ctypes.c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_void_p,
                                                                 c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                                                 c_int32, c_void_p]),
            "gpt_layernorm": (ctypes.c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                             c_void_p, c_void_p, c_void_p]),
            "gpt_attention_prefill": (ctypes.c_int, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32,
                                                     c_int32, c_int32, c_int32, c_void_p, c_void_p]),
            "gpt_attention_decode": (ctypes.c_int, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32,
                                                    c_int32, c_void_p, c_int32, c_void_p, c_void_p, c_void_p]),
            "gpt_sample": (ctypes.c_int, [c_void_p, c_int32, c_int32, c_float, c_int32, c_uint64, c_int32, c_void_p,
                                          c_void_p, c_void_p, c_void_p]),
            "gpt_op_status": (ctypes.c_int, []),
            "gpt_debug_bounded_wait": (ctypes.c_int, [c_int32, c_int32, c_void_p]),
            "gpt_debug_fail_allocation": (ctypes.c_int, [c_int32]),
            "gpt_attention_decode_noalloc": (ctypes.c_int, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                                            c_int32, c_int32, c_void_p, c_int32, c_void_p, c_void_p,
                                                            c_void_p, c_void_p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(code: int, where: str) -> None:
    if code != GPT_OK:
        raise GptError(code, where)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _dtype_code(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return GPT_DTYPE_BF16
    if dtype == torch.float32:
        return GPT_DTYPE_F32
    raise ValueError(f"unsupported dtype {dtype}")


# ------------------------------------------------------------------ model entry points


def gpt_create(n_layer: int, n_head: int, n_embd: int, block_size: int, vocab_size: int, bias: bool,
               dtype: torch.dtype, max_batch: int, state_dict: dict[str, torch.Tensor], page_size: int = 0,
               n_pages: int = 0) -> int:
    """Create a model from nanoGPT-named CUDA tensors of ``dtype``; returns the handle.  With
    page_size > 0 the KV cache is a pool of n_pages pages (gpt_create_paged)."""
    cfg = gpt_config_t(n_layer, n_head, n_embd, block_size, vocab_size, 1 if bias else 0, _dtype_code(dtype),
                       max_batch)
    layers = (gpt_layer_weights_t * max(n_layer, 1))()
    for l in range(n_layer):
        for field, key in zip(LAYER_FIELDS, LAYER_KEYS):
            setattr(layers[l], field, _ptr(state_dict.get(f"transformer.h.{l}.{key}")))
    w = gpt_weights_t(_ptr(state_dict["transformer.wte.weight"]), _ptr(state_dict["transformer.wpe.weight"]),
                      _ptr(state_dict["transformer.ln_f.weight"]), _ptr(state_dict.get("transformer.ln_f.bias")),
                      layers)
    handle = c_void_p()
    if page_size > 0:
        _check(lib().gpt_create_paged(ctypes.byref(cfg), ctypes.byref(w), _stream(), page_size, n_pages,
                                      ctypes.byref(handle)), "gpt_create_paged")
    else:
        _check(lib().gpt_create(ctypes.byref(cfg), ctypes.byref(w), _stream(), ctypes.byref(handle)), "gpt_create")
    return handle.value


def gpt_destroy(model: int) -> None:
    lib().gpt_destroy(model)


def gpt_prefill(model: int, tokens: torch.Tensor, logits: torch.Tensor) -> None:
    B, T = tokens.shape
    _check(lib().gpt_prefill(model, _ptr(tokens), B, T, _ptr(logits)), "gpt_prefill")


def gpt_prefill_ragged(model: int, tokens: torch.Tensor, lengths, logits: torch.Tensor) -> None:
    """Prefill sequences of different lengths: row b's first lengths[b] tokens (host lengths)."""
    B, T = tokens.shape
    lens = (ctypes.c_int32 * B)(*[int(v) for v in lengths])
    _check(lib().gpt_prefill_ragged(model, _ptr(tokens), lens, B, T, _ptr(logits)), "gpt_prefill_ragged")


def gpt_extend(model: int, tokens: torch.Tensor, logits: torch.Tensor) -> None:
    """Append a chunk of tokens (B, T) after the cache (offset causal mask)."""
    _check(lib().gpt_extend(model, _ptr(tokens), tokens.shape[1], _ptr(logits)), "gpt_extend")


def gpt_decode_step(model: int, tokens: torch.Tensor, logits: torch.Tensor) -> None:
    _check(lib().gpt_decode_step(model, _ptr(tokens), _ptr(logits)), "gpt_decode_step")


def gpt_generate(model: int, idx: torch.Tensor, max_new_tokens: int, temperature: float, top_k: int | None,
                 seed: int, out: torch.Tensor) -> None:
    B, T = idx.shape
    _check(lib().gpt_generate(model, _ptr(idx), B, T, max_new_tokens, float(temperature), top_k or 0,
                              seed & (2**64 - 1), _ptr(out)), "gpt_generate")


def gpt_last_timing(model: int) -> tuple[float, float]:
    a, b = c_float(), c_float()
    _check(lib().gpt_last_timing(model, ctypes.byref(a), ctypes.byref(b)), "gpt_last_timing")
    return a.value, b.value


def gpt_profile_gemms(model: int, enable: bool) -> None:
    _check(lib().gpt_profile_gemms(model, 1 if enable else 0), "gpt_profile_gemms")


def gpt_gemm_timing(model: int) -> tuple[float, float]:
    """(ms, FLOPs) of the Linear layers of the last timed prefill."""
    ms, fl = c_float(), ctypes.c_double()
    _check(lib().gpt_gemm_timing(model, ctypes.byref(ms), ctypes.byref(fl)), "gpt_gemm_timing")
    return ms.value, fl.value


def gpt_cache_length(model: int) -> int:
    return lib().gpt_cache_length(model)


def gpt_kernel_launches(model: int) -> int:
    return lib().gpt_kernel_launches(model)


def gpt_sync_status(model: int) -> int:
    return lib().gpt_sync_status(model)


# ------------------------------------------------------------------ stand-alone operations


def gpt_linear_bf16(A: torch.Tensor, W: torch.Tensor, bias: torch.Tensor | None, out: torch.Tensor, M: int,
                    hilo: bool = False, block_n: int = 0, splits: int = 1) -> None:
    N, K = W.shape
    _check(lib().gpt_linear_bf16(_ptr(A), _ptr(W), _ptr(bias), _ptr(out), M, N, K, 1 if hilo else 0, block_n, splits,
                                 _stream()), "gpt_linear_bf16")


def gpt_linear_decode_bf16(A: torch.Tensor, W: torch.Tensor, bias: torch.Tensor | None, out: torch.Tensor, M: int,
                           splits: int = 0) -> None:
    """out = (A[:M] + A[M:2M]) W^T (+ bias) on the decode-step kernel; A holds the hi and lo rows."""
    N, K = W.shape
    _check(lib().gpt_linear_decode_bf16(_ptr(A), _ptr(W), _ptr(bias), _ptr(out), M, N, K, splits, _stream()),
           "gpt_linear_decode_bf16")


def gpt_layernorm_linear_decode_bf16(x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor | None,
                                     W: torch.Tensor, bias: torch.Tensor | None, out: torch.Tensor, M: int,
                                     splits: int = 0, x_stride: int | None = None) -> None:
    """out = LayerNorm(x[:M]) W^T (+ bias) on the decode-step kernel, the LayerNorm inside it."""
    N, K = W.shape
    _check(lib().gpt_layernorm_linear_decode_bf16(_ptr(x), x_stride if x_stride is not None else x.stride(0),
                                                  _ptr(gamma), _ptr(beta), _ptr(W), _ptr(bias), _ptr(out), M, N, K,
                                                  splits, _stream()), "gpt_layernorm_linear_decode_bf16")


def gpt_layernorm(x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor | None, y: torch.Tensor,
                  y_lo: torch.Tensor | None = None, x_stride: int | None = None, rows: int | None = None) -> None:
    C = gamma.shape[0]
    rows = rows if rows is not None else y.shape[0]
    _check(lib().gpt_layernorm(_ptr(x), x_stride or C, _ptr(gamma), _ptr(beta), rows, C, _dtype_code(y.dtype),
                               _ptr(y), _ptr(y_lo), _stream()), "gpt_layernorm")


def gpt_attention_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, pos0: int,
                          y: torch.Tensor) -> None:
    B, nh, T, hs = q.shape
    block = k_cache.shape[2]
    _check(lib().gpt_attention_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), _dtype_code(q.dtype), B, nh, hs, T,
                                       block, pos0, _ptr(y), _stream()), "gpt_attention_prefill")


def gpt_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, pos0: torch.Tensor,
                         splits: int, y: torch.Tensor, y_lo: torch.Tensor | None = None) -> None:
    B, nh, hs = q.shape[0], q.shape[1], q.shape[-1]
    block = k_cache.shape[2]
    _check(lib().gpt_attention_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _dtype_code(q.dtype), B, nh, hs, block,
                                      _ptr(pos0), splits, _ptr(y), _ptr(y_lo), _stream()), "gpt_attention_decode")


def gpt_sample(logits: torch.Tensor, temperature: float, top_k: int | None, seed: int, step: int,
               tokens: torch.Tensor, thresholds: torch.Tensor | None = None,
               weights: torch.Tensor | None = None) -> None:
    B, V = logits.shape
    _check(lib().gpt_sample(_ptr(logits), B, V, float(temperature), top_k or 0, seed & (2**64 - 1), step,
                            _ptr(tokens), _ptr(thresholds), _ptr(weights), _stream()), "gpt_sample")


def gpt_op_status() -> int:
    return lib().gpt_op_status()


def gpt_debug_bounded_wait(limit_us: int, arrive: bool) -> None:
    """Launch the bounded-wait probe (arrive=False lets the wait run out: GPT_ETIMEOUT)."""
    _check(lib().gpt_debug_bounded_wait(limit_us, 1 if arrive else 0, _stream()), "gpt_debug_bounded_wait")


def gpt_debug_fail_allocation(k: int) -> None:
    """Fail the k-th next model allocation (0: off)."""
    _check(lib().gpt_debug_fail_allocation(k), "gpt_debug_fail_allocation")


def gpt_attention_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, pos0: torch.Tensor,
                                 splits: int, y: torch.Tensor, y_lo: torch.Tensor | None = None,
                                 err: torch.Tensor | None = None) -> None:
    """gpt_attention_decode with its scratch in the library's fixed device array (no allocation)."""
    B, nh, hs = q.shape[0], q.shape[1], q.shape[-1]
    block = k_cache.shape[2]
    _check(lib().gpt_attention_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _dtype_code(q.dtype), B, nh, hs,
                                              block, _ptr(pos0), splits, _ptr(y), _ptr(y_lo), _ptr(err), _stream()),
           "gpt_attention_decode_noalloc")


# ------------------------------------------------------------------ convenience wrapper


class GPT:
    """A model handle plus the buffers the calls need (marshalling only)."""

    def __init__(self, n_layer, n_head, n_embd, block_size, vocab_size, bias, dtype, max_batch, state_dict,
                 page_size: int = 0, n_pages: int = 0):
        self.vocab_size = vocab_size
        self.handle = gpt_create(n_layer, n_head, n_embd, block_size, vocab_size, bias, dtype, max_batch, state_dict,
                                 page_size, n_pages)

    def prefill(self, tokens: torch.Tensor) -> torch.Tensor:
        logits = torch.empty(tokens.shape[0], self.vocab_size, device=tokens.device, dtype=torch.float32)
        gpt_prefill(self.handle, tokens, logits)
        return logits

    def prefill_ragged(self, tokens: torch.Tensor, lengths) -> torch.Tensor:
        logits = torch.empty(tokens.shape[0], self.vocab_size, device=tokens.device)
        gpt_prefill_ragged(self.handle, tokens, lengths, logits)
        return logits

    def extend(self, tokens: torch.Tensor) -> torch.Tensor:
        logits = torch.empty(tokens.shape[0], self.vocab_size, device=tokens.device)
        gpt_extend(self.handle, tokens, logits)
        return logits

    def decode_step(self, tokens: torch.Tensor) -> torch.Tensor:
        logits = torch.empty(tokens.shape[0], self.vocab_size, device=tokens.device, dtype=torch.float32)
        gpt_decode_step(self.handle, tokens, logits)
        return logits

    def generate(self, idx: torch.Tensor, max_new_tokens: int, temperature: float = 1.0, top_k: int | None = None,
                 seed: int = 0, out: torch.Tensor | None = None) -> torch.Tensor:
        B, T = idx.shape
        if out is None:
            out = torch.empty(B, T + max_new_tokens, device=idx.device, dtype=torch.int32)
        gpt_generate(self.handle, idx, max_new_tokens, temperature, top_k, seed, out)
        return out

    def sync_status(self) -> int:
        return gpt_sync_status(self.handle)

    @property
    def cache_length(self) -> int:
        return gpt_cache_length(self.handle)

    def close(self) -> None:
        if self.handle:
            gpt_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
