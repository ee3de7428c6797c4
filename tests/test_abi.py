"""The C-ABI library builds, loads, and exports every function include/gpt.h declares (CPU only)."""
import ctypes
import os
import re

import pytest

from kv_cached_generation_gpt_b300 import build
from kv_cached_generation_gpt_b300 import gpt as G

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gpt.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**(gpt_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declares_the_model_boundary():
    names = declared_functions()
    for must in ("gpt_create", "gpt_prefill", "gpt_decode_step", "gpt_generate", "gpt_destroy"):
        assert must in names
    assert set(names) == set(G.EXPORTED)


def test_library_loads_and_exports_every_declared_symbol():
    path = build.build()
    lib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_host_side_strings_and_null_handling():
    lib = G.lib()
    assert lib.gpt_strerror(G.GPT_ECONTEXT).decode().startswith("context overflow")
    assert lib.gpt_strerror(12345).decode() == "unknown error"
    assert lib.gpt_cache_length(None) == -1
    lib.gpt_destroy(None)  # no-op
    assert lib.gpt_sync_status(None) == G.GPT_EINVAL
    assert lib.gpt_prefill(None, None, 1, 1, None) == G.GPT_EINVAL
    assert lib.gpt_create(None, None, None, None) == G.GPT_EINVAL


def test_create_rejects_bad_configs_before_touching_a_device():
    lib = G.lib()
    handle = ctypes.c_void_p()
    w = G.gpt_weights_t()
    for cfg in [G.gpt_config_t(2, 2, 100, 16, 50, 0, 1, 1),   # n_embd not a multiple of 64
                G.gpt_config_t(2, 4, 128, 16, 50, 0, 1, 1),   # head size 32 needs fp32
                G.gpt_config_t(2, 3, 192, 16, 50, 0, 0, 1),   # fp32 with head size 64 is fine, but
                G.gpt_config_t(2, 8, 128, 16, 50, 0, 0, 1),   # head size 16 is not
                G.gpt_config_t(2, 2, 128, 0, 50, 0, 1, 1),    # block_size 0
                G.gpt_config_t(2, 2, 128, 16, 0, 0, 1, 1),    # vocab 0
                G.gpt_config_t(2, 2, 128, 16, 60000, 0, 1, 1),  # vocab above the sampler's limit
                G.gpt_config_t(2, 2, 128, 16, 50, 2, 1, 1),   # bias not 0/1
                G.gpt_config_t(2, 2, 128, 16, 50, 0, 7, 1),   # dtype
                G.gpt_config_t(2, 2, 128, 16, 50, 0, 1, 0)]:  # max_batch 0
        assert lib.gpt_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(handle)) == G.GPT_EINVAL
        assert handle.value is None
    # valid config but missing weight pointers
    cfg = G.gpt_config_t(2, 2, 128, 16, 50, 0, 1, 1)
    assert lib.gpt_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(handle)) == G.GPT_EINVAL


def test_stand_alone_ops_reject_bad_arguments_on_the_host():
    lib = G.lib()
    p = ctypes.c_void_p(16)  # never dereferenced: rejected before any launch
    assert lib.gpt_linear_bf16(p, p, None, p, 4, 64, 100, 0, 0, 1, None) == G.GPT_EINVAL  # K % 64
    assert lib.gpt_linear_bf16(p, p, None, p, 4, 64, 128, 1, 256, 1, None) == G.GPT_EINVAL  # hilo + 256
    assert lib.gpt_linear_bf16(p, p, None, p, 4, 65, 128, 0, 0, 2, None) == G.GPT_EINVAL  # split with N % 16
    assert lib.gpt_layernorm(p, 96, p, None, 4, 96, 1, p, None, None) == G.GPT_EINVAL  # C % 64
    assert lib.gpt_layernorm(p, 129, p, None, 4, 128, 1, p, None, None) == G.GPT_EINVAL  # odd row stride
    assert lib.gpt_layernorm(ctypes.c_void_p(20), 128, p, None, 4, 128, 1, p, None, None) == G.GPT_EINVAL  # x % 8
    q = ctypes.c_void_p(24)  # 8-byte but not 16-byte aligned
    assert lib.gpt_linear_bf16(p, p, None, q, 4, 64, 128, 0, 0, 1, None) == G.GPT_EINVAL  # out % 16
    assert lib.gpt_linear_decode_bf16(p, p, None, q, 4, 64, 128, 0, None) == G.GPT_EINVAL  # out % 16
    assert lib.gpt_attention_prefill(q, p, p, 1, 1, 2, 64, 4, 8, 0, p, None) == G.GPT_EINVAL  # q % 16
    assert lib.gpt_attention_decode(p, q, p, 1, 1, 2, 64, 8, p, 1, p, None, None) == G.GPT_EINVAL  # k % 16
    ln_lin = lib.gpt_layernorm_linear_decode_bf16
    assert ln_lin(p, 768, p, None, p, None, p, 9, 64, 768, 0, None) == G.GPT_EINVAL  # more than 8 rows
    assert ln_lin(ctypes.c_void_p(24), 768, p, None, p, None, p, 4, 64, 768, 0, None) == G.GPT_EINVAL  # x % 16
    assert ln_lin(p, 768, ctypes.c_void_p(40), None, p, None, p, 4, 64, 768, 0, None) == G.GPT_EINVAL  # gamma
    assert ln_lin(p, 770, p, None, p, None, p, 4, 64, 768, 0, None) == G.GPT_EINVAL  # stride % 4
    assert lib.gpt_attention_prefill(p, p, p, 1, 1, 2, 64, 8, 4, 0, p, None) == G.GPT_EINVAL  # T > block
    assert lib.gpt_attention_prefill(p, p, p, 1, 1, 2, 32, 4, 8, 0, p, None) == G.GPT_EINVAL  # bf16 needs hs 64
    assert lib.gpt_sample(p, 1, 60000, ctypes.c_float(1.0), 0, 0, 0, p, None, None, None) == G.GPT_EINVAL
    assert lib.gpt_sample(p, 1, 100, ctypes.c_float(-1.0), 0, 0, 0, p, None, None, None) == G.GPT_EINVAL
