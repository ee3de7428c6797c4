"""Failure detection without a GPU fault (GPU): a bounded device wait that runs out comes back as
GPT_ETIMEOUT with the context still usable, and an allocation that fails inside gpt_create
returns GPT_ENOMEM with nothing left allocated.  The failure is made on purpose but safely: a
barrier nobody arrives at with a 2 ms limit, and an injected host-side allocation error."""
import ctypes

import numpy as np
import pytest
import torch

from kv_cached_generation_gpt_b300 import gpt as G
from kv_cached_generation_gpt_b300 import synthetic as syn

from gpu_common import device_state_dict, make_gpu_model

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_survives():
    assert G.gpt_op_status() == G.GPT_OK
    G.gpt_debug_bounded_wait(2000, arrive=True)
    assert G.gpt_op_status() == G.GPT_OK
    G.gpt_debug_bounded_wait(2000, arrive=False)  # nothing arrives: the wait gives up after 2 ms
    assert G.gpt_op_status() == G.GPT_ETIMEOUT
    assert G.gpt_op_status() == G.GPT_OK  # read and cleared
    # the context still runs kernels correctly
    x = torch.randn(4, 128, device="cuda")
    g = torch.ones(128, device="cuda")
    y = torch.empty(4, 128, device="cuda")
    G.gpt_layernorm(x, g, None, y)
    ref = torch.nn.functional.layer_norm(x, (128,), g, None, 1e-5)
    assert torch.allclose(y, ref, atol=1e-5)
    assert G.gpt_op_status() == G.GPT_OK
    with pytest.raises(G.GptError) as ex:
        G.gpt_debug_bounded_wait(0, arrive=True)
    assert ex.value.code == G.GPT_EINVAL


def _create(shape, dsd, max_batch, page_size=0, n_pages=0):
    """gpt_create through the C ABI without raising: (status, handle)."""
    cfg = G.gpt_config_t(shape.n_layer, shape.n_head, shape.n_embd, shape.block_size, shape.vocab_size,
                         1 if shape.bias else 0, G.GPT_DTYPE_BF16, max_batch)
    layers = (G.gpt_layer_weights_t * shape.n_layer)()
    for l in range(shape.n_layer):
        for field, key in zip(G.LAYER_FIELDS, G.LAYER_KEYS):
            t = dsd.get(f"transformer.h.{l}.{key}")
            setattr(layers[l], field, t.data_ptr() if t is not None else None)
    w = G.gpt_weights_t(dsd["transformer.wte.weight"].data_ptr(), dsd["transformer.wpe.weight"].data_ptr(),
                        dsd["transformer.ln_f.weight"].data_ptr(),
                        dsd["transformer.ln_f.bias"].data_ptr() if shape.bias else None, layers)
    handle = ctypes.c_void_p(12345)
    stream = torch.cuda.current_stream().cuda_stream
    if page_size:
        rc = G.lib().gpt_create_paged(ctypes.byref(cfg), ctypes.byref(w), stream, page_size, n_pages,
                                      ctypes.byref(handle))
    else:
        rc = G.lib().gpt_create(ctypes.byref(cfg), ctypes.byref(w), stream, ctypes.byref(handle))
    return rc, handle.value


@pytest.mark.parametrize("paged", [False, True])
def test_every_allocation_failure_in_create_leaves_nothing_behind(paged):
    # a KV cache of 384 MiB, so that leaking it (or any large buffer) shows in the free memory
    shape = syn.ModelShape(2, 2, 128, 1024, 300, True, "bf16")
    dsd = device_state_dict(shape, syn.make_weights(shape, seed=3, bias_std=0.02))
    max_batch = 384
    kw = dict(page_size=256, n_pages=max_batch * 4) if paged else {}
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    failures = 0
    try:
        for k in range(1, 200):
            G.gpt_debug_fail_allocation(k)
            rc, handle = _create(shape, dsd, max_batch, **kw)
            if rc == G.GPT_OK:  # k is past the last allocation: nothing was injected
                G.gpt_destroy(handle)
                break
            assert rc == G.GPT_ENOMEM, (k, G.lib().gpt_strerror(rc))
            assert handle is None, k
            failures += 1
            torch.cuda.synchronize()
            free = torch.cuda.mem_get_info()[0]
            assert free0 - free < (32 << 20), (k, free0 - free)
        else:
            pytest.fail("gpt_create never succeeded")
    finally:
        G.gpt_debug_fail_allocation(0)
    assert failures >= 20  # every weight, the cache, the activations and the scratch were visited
    # with the injection off the model works
    model = make_gpu_model(shape, syn.make_weights(shape, seed=3, bias_std=0.02), 2)
    logits = model.prefill(torch.from_numpy(syn.make_tokens(2, 9, 300, seed=1)).cuda())
    assert bool(torch.isfinite(logits).all())
    assert model.sync_status() == G.GPT_OK
    model.close()
    torch.cuda.synchronize()
    assert free0 - torch.cuda.mem_get_info()[0] < (32 << 20)
    assert G.lib().gpt_debug_fail_allocation(-1) == G.GPT_EINVAL
    assert np.isfinite(free0)
