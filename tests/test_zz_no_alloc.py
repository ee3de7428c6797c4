"""gpt_attention_decode_noalloc: decode attention for callers that cannot allocate (GPU).

Such callers (a process whose device memory belongs to another allocator, or code that must
not call cudaMalloc) get the same split-KV decode attention with its scratch in the
library's fixed device array.  Its results must match gpt_attention_decode, the entry point
that keeps its scratch in library-allocated memory, on consecutive calls that reuse the
array.  This file is collected last so that a run stopping at its first failure has run
every other test already.
"""
import ctypes

import numpy as np
import pytest
import torch

from kv_cached_generation_gpt_b300 import gpt as G

pytestmark = pytest.mark.gpu


def _inputs(seed, B, nh, hs, block, t, dt):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, nh, 1, hs, generator=g).to(dt).cuda()
    k = torch.randn(B, nh, block, hs, generator=g)
    v = torch.randn(B, nh, block, hs, generator=g)
    k[:, :, t:] = float("nan")  # rows past the live length must not be read
    v[:, :, t:] = float("nan")
    pos0 = torch.tensor([t - 1], dtype=torch.int32, device="cuda")
    return q, k.to(dt).cuda(), v.to(dt).cuda(), pos0


@pytest.mark.parametrize("dt,hs,B,nh,t,splits", [
    (torch.bfloat16, 64, 64, 12, 700, 1),
    (torch.bfloat16, 64, 1, 12, 1000, 16),
    (torch.bfloat16, 64, 3, 4, 333, 5),
    (torch.float32, 32, 2, 4, 65, 3),
])
def test_noalloc_matches_allocating_entry_point_twice(dt, hs, B, nh, t, splits):
    block = 1024
    for call in range(2):  # the second call reuses the array the first one left behind
        q, kc, vc, pos0 = _inputs(100 * call + B + t, B, nh, hs, block, t, dt)
        y_ref = torch.empty(B, nh * hs, device="cuda", dtype=dt)
        lo_ref = torch.empty_like(y_ref) if dt == torch.bfloat16 else None
        G.gpt_attention_decode(q, kc, vc, pos0, splits, y_ref, lo_ref)
        y = torch.full_like(y_ref, float("nan"))
        lo = torch.full_like(y_ref, float("nan")) if dt == torch.bfloat16 else None
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        G.gpt_attention_decode_noalloc(q, kc, vc, pos0, splits, y, lo, err)
        torch.cuda.synchronize()
        assert G.gpt_op_status() == G.GPT_OK
        assert int(err.item()) == 0
        got = y.float().cpu().numpy().astype(np.float64)
        ref = y_ref.float().cpu().numpy().astype(np.float64)
        if dt == torch.bfloat16:
            got = got + lo.float().cpu().numpy()
            ref = ref + lo_ref.float().cpu().numpy()
        assert np.max(np.abs(got - ref)) < 2e-5


def test_noalloc_reports_position_errors_to_the_caller_word():
    q, kc, vc, _ = _inputs(1, 1, 2, 64, 16, 16, torch.bfloat16)
    pos0 = torch.tensor([16], dtype=torch.int32, device="cuda")  # 17 keys in a 16-row cache
    y = torch.empty(1, 128, device="cuda", dtype=torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.gpt_attention_decode_noalloc(q, kc, vc, pos0, 2, y, None, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 4  # the position bit of the error word


def test_noalloc_rejects_requests_beyond_its_scratch():
    lib = G.lib()
    p = ctypes.c_void_p(16)  # never dereferenced: the size check comes first
    # 65 x 256 (b, h) pairs: more merge tickets than the array holds (16384)
    assert lib.gpt_attention_decode_noalloc(p, p, p, 1, 65, 256, 64, 1024, p, 1, p, None, None, None) == G.GPT_ETOOBIG
    # 64 x 12 pairs x 32 splits x 66 floats = 6.5 MB of partials > 4 MiB
    assert lib.gpt_attention_decode_noalloc(p, p, p, 1, 64, 12, 64, 1024, p, 32, p, None, None, None) == G.GPT_ETOOBIG
    assert "max" in lib.gpt_last_error_detail().decode()


def test_noalloc_captured_in_a_graph_and_replayed_between_eager_calls():
    """The shared ticket area sees eager calls and graph replays of the same entry point in
    turn, with split-KV merges in both; each result must equal the allocating entry point's."""
    B, nh, hs, block, t, splits = 3, 4, 64, 256, 200, 5
    dt = torch.bfloat16
    q, kc, vc, pos0 = _inputs(7, B, nh, hs, block, t, dt)
    y_ref = torch.empty(B, nh * hs, device="cuda", dtype=dt)
    lo_ref = torch.empty_like(y_ref)
    G.gpt_attention_decode(q, kc, vc, pos0, splits, y_ref, lo_ref)
    ref = y_ref.float().cpu().numpy().astype(np.float64) + lo_ref.float().cpu().numpy()
    y = torch.zeros_like(y_ref)
    lo = torch.zeros_like(y_ref)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.gpt_attention_decode_noalloc(q, kc, vc, pos0, splits, y, lo, err)  # first call: the address is cached
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        G.gpt_attention_decode_noalloc(q, kc, vc, pos0, splits, y, lo, err)
    for _ in range(2):
        for replay in (False, True):
            y.zero_()
            lo.zero_()
            if replay:
                graph.replay()
            else:
                G.gpt_attention_decode_noalloc(q, kc, vc, pos0, splits, y, lo, err)
            torch.cuda.synchronize()
            assert G.gpt_op_status() == G.GPT_OK
            assert int(err.item()) == 0
            got = y.float().cpu().numpy().astype(np.float64) + lo.float().cpu().numpy()
            assert np.max(np.abs(got - ref)) < 2e-5, replay
