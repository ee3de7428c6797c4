"""The algorithmic work bench.py divides by, checked against the closed forms of the workloads:
decode bytes per step (every bf16 weight once, the KV cache through the new position, the new
K/V rows, the fp32 logits written and read) and prefill FLOPs (the Linear layers on every
prompt token, causal attention over the visible half, the lm_head on the last position)."""
import importlib.util
import os

import pytest

from kv_cached_generation_gpt_b300 import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_arith_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _closed_form_decode_bytes(L, C, V, B, P, steps):
    weights = 2 * (12 * L * C * C + V * C)
    # sum over steps i of the keys attended, P + i + 1: an arithmetic series
    keys = steps * (P + 1) + steps * (steps - 1) // 2
    kv = (2 * L * B * C * 2) * keys / steps + 2 * L * B * C * 2
    return weights + kv + 2 * B * V * 4


@pytest.mark.parametrize("name,expect_mb", [
    ("gpt2_124m_b1_p128_d896", 268.8),     # B = 1: weights dominate
    ("gpt2_124m_b64_p512_d512", 2088.4),   # B = 64: the KV cache dominates
    ("gpt2_350m_b8_p768_d256", 1415.9),
])
def test_decode_step_bytes(name, expect_mb):
    b = _bench()
    wl = syn.WORKLOADS[name]
    s = wl.model
    got = b.decode_step_bytes(s, wl.batch, wl.prompt, wl.decode_steps)
    assert got == pytest.approx(_closed_form_decode_bytes(s.n_layer, s.n_embd, s.vocab_size, wl.batch, wl.prompt,
                                                          wl.decode_steps), rel=1e-12)
    assert got / 1e6 == pytest.approx(expect_mb, abs=0.1)


def test_headline_roofline_rate():
    b = _bench()
    wl = syn.WORKLOADS[b.WORKLOAD]
    step = b.decode_step_bytes(wl.model, wl.batch, wl.prompt, wl.decode_steps)
    # 64 tokens per step at 6,471.4 GB/s (one B300 copy-bandwidth measurement): ~198.3k tok/s
    assert wl.batch * 6471.4e9 / step == pytest.approx(198.3e3, rel=1e-3)


@pytest.mark.parametrize("name,gemm_tflop,total_tflop", [
    ("gpt2_124m_b64_p512_d512", 5.566, 5.881),
    ("gpt2_350m_b8_p768_d256", None, 3.944),
])
def test_prefill_flops(name, gemm_tflop, total_tflop):
    b = _bench()
    wl = syn.WORKLOADS[name]
    s = wl.model
    B, P, L, C, V = wl.batch, wl.prompt, s.n_layer, s.n_embd, s.vocab_size
    got = b.prefill_flops(s, B, P)
    assert got == 2 * B * P * 12 * L * C * C + 2 * C * P * (P + 1) * L * B + 2 * B * C * V
    if gemm_tflop is not None:
        assert 2 * B * P * 12 * L * C * C / 1e12 == pytest.approx(gemm_tflop, abs=5e-4)
    assert got / 1e12 == pytest.approx(total_tflop, abs=5e-4)


def test_decode_attention_bytes_per_launch():
    b = _bench()
    # B = 64, 12 heads of 64, 768 keys: K and V rows read once, q read, y hi and lo written
    assert b.decode_attn_bytes(64, 12, 64, 768) == 2 * 64 * 12 * 768 * 64 * 2 + 64 * 12 * 64 * 2 * 3


def test_committed_attention_profile_describes_the_kernel_source():
    """The ncu summary behind the roofline's `traffic` was taken on the committed decode
    attention source (its recorded hash matches), and its DRAM bytes per launch are the
    algorithmic bytes of that capture (32 sequences, 12 heads, 768 keys) within 2 %: no
    re-reads."""
    import hashlib
    b = _bench()
    src = hashlib.sha256(open(b.ATTN_SOURCE, "rb").read()).hexdigest()[:16]
    text = open(b.ATTN_PROFILE).read()
    assert f"source_sha256_16: {src}" in text
    traffic = b.attn_traffic_per_launch()
    assert traffic is not None
    algorithmic = b.decode_attn_bytes(32, 12, 64, 768)
    assert algorithmic <= traffic <= 1.02 * algorithmic


def test_cpu_baseline_thread_count_follows_the_blas_limit():
    """cpu_baseline reports the threads numpy's BLAS ran with: a one-thread limit on the BLAS
    pools (numpy's and scipy's, loaded with the oracle) reads back as 1, whatever other thread
    pools (torch's OpenMP) hold."""
    threadpoolctl = pytest.importorskip("threadpoolctl")
    import oracle.gpt  # noqa: F401
    import oracle.sampler  # noqa: F401

    b = _bench()
    with threadpoolctl.threadpool_limits(limits=1, user_api="blas"):
        assert b.blas_threads() == 1
    assert b.blas_threads() >= 1
