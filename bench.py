#!/usr/bin/env python
"""Benchmark of KV-cached GPT-2 124M generation on B300 (one JSON line on rank 0).

Headline workload (gpt2_124m_b64_p512_d512): GPT-2 124M (12 x 768, vocab 50304, bias=False,
tied lm_head), bf16 random-init weights, batch 64, 512-token uniform-random prompts, then 512
KV-cached decode steps with temperature 1.0 / top-k 50 sampling per row.  One bench step is
one gpt_generate call: prefill 512 tokens, draw, and 512 decode steps each with its draw
(the cache ends at block_size = 1024).  `value` is decode tokens/s (64 x 512 tokens per step
over the device time of the decode part, CUDA events inside the call).

Also reported: prefill tok/s and its fraction of dense bf16 peak, B=1 decode tok/s
(gpt2_124m_b1_p128_d896), the roofline of the dominant kernel (decode attention streaming
the KV cache), an end-to-end number through the C ABI with host buffers, and the CPU oracle
timed on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU (torchrun): every rank runs an independent replica (no collective on the data
path); value = all ranks' decode tokens / max over ranks of the decode time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GPT-2 124M KV-cache decode tok/s (B=1,64), prefill tok/s, % HBM/TC roofline"
WORKLOAD = "gpt2_124m_b64_p512_d512"
B1_WORKLOAD = "gpt2_124m_b1_p128_d896"
# char-level model (21 MB of weights: L2-resident, the HBM fraction is nominal) and the
# 350M-shape model with biases
SECONDARY_WORKLOADS = ("char_b1_p1_d255", "gpt2_350m_b8_p768_d256")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
ATTN_PROFILE = os.path.join(ROOT, "profiles", "attn_decode_b32_gpt2_124m.md")
ATTN_SOURCE = os.path.join(ROOT, "kv_cached_generation_gpt_b300", "csrc", "attention.cuh")


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


def prefill_flops(shape, B, P):
    """Algorithmic prefill FLOPs: the Linear layers on every prompt token, causal attention
    (q k^T and p v over the visible half), and the lm_head on the last position only."""
    C, L, V = shape.n_embd, shape.n_layer, shape.vocab_size
    gemm = 2 * B * P * 12 * L * C * C
    attn = 2 * C * P * (P + 1) * L * B
    head = 2 * B * C * V
    return gemm + attn + head


def decode_step_bytes(shape, B, P, steps):
    """Algorithmic HBM bytes of one decode step, averaged over the workload's steps: every bf16
    weight read once (the Linear layers and the tied lm_head), the KV cache read up to and
    including the new position and the new K/V rows written, and the fp32 logits written by the
    lm_head and read by the sampler.  Step i appends at position P + i."""
    C, L, V = shape.n_embd, shape.n_layer, shape.vocab_size
    weights = 2 * (12 * L * C * C + V * C)
    logits = 2 * B * V * 4
    kv = sum(2 * L * B * (P + i + 1) * C * 2 + 2 * L * B * C * 2 for i in range(steps)) / steps
    return weights + kv + logits


def secondary_workload(G, syn, name, dev, seed, hbm):
    """Prefill and decode rates of another workload configuration (one gpt_generate per run:
    a prefill of the prompt, then the workload's decode steps; median of 3 runs after one
    warm-up), with the decode step's fraction of the HBM roofline."""
    import torch

    wl = syn.WORKLOADS[name]
    shape = wl.model
    sd = {k: torch.from_numpy(v).to(torch.bfloat16).to(dev)
          for k, v in syn.make_weights(shape, bias_std=wl.bias_std).items()}
    model = G.GPT(shape.n_layer, shape.n_head, shape.n_embd, shape.block_size, shape.vocab_size, shape.bias,
                  torch.bfloat16, wl.batch, sd)
    del sd
    prompt = torch.from_numpy(syn.make_tokens(wl.batch, wl.prompt, wl.token_hi)).to(dev)
    N = wl.decode_steps + 1
    out = torch.empty(wl.batch, wl.prompt + N, dtype=torch.int32, device=dev)
    pre, dec = [], []
    for i in range(4):
        G.gpt_generate(model.handle, prompt, N, wl.temperature, wl.top_k, seed, out)
        a, b = G.gpt_last_timing(model.handle)
        if i >= 1:
            pre.append(a)
            dec.append(b)
    if model.sync_status() != G.GPT_OK:
        raise RuntimeError(f"device error word after {name}")
    model.close()
    step_s = statistics.median(dec) / 1000.0 / wl.decode_steps
    step_bytes = decode_step_bytes(shape, wl.batch, wl.prompt, wl.decode_steps)
    return {"workload": name, "prefill_tok_s": wl.batch * wl.prompt / (statistics.median(pre) / 1000.0),
            "prefill_tflops": prefill_flops(shape, wl.batch, wl.prompt) / (statistics.median(pre) / 1000.0) / 1e12,
            "decode_tok_s": wl.batch / step_s, "decode_step_us": step_s * 1e6,
            "decode_frac_of_hbm": step_bytes / step_s / 1e9 / hbm,
            "decode_bytes_per_step": step_bytes}


def attention_leg(G, torch, dev, rows, nh, hs, block, P, N):
    """Decode attention over `rows` sequences, one launch per cache length of the workload
    (t = P+1 .. P+N-1), CUDA events around each launch on torch's current stream; returns
    (rows, mean algorithmic bytes per launch, achieved GB/s)."""
    kc = torch.randn(rows, nh, block, hs, device=dev).to(torch.bfloat16)
    vc = torch.randn(rows, nh, block, hs, device=dev).to(torch.bfloat16)
    q = torch.randn(rows, nh, 1, hs, device=dev).to(torch.bfloat16)
    y = torch.empty(rows, nh * hs, device=dev, dtype=torch.bfloat16)
    ylo = torch.empty_like(y)
    pos = torch.arange(P, P + N - 1, dtype=torch.int32, device=dev)  # cache length before each append
    for i in range(3):
        G.gpt_attention_decode(q, kc, vc, pos[i:i + 1], 1, y, ylo)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(N - 1)]
    # A spin kernel at the head of the stream holds the GPU while the host enqueues every
    # launch with its two events, so that each event pair brackets exactly one kernel (from
    # the end of the previous one) and never host time between launches.
    torch.cuda._sleep(int(2e8))
    for i, (a, b) in enumerate(evs):
        a.record()
        G.gpt_attention_decode(q, kc, vc, pos[i:i + 1], 1, y, ylo)
        b.record()
    torch.cuda.synchronize()
    assert G.gpt_op_status() == G.GPT_OK
    durs = [a.elapsed_time(b) / 1000.0 for a, b in evs]
    bytes_per_launch = statistics.mean(decode_attn_bytes(rows, nh, hs, P + 1 + i) for i in range(N - 1))
    return rows, bytes_per_launch, bytes_per_launch / statistics.mean(durs) / 1e9


def decode_attn_bytes(B, nh, hs, t):
    """Algorithmic bytes of one decode-attention launch with t cached keys: K and V rows read
    once, q read, y (hi and lo halves) written, all bf16."""
    return 2 * B * nh * t * hs * 2 + B * nh * hs * 2 + 2 * B * nh * hs * 2


# ------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", self.gpu_id], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ CPU oracle


def blas_threads() -> int:
    """Threads numpy's BLAS runs with (all usable host cores unless capped by the environment
    or a threadpool limit); other thread pools in the process (torch's OpenMP) do not count."""
    try:
        from threadpoolctl import threadpool_info

        return max([i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"] or [1])
    except ImportError:
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            if os.environ.get(var, "").isdigit():
                return int(os.environ[var])
        return len(os.sched_getaffinity(0))


def oracle_sample(n_rows: int, n_decode: int):
    """Time the oracle on `n_rows` sequences of the headline workload: 512-token prefill, then
    n_decode KV-cached steps with the workload's sampling.  Returns (prefill tok/s, decode tok/s,
    threads, seconds)."""
    from kv_cached_generation_gpt_b300 import synthetic as syn
    from oracle import gpt as og
    from oracle import sampler as osm

    wl = syn.WORKLOADS[WORKLOAD]
    shape = wl.model
    sd = syn.storage_values(shape, syn.make_weights(shape))
    cfg = og.Config(shape.n_layer, shape.n_head, shape.n_embd, shape.block_size, shape.vocab_size, shape.bias)
    w = og.weights_from_state_dict(cfg, sd)
    prompt = syn.make_tokens(wl.batch, wl.prompt, wl.token_hi)[:n_rows]
    t0 = time.perf_counter()
    logits, cache = og.prefill(cfg, w, prompt)
    t1 = time.perf_counter()
    for j in range(n_decode):
        tok = osm.sample(logits.astype(np.float32), wl.temperature, wl.top_k, 1, j)
        logits, cache = og.decode(cfg, w, cache, tok)
    t2 = time.perf_counter()
    threads = blas_threads()
    return n_rows * wl.prompt / (t1 - t0), n_rows * n_decode / (t2 - t1), threads, t2 - t0


ONE_THREAD_ENV = {"OPENBLAS_NUM_THREADS": "1", "OMP_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}


def oracle_single_thread(n_rows: int = 1, n_decode: int = 2):
    """The oracle's decode rate with numpy's BLAS held to one thread: a fresh interpreter (this
    file's --oracle-leg mode) started with the BLAS thread variables set to 1, on a smaller sample
    (one sequence's 512-token prefill and two decode steps)."""
    env = dict(os.environ, **ONE_THREAD_ENV)
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-leg", f"{n_rows},{n_decode}"],
                         env=env, capture_output=True, text=True, timeout=600)
    if res.returncode != 0:
        raise RuntimeError(res.stderr[-300:])
    pre, dec, threads, secs = json.loads(res.stdout.strip().splitlines()[-1])
    return {"value": dec, "unit": "tok/s", "cores": threads, "seconds": secs, "prefill_tok_s": pre,
            "sample": f"{n_rows} sequence: {syn_prompt_len()}-token prefill + {n_decode} decode steps, "
                      f"BLAS held to one thread"}


def syn_prompt_len() -> int:
    from kv_cached_generation_gpt_b300 import synthetic as syn

    return syn.WORKLOADS[WORKLOAD].prompt


def host_facts() -> dict:
    """Host CPU count and model (from /proc/cpuinfo)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"host_cpus": os.cpu_count(), "usable_cpus": len(os.sched_getaffinity(0)), "cpu_model": model}


def oracle_configs(max_b1_steps: int = 48):
    """The oracle on the other workload configurations: the tiny (fp32, greedy) and char-level
    (temperature 0.8, top-k 200) ones in full, GPT-2 124M at batch 1 on a bounded sample (its
    128-token prefill and the first max_b1_steps of its 896 decode steps)."""
    from kv_cached_generation_gpt_b300 import synthetic as syn
    from oracle import gpt as og
    from oracle import sampler as osm

    rows = []
    for name, n_dec in (("tiny_b1_p16_d32", None), ("char_b1_p1_d255", None), (B1_WORKLOAD, max_b1_steps)):
        wl = syn.WORKLOADS[name]
        shape = wl.model
        n = wl.decode_steps if n_dec is None else min(n_dec, wl.decode_steps)
        sd = syn.storage_values(shape, syn.make_weights(shape, bias_std=wl.bias_std))
        cfg = og.Config(shape.n_layer, shape.n_head, shape.n_embd, shape.block_size, shape.vocab_size, shape.bias)
        w = og.weights_from_state_dict(cfg, sd)
        prompt = syn.make_tokens(wl.batch, wl.prompt, wl.token_hi)
        t0 = time.perf_counter()
        logits, cache = og.prefill(cfg, w, prompt)
        t1 = time.perf_counter()
        for j in range(n):
            tok = osm.sample(logits.astype(np.float32), wl.temperature, wl.top_k, 1, j)
            logits, cache = og.decode(cfg, w, cache, tok)
        t2 = time.perf_counter()
        rows.append({"workload": name, "prefill_tok_s": wl.batch * wl.prompt / (t1 - t0),
                     "decode_tok_s": wl.batch * n / (t2 - t1), "decode_steps_timed": n,
                     "full": n == wl.decode_steps})
    return rows


# ------------------------------------------------------------------ reference arm (the oracle)


def run_reference(args, rank):
    if rank != 0:
        return
    from kv_cached_generation_gpt_b300 import synthetic as syn

    wl = syn.WORKLOADS[WORKLOAD]
    rows, dec = 2, 4
    for _ in range(args.warmup):
        oracle_sample(rows, dec)
    vals, secs = [], []
    threads = 1
    for _ in range(args.steps):
        _, d, threads, s = oracle_sample(rows, dec)
        vals.append(d)
        secs.append(s)
    value = statistics.median(vals)
    sample = f"{rows} of {wl.batch} sequences, {wl.prompt}-token prefill + {dec} decode steps per bench step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * statistics.median(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded random-init GPT-2 124M weights rounded to bf16, uniform token ids)",
        "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": threads, "kind": "oracle", "sample": sample,
                         **host_facts()},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def aggregate_replicas(local: dict, world: int, device) -> dict:
    """Whole-job times of N independent replicas (one per rank, no exchange on the data path):
    every timed quantity is the maximum over ranks (the job ends when its slowest replica does);
    whole-job throughput is then all ranks' units over that time."""
    if world <= 1:
        return dict(local)
    import torch
    import torch.distributed as dist

    keys = sorted(local)
    t = torch.tensor([float(local[k]) for k in keys], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return dict(zip(keys, t.tolist()))


def workload_config(wl):
    return {"workload": wl.name, "batch": wl.batch, "prompt_tokens": wl.prompt, "decode_steps": wl.decode_steps,
            "temperature": wl.temperature, "top_k": wl.top_k,
            "l2": "inputs larger than L2: 248 MB of weights and a 2.4 GB KV cache per step (126 MB L2)"}


# ------------------------------------------------------------------ our arm


def attn_traffic_per_launch():
    """dram bytes per decode-attention launch from the committed ncu summary, if it was taken
    on the current source of the kernel (else None)."""
    try:
        text = open(ATTN_PROFILE).read()
        src = hashlib.sha256(open(ATTN_SOURCE, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha256_16") != src:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from kv_cached_generation_gpt_b300 import build
    from kv_cached_generation_gpt_b300 import gpt as G
    from kv_cached_generation_gpt_b300 import synthetic as syn

    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pk, pk_kind = peaks()

    wl = syn.WORKLOADS[WORKLOAD]
    shape = wl.model
    sd = {k: torch.from_numpy(v).to(torch.bfloat16).to(dev) for k, v in syn.make_weights(shape).items()}
    model = G.GPT(shape.n_layer, shape.n_head, shape.n_embd, shape.block_size, shape.vocab_size, shape.bias,
                  torch.bfloat16, wl.batch, sd)
    del sd
    B, P, N = wl.batch, wl.prompt, wl.decode_steps + 1  # N draws = 1 after prefill + one per decode step
    prompt = torch.from_numpy(syn.make_tokens(B, P, wl.token_hi)).to(dev)
    out = torch.empty(B, P + N, dtype=torch.int32, device=dev)
    seed = 1234 + rank

    def step():
        G.gpt_generate(model.handle, prompt, N, wl.temperature, wl.top_k, seed, out)
        return G.gpt_last_timing(model.handle)

    for _ in range(max(args.warmup, 3)):
        step()
    assert model.sync_status() == G.GPT_OK

    gpu_id = str(local_rank)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(gpu_id) if rank == 0 else None
    if clocks:
        clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = G.gpt_kernel_launches(model.handle)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("bench_timed")  # lets ncu restrict a launch list to the timed steps
    ev0.record()
    pre_ms, dec_ms = [], []
    for _ in range(args.steps):
        a, b = step()
        pre_ms.append(a)
        dec_ms.append(b)
    ev1.record()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    if world > 1:
        dist.barrier()
    total_ms = ev0.elapsed_time(ev1)
    launches = G.gpt_kernel_launches(model.handle) - launches0
    clk = clocks.stop() if clocks else None
    status = model.sync_status()
    if status != G.GPT_OK:
        raise RuntimeError(f"device error word after the timed region: {G.lib().gpt_strerror(status).decode()}")

    agg = aggregate_replicas({"decode_s": sum(dec_ms) / 1000.0, "prefill_s": sum(pre_ms) / 1000.0,
                              "total_ms": total_ms}, world, dev)
    dec_s, pre_s, total_ms = agg["decode_s"], agg["prefill_s"], agg["total_ms"]
    dec_tokens = world * args.steps * B * (N - 1)
    value = dec_tokens / dec_s
    prefill_tok_s = world * args.steps * B * P / pre_s
    pf = prefill_flops(shape, B, P)
    prefill_tflops = world * args.steps * pf / pre_s / 1e12

    # ---- end to end through the C ABI with host buffers (rank-local, same metric)
    h_prompt = torch.from_numpy(syn.make_tokens(B, P, wl.token_hi)).pin_memory()
    h_out = torch.empty(B, P + N, dtype=torch.int32).pin_memory()
    d_prompt = torch.empty_like(prompt)
    torch.cuda.synchronize()
    e2e_s = []
    for _ in range(max(2, args.steps)):
        t0 = time.perf_counter()
        d_prompt.copy_(h_prompt, non_blocking=True)
        G.gpt_generate(model.handle, d_prompt, N, wl.temperature, wl.top_k, seed, out)
        h_out.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        e2e_s.append(time.perf_counter() - t0)
    e2e_value = B * N / statistics.median(e2e_s)

    # ---- prefill GEMMs alone: CUDA events around each Linear-layer launch of a prefill
    #      (on the model's stream), three prefills of the workload's prompts, median
    G.gpt_profile_gemms(model.handle, True)
    gemm_ms, gemm_flops = [], 0.0
    logits = torch.empty(B, shape.vocab_size, device=dev)
    for _ in range(3):
        G.gpt_prefill(model.handle, prompt, logits)
        ms, fl = G.gpt_gemm_timing(model.handle)
        gemm_ms.append(ms)
        gemm_flops = fl
    G.gpt_profile_gemms(model.handle, False)
    gemm_tflops = gemm_flops / (statistics.median(gemm_ms) / 1000.0) / 1e12

    # ---- B = 1 decode (secondary line of the same metric)
    b1 = syn.WORKLOADS[B1_WORKLOAD]
    p1 = torch.from_numpy(syn.make_tokens(b1.batch, b1.prompt, b1.token_hi)).to(dev)
    o1 = torch.empty(1, b1.prompt + b1.decode_steps + 1, dtype=torch.int32, device=dev)
    b1_dec, b1_pre = [], []
    for i in range(4):
        G.gpt_generate(model.handle, p1, b1.decode_steps + 1, 1.0, b1.top_k, seed, o1)
        a, b = G.gpt_last_timing(model.handle)
        if i >= 1:
            b1_pre.append(a)
            b1_dec.append(b)
    b1_tok_s = b1.decode_steps / (statistics.median(b1_dec) / 1000.0)
    b1_weight_bytes = 2 * (12 * shape.n_layer * shape.n_embd ** 2 + shape.vocab_size * shape.n_embd)

    # ---- the other configurations of the measurement table (rank 0 only)
    secondary = []
    if rank == 0:
        for name in SECONDARY_WORKLOADS:
            secondary.append(secondary_workload(G, syn, name, dev, seed, pk["hbm_gbs"]))

    # ---- dominant kernel: decode attention, one launch per cache length of the workload, at the
    #      32-sequence half batch the decode graph issues (two chains), and at 64 sequences
    nh, hs = shape.n_head, shape.n_embd // shape.n_head
    half, bytes_per_launch, achieved = attention_leg(G, torch, dev, B // 2, nh, hs, shape.block_size, P, N)
    _, bytes_b64, achieved_b64 = attention_leg(G, torch, dev, B, nh, hs, shape.block_size, P, N)

    # ---- CPU oracle on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows, dec = 2, 6
        _, d, threads, _ = oracle_sample(rows, dec)
        cpu = {"value": d, "unit": "tok/s", "cores": threads, "kind": "oracle",
               "sample": f"{rows} of {B} sequences: {P}-token prefill + {dec} decode steps with the workload's "
                         f"sampling, fp64 numpy on the host"}
        cpu.update(host_facts())
        try:
            cpu["single_thread"] = oracle_single_thread()
        except Exception as ex:  # a reported extra: never let it cost the bench line
            cpu["single_thread"] = {"error": str(ex)[:200]}
        try:
            cpu["configs"] = oracle_configs()
        except Exception as ex:
            cpu["configs"] = {"error": str(ex)[:200]}

    if rank != 0:
        return
    hbm = pk["hbm_gbs"]
    step_bytes = decode_step_bytes(shape, B, P, N - 1)
    step_gbs = step_bytes * args.steps * (N - 1) / dec_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded random-init GPT-2 124M weights in bf16, uniform token ids)",
        "config": workload_config(wl),
        "roofline": {"bound": "hbm",
                     "kernel": f"attn_decode_bulk<bf16,64> at {half} sequences (one decode chain), launched alone",
                     "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": attn_traffic_per_launch(),
                     "algorithmic_bytes_per_launch": bytes_per_launch, "peak_source": pk_kind,
                     "launches_timed": N - 1,
                     "at_64_sequences": {"achieved": achieved_b64, "frac": achieved_b64 / hbm,
                                         "algorithmic_bytes_per_launch": bytes_b64}},
        "prefill": {"tok_s": prefill_tok_s, "tflops": prefill_tflops, "ms": 1000 * pre_s / args.steps / world,
                    "frac_of_bf16_peak": prefill_tflops / pk["bf16_tflops"], "peak_source": pk_kind},
        "prefill_gemm": {"tflops": gemm_tflops, "ms": statistics.median(gemm_ms), "flops": gemm_flops,
                         "frac_of_bf16_peak": gemm_tflops / pk["bf16_tflops"],
                         "frac_of_bf16_sustained": gemm_tflops / pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                         "method": "CUDA events around each Linear-layer launch of a 64 x 512 prefill (lm_head "
                                   "excluded), on the model's stream; median of 3"},
        "decode_step": {"bytes_per_step": step_bytes, "achieved_gbs": step_gbs, "peak_gbs": hbm,
                        "frac_of_hbm": step_gbs / hbm, "roofline_tok_s": B * hbm * 1e9 / step_bytes,
                        "note": "weights + KV cache + logits bytes per decode step (mean over the workload's "
                                "steps) over the measured decode time per step"},
        "secondary": secondary,
        "decode_b1": {"workload": b1.name, "tok_s": b1_tok_s,
                      "weight_stream_gbs": b1_weight_bytes * b1_tok_s / 1e9,
                      "frac_of_hbm_weights_only": b1_weight_bytes * b1_tok_s / 1e9 / hbm,
                      "prefill_ms": statistics.median(b1_pre)},
        "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": int(B * P * 4),
                "d2h_bytes_per_step": int(B * (P + N) * 4),
                "note": "new tokens per second of a whole gpt_generate call (prefill included) with the prompt "
                        "copied from pinned host memory and the output copied back"},
        "gpu_launches": int(launches),
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    model.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-leg", default=None, help=argparse.SUPPRESS)  # "rows,decode": CPU only
    args = ap.parse_args()
    if args.oracle_leg:
        rows, dec = (int(v) for v in args.oracle_leg.split(","))
        print(json.dumps(list(oracle_sample(rows, dec))), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
