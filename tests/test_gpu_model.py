"""Whole-model parity through the C ABI: teacher-forced logits against the oracle (GPU).

Tolerances: fp32 model 1e-3 max abs on every step's logits; bf16 models 5e-2 max abs
and at least 99% agreement of the greedy argmax over all checked (row, step) pairs.
"""
import numpy as np
import pytest
import torch

from kv_cached_generation_gpt_b300 import gpt as G
from kv_cached_generation_gpt_b300 import synthetic as syn
from oracle import gpt as og
from oracle import sampler as osm

from gpu_common import argmax_agreement, gpu_teacher_forced, make_gpu_model, oracle_model

pytestmark = pytest.mark.gpu

BF16_TOL = 5e-2
F32_TOL = 1e-3


def _weights(wl: syn.Workload):
    return syn.make_weights(wl.model, bias_std=wl.bias_std)


def test_tiny_f32_greedy_teacher_forced():
    """tiny_b1_p16_d32: fp32 weights, 32 greedy decode steps, the oracle's greedy tokens fed to both."""
    wl = syn.WORKLOADS["tiny_b1_p16_d32"]
    sd = _weights(wl)
    cfg, w = oracle_model(wl.model, sd)
    prompt = syn.make_tokens(wl.batch, wl.prompt, wl.token_hi)
    fed, ref = og.teacher_forced(cfg, w, prompt, n_steps=wl.decode_steps)
    model = make_gpu_model(wl.model, sd, wl.batch)
    got = gpu_teacher_forced(model, prompt, fed)
    assert got.shape == ref.shape
    assert np.max(np.abs(got - ref)) < F32_TOL
    assert argmax_agreement(got, ref) == 1.0
    assert model.cache_length == wl.prompt + wl.decode_steps


@pytest.mark.parametrize("shape,B,P,N,bias_std", [
    (syn.ModelShape(2, 2, 128, 96, 300, True, "bf16"), 3, 9, 20, 0.05),
    (syn.ModelShape(3, 3, 192, 80, 1000, False, "bf16"), 2, 65, 15, None),  # C % 128 != 0, ragged prompt tile
    (syn.ModelShape(1, 4, 256, 64, 129, True, "f32"), 2, 30, 34, None),     # fills block_size exactly
])
def test_small_models_teacher_forced(shape, B, P, N, bias_std):
    sd = syn.make_weights(shape, seed=21, bias_std=bias_std, random_gamma=True)
    cfg, w = oracle_model(shape, sd)
    prompt = syn.make_tokens(B, P, shape.vocab_size, seed=3)
    forced = syn.make_tokens(B, N, shape.vocab_size, seed=4)
    _, ref = og.teacher_forced(cfg, w, prompt, forced)
    got = gpu_teacher_forced(make_gpu_model(shape, sd, B + 1), prompt, forced)
    tol = F32_TOL if shape.dtype == "f32" else BF16_TOL
    assert np.max(np.abs(got - ref)) < tol
    assert argmax_agreement(got, ref) >= 0.99


def test_char_b1_p1_d255_sampled_tokens_teacher_forced():
    """char_b1_p1_d255: the oracle's own temperature-0.8 / top-200 draws are fed to both sides."""
    wl = syn.WORKLOADS["char_b1_p1_d255"]
    sd = _weights(wl)
    cfg, w = oracle_model(wl.model, sd)
    prompt = syn.make_tokens(wl.batch, wl.prompt, wl.token_hi)
    seq = og.generate(cfg, w, prompt, wl.decode_steps + 1, wl.temperature, wl.top_k, seed=5)
    forced = seq[:, wl.prompt:wl.prompt + wl.decode_steps]
    _, ref = og.teacher_forced(cfg, w, prompt, forced)
    got = gpu_teacher_forced(make_gpu_model(wl.model, sd, wl.batch), prompt, forced)
    assert np.max(np.abs(got - ref)) < BF16_TOL
    assert argmax_agreement(got, ref) >= 0.99


def test_gpt2_124m_b1_greedy_teacher_forced():
    """gpt2_124m_b1_p128_d896: 896 greedy steps, the oracle's greedy tokens fed to both (fills 1024)."""
    wl = syn.WORKLOADS["gpt2_124m_b1_p128_d896"]
    sd = _weights(wl)
    cfg, w = oracle_model(wl.model, sd)
    prompt = syn.make_tokens(wl.batch, wl.prompt, wl.token_hi)
    fed, ref = og.teacher_forced(cfg, w, prompt, n_steps=wl.decode_steps)
    got = gpu_teacher_forced(make_gpu_model(wl.model, sd, wl.batch), prompt, fed)
    err = np.max(np.abs(got - ref))
    agree = argmax_agreement(got, ref)
    print(f"gpt2_124m B=1: max|err| {err:.3e}, argmax agreement {agree:.4f}")
    assert err < BF16_TOL
    assert agree >= 0.99


@pytest.mark.parametrize("name,rows", [("gpt2_124m_b64_p512_d512", [0, 21, 42, 63]),
                                       ("gpt2_350m_b8_p768_d256", [0, 7])])
def test_full_size_sampled_rows(name, rows):
    """Full batch and cache at the benchmark's sizes.  The prefill's logits are checked for
    every row of the batch; sampled rows are then checked at every decode position against
    the oracle's no-cache forward over the whole fed sequence."""
    wl = syn.WORKLOADS[name]
    sd = _weights(wl)
    prompt = syn.make_tokens(wl.batch, wl.prompt, wl.token_hi)
    forced = syn.make_tokens(wl.batch, wl.decode_steps, wl.token_hi, seed=77)
    model = make_gpu_model(wl.model, sd, wl.batch)
    pre_all = model.prefill(torch.from_numpy(prompt).cuda()).cpu().numpy()  # (B, V), every row
    got = gpu_teacher_forced(model, prompt, forced, rows=rows)  # (N+1, rows, V)
    assert model.cache_length == wl.prompt + wl.decode_steps == wl.model.block_size
    del model
    cfg, w = oracle_model(wl.model, sd)
    pre_ref = np.concatenate([og.prefill(cfg, w, prompt[b:b + 8])[0] for b in range(0, wl.batch, 8)])
    pre_err = np.max(np.abs(pre_all - pre_ref))
    pre_agree = np.argmax(pre_all, axis=-1) == np.argmax(pre_ref, axis=-1)
    print(f"{name}: prefill of all {wl.batch} rows: max|err| {pre_err:.3e}, "
          f"argmax agreement {np.mean(pre_agree):.4f}")
    assert pre_err < BF16_TOL
    errs, agree = [], []
    for i, r in enumerate(rows):
        seq = np.concatenate([prompt[r:r + 1], forced[r:r + 1]], axis=1)
        full = og.forward_full(cfg, w, seq)[0, wl.prompt - 1:]  # positions P-1 .. P+N-1
        errs.append(np.max(np.abs(got[:, i] - full)))
        agree.append(np.argmax(got[:, i], axis=-1) == np.argmax(full, axis=-1))
    # the agreement criterion pools every checked (row, step) pair: the prefill's rows and the
    # sampled rows' decode positions
    agree = float(np.mean(np.concatenate(agree + [pre_agree])))
    print(f"{name}: max|err| {max(errs):.3e}, argmax agreement {agree:.4f}")
    assert max(errs) < BF16_TOL
    assert agree >= 0.99


def test_generate_matches_step_by_step_and_oracle_sampler():
    """gpt_generate (prefill + graph-replayed decode + draws) equals the same draws made with
    gpt_prefill / gpt_decode_step / gpt_sample, and the oracle's sampler on the GPU logits."""
    shape = syn.ModelShape(2, 2, 128, 64, 500, True, "bf16")
    sd = syn.make_weights(shape, seed=8, bias_std=0.02)
    B, T, N, temp, k, seed = 3, 5, 20, 0.9, 40, 4242
    prompt = torch.from_numpy(syn.make_tokens(B, T, 500, seed=6)).cuda()
    model = make_gpu_model(shape, sd, B)
    out = model.generate(prompt, N, temperature=temp, top_k=k, seed=seed)
    assert model.sync_status() == G.GPT_OK
    assert torch.equal(out[:, :T], prompt)
    assert model.cache_length == T + N - 1
    pre, dec = G.gpt_last_timing(model.handle)
    assert pre > 0 and dec > 0
    # replay the same computation step by step
    logits = model.prefill(prompt)
    toks = []
    for j in range(N):
        tok = torch.empty(B, dtype=torch.int32, device="cuda")
        G.gpt_sample(logits, temp, k, seed, j, tok)
        toks.append(tok)
        ref = np.array([osm.sample_row(logits[b].cpu().numpy(), temp, k, seed, b, j) for b in range(B)])
        assert np.array_equal(tok.cpu().numpy(), ref)
        if j + 1 < N:
            logits = model.decode_step(tok)
    assert torch.equal(out[:, T:], torch.stack(toks, dim=1))
    # a second generate reuses the captured graph and gives the same tokens
    out2 = model.generate(prompt, N, temperature=temp, top_k=k, seed=seed)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("B", [64, 33])  # 33: chains of 16 and 17 sequences
def test_generate_at_the_benchmark_configuration(B):
    """The path the benchmark times: GPT-2 124M, prompt 512, temperature 1.0, top_k 50, per-row
    Philox streams, with 40 draws.  (a) gpt_generate's tokens equal the step-by-step chain
    gpt_prefill -> [gpt_sample -> gpt_decode_step] with the same seed and draw indices; (b) each
    draw of the first and last row of both decode chains equals the oracle's sampler applied to
    the GPU logits of that step; (c) those logits match the oracle's no-cache forward over the
    generated sequence (teacher-forced), within the bf16 tolerance and >= 99% argmax agreement.
    ("原生 nanoGPT 模型服务首选", §2 generate(); "极速上手nanoGPT", §关键参数: temperature, top_k.)"""
    wl = syn.WORKLOADS["gpt2_124m_b64_p512_d512"]
    sd = _weights(wl)
    N, seed = 40, 20240
    P, temp, k = wl.prompt, wl.temperature, wl.top_k
    prompt = syn.make_tokens(wl.batch, P, wl.token_hi)[:B].copy()
    pd = torch.from_numpy(prompt).cuda()
    model = make_gpu_model(wl.model, sd, wl.batch)
    out = model.generate(pd, N, temperature=temp, top_k=k, seed=seed)
    assert model.sync_status() == G.GPT_OK
    assert torch.equal(out[:, :P], pd)
    B0 = B // 2
    rows = [0, B0 - 1, B0, B - 1]  # first and last rows of both chains
    logits = model.prefill(pd)
    toks, kept = [], []
    for j in range(N):
        tok = torch.empty(B, dtype=torch.int32, device="cuda")
        G.gpt_sample(logits, temp, k, seed, j, tok)
        toks.append(tok)
        lg = logits[rows].cpu().numpy()
        kept.append(lg)
        t_host = tok.cpu().numpy()
        for i, r in enumerate(rows):
            assert t_host[r] == osm.sample_row(lg[i], temp, k, seed, r, j), (r, j)
        if j + 1 < N:
            logits = model.decode_step(tok)
    assert model.sync_status() == G.GPT_OK
    assert torch.equal(out[:, P:], torch.stack(toks, dim=1))
    gen = out.cpu().numpy()
    del model
    cfg, w = oracle_model(wl.model, sd)
    got = np.stack(kept)  # (N, rows, V): logits before draw j
    errs, agree = [], []
    for i, r in enumerate(rows):
        full = og.forward_full(cfg, w, gen[r:r + 1, :P + N - 1])[0, P - 1:]  # positions P-1 .. P+N-2
        errs.append(np.max(np.abs(got[:, i] - full)))
        agree.append(np.argmax(got[:, i], axis=-1) == np.argmax(full, axis=-1))
    agree = float(np.mean(np.concatenate(agree)))
    print(f"generate B={B}: max|err| {max(errs):.3e}, argmax agreement {agree:.4f}")
    assert max(errs) < BF16_TOL
    assert agree >= 0.99


def test_generate_greedy_equals_oracle_greedy_on_fp32_model():
    wl = syn.WORKLOADS["tiny_b1_p16_d32"]
    sd = _weights(wl)
    cfg, w = oracle_model(wl.model, sd)
    prompt = syn.make_tokens(2, 16, 65, seed=2)
    ref = og.generate(cfg, w, prompt, 40, 0.0, None, 0)
    model = make_gpu_model(wl.model, sd, 2)
    out = model.generate(torch.from_numpy(prompt).cuda(), 40, temperature=0.0)
    assert model.sync_status() == G.GPT_OK
    assert np.array_equal(out.cpu().numpy(), ref)


def test_error_paths():
    shape = syn.ModelShape(1, 2, 128, 16, 100, False, "bf16")
    sd = syn.make_weights(shape, seed=1)
    model = make_gpu_model(shape, sd, 2)
    h = model.handle
    logits = torch.empty(3, 100, device="cuda")
    tok = torch.zeros(3, 16, dtype=torch.int32, device="cuda")
    assert G.lib().gpt_decode_step(h, tok.data_ptr(), logits.data_ptr()) == G.GPT_ESTATE
    assert G.lib().gpt_prefill(h, tok.data_ptr(), 3, 4, logits.data_ptr()) == G.GPT_EINVAL  # B > max_batch
    assert G.lib().gpt_prefill(h, tok.data_ptr(), 1, 17, logits.data_ptr()) == G.GPT_ECONTEXT
    # past block_size generate crops the context (see the overflow tests); 10 + 8 > 16 is fine
    assert G.lib().gpt_generate(h, tok.data_ptr(), 1, 10, 8, 1.0, 0, 0, logits.data_ptr()) == G.GPT_OK
    assert G.lib().gpt_generate(h, tok.data_ptr(), 1, 4, 2, float("nan"), 0, 0, logits.data_ptr()) == G.GPT_EINVAL
    # a token id out of range is flagged by the device error word; its embedding row is zeroed
    bad = torch.tensor([[1, 2, 100]], dtype=torch.int32, device="cuda")
    model.prefill(bad)
    assert model.sync_status() == G.GPT_ETOKEN
    assert model.sync_status() == G.GPT_OK  # cleared
    good = torch.tensor([[1, 2, 3]], dtype=torch.int32, device="cuda")
    model.prefill(good)
    for _ in range(13):
        model.decode_step(torch.tensor([5], dtype=torch.int32, device="cuda"))
    assert model.cache_length == 16
    with pytest.raises(G.GptError) as ei:
        model.decode_step(torch.tensor([5], dtype=torch.int32, device="cuda"))
    assert ei.value.code == G.GPT_ECONTEXT
    assert model.sync_status() == G.GPT_OK
    model.close()


def test_prefill_gemm_timing_counts_the_linear_layers():
    """gpt_profile_gemms: events around every prefill Linear layer; FLOPs = sum of 2 M N K."""
    shape = syn.ModelShape(2, 2, 128, 96, 300, False, "bf16")
    sd = syn.make_weights(shape, seed=5)
    model = make_gpu_model(shape, sd, 2)
    tokens = torch.from_numpy(syn.make_tokens(2, 40, shape.vocab_size, seed=6)).cuda()
    with pytest.raises(G.GptError):
        G.gpt_gemm_timing(model.handle)  # nothing timed yet
    G.gpt_profile_gemms(model.handle, True)
    model.prefill(tokens)
    ms, flops = G.gpt_gemm_timing(model.handle)
    C, L, M = shape.n_embd, shape.n_layer, 2 * 40
    assert flops == 2.0 * M * 12 * C * C * L  # c_attn 3C^2, c_proj C^2, c_fc and mlp c_proj 4C^2 each
    assert ms > 0.0
    model.decode_step(tokens[:, 0].contiguous())  # decode steps are not timed: the prefill's numbers stay
    assert G.gpt_gemm_timing(model.handle)[1] == flops
    G.gpt_profile_gemms(model.handle, False)
    assert model.sync_status() == G.GPT_OK


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_extend_appends_chunks_with_the_offset_mask(dtype):
    """gpt_extend: chunks appended after a prompt see the cache through the offset causal mask;
    each chunk's last-position logits equal the oracle's no-cache forward over everything fed,
    and decode steps continue from the extended cache."""
    shape = syn.ModelShape(2, 2, 128, 160, 300, True, dtype)
    sd = syn.make_weights(shape, seed=17, bias_std=0.05, random_gamma=True)
    cfg, w = oracle_model(shape, sd)
    B = 3
    prompt = syn.make_tokens(B, 20, shape.vocab_size, seed=1)
    chunks = [syn.make_tokens(B, n, shape.vocab_size, seed=10 + n) for n in (7, 1, 30, 64)]
    model = make_gpu_model(shape, sd, B)
    tol = F32_TOL if dtype == "f32" else BF16_TOL
    fed = prompt
    got = model.prefill(torch.from_numpy(prompt).cuda()).cpu().numpy()
    assert np.max(np.abs(got - og.forward(cfg, w, fed)[0])) < tol
    for ch in chunks:
        fed = np.concatenate([fed, ch], axis=1)
        got = model.extend(torch.from_numpy(np.ascontiguousarray(ch)).cuda()).cpu().numpy()
        ref = og.forward(cfg, w, fed)[0]
        assert np.max(np.abs(got - ref)) < tol, ch.shape
        assert model.cache_length == fed.shape[1]
    for step in range(3):  # the decode kernels read the cache the chunks wrote
        tok = syn.make_tokens(B, 1, shape.vocab_size, seed=40 + step)
        fed = np.concatenate([fed, tok], axis=1)
        got = model.decode_step(torch.from_numpy(np.ascontiguousarray(tok[:, 0])).cuda()).cpu().numpy()
        assert np.max(np.abs(got - og.forward(cfg, w, fed)[0])) < tol
    assert model.sync_status() == G.GPT_OK
    model.close()


def test_extend_errors():
    shape = syn.ModelShape(1, 2, 128, 32, 100, False, "bf16")
    sd = syn.make_weights(shape, seed=2)
    model = make_gpu_model(shape, sd, 2)
    toks = torch.from_numpy(syn.make_tokens(2, 8, shape.vocab_size, seed=3)).cuda()
    with pytest.raises(G.GptError) as ex:
        model.extend(toks)
    assert ex.value.code == G.GPT_ESTATE  # no prefill yet
    model.prefill(toks)
    model.extend(toks)
    model.extend(toks)
    model.extend(toks)  # 32 positions: the cache is full
    with pytest.raises(G.GptError) as ex:
        model.extend(toks[:, :1].contiguous())
    assert ex.value.code == G.GPT_ECONTEXT
    assert model.cache_length == 32
    assert model.sync_status() == G.GPT_OK


@pytest.mark.parametrize("T,N", [(16, 80), (70, 5)])
def test_generate_past_block_size_crops_like_the_pages(T, N):
    """Past block_size every draw sees the last block_size tokens (nanoGPT's crop, positions
    restarting at 0 in the window): fp32 tiny model, greedy, tokens equal to the oracle's
    literal generate() loop -- overflow in the middle, and a prompt longer than the block."""
    wl = syn.WORKLOADS["tiny_b1_p16_d32"]
    sd = _weights(wl)
    cfg, w = oracle_model(wl.model, sd)
    prompt = syn.make_tokens(2, T, 65, seed=7)
    ref = og.generate_cropped(cfg, w, prompt, N, 0.0, None, 0)
    model = make_gpu_model(wl.model, sd, 2)
    out = model.generate(torch.from_numpy(prompt).cuda(), N, temperature=0.0)
    assert model.sync_status() == G.GPT_OK
    assert np.array_equal(out.cpu().numpy(), ref)
    assert model.cache_length == cfg.block_size


def test_generate_past_block_size_sampled_draws_are_window_prefills():
    """bf16: each draw past the cache equals the library's own prefill of the last block_size
    tokens followed by the sampler with that draw's index."""
    shape = syn.ModelShape(2, 2, 128, 48, 300, True, "bf16")
    sd = syn.make_weights(shape, seed=23, bias_std=0.02)
    model = make_gpu_model(shape, sd, 2)
    prompt = torch.from_numpy(syn.make_tokens(2, 30, 300, seed=5)).cuda()
    out = model.generate(prompt, 30, temperature=0.9, top_k=40, seed=11).cpu()
    assert model.sync_status() == G.GPT_OK
    first_windowed = shape.block_size - 30 + 1  # draws 0..18 run on the cache
    for j in (first_windowed, first_windowed + 5, 29):
        window = out[:, 30 + j - shape.block_size:30 + j].contiguous().cuda()
        logits = model.prefill(window)
        tok = torch.empty(2, dtype=torch.int32, device="cuda")
        G.gpt_sample(logits, 0.9, 40, 11, j, tok)
        assert torch.equal(tok.cpu(), out[:, 30 + j])
    assert G.gpt_op_status() == G.GPT_OK


@pytest.mark.parametrize("dtype,B", [("bf16", 4), ("bf16", 70), ("f32", 3)])
def test_ragged_prefill_then_decode_each_sequence_at_its_own_length(dtype, B):
    """gpt_prefill_ragged: rows of different prompt lengths (padding ids -1, ignored); each
    row's logits at its own last prompt position, then decode steps appending every row at its
    own length -- all against the oracle run on each row alone."""
    shape = syn.ModelShape(2, 2, 128, 64, 300, True, dtype)
    sd = syn.make_weights(shape, seed=29, bias_std=0.05, random_gamma=True)
    cfg, w = oracle_model(shape, sd)
    r = np.random.default_rng(B)
    T = 30
    lengths = r.integers(1, T + 1, size=B)
    lengths[0], lengths[-1] = 1, T
    tokens = syn.make_tokens(B, T, shape.vocab_size, seed=31)
    for b in range(B):
        tokens[b, lengths[b]:] = -1
    model = make_gpu_model(shape, sd, B)
    tol = F32_TOL if dtype == "f32" else BF16_TOL
    seqs = [tokens[b, :lengths[b]] for b in range(B)]
    got = model.prefill_ragged(torch.from_numpy(tokens).cuda(), lengths).cpu().numpy()
    ref = np.stack([og.forward(cfg, w, s[None, :])[0][0] for s in seqs])
    assert np.max(np.abs(got - ref)) < tol
    assert model.cache_length == T
    for step in range(4):
        tok = syn.make_tokens(B, 1, shape.vocab_size, seed=50 + step)[:, 0]
        seqs = [np.concatenate([s, tok[b:b + 1]]) for b, s in enumerate(seqs)]
        got = model.decode_step(torch.from_numpy(np.ascontiguousarray(tok)).cuda()).cpu().numpy()
        ref = np.stack([og.forward(cfg, w, s[None, :])[0][0] for s in seqs])
        assert np.max(np.abs(got - ref)) < tol, step
        if dtype != "f32":
            assert argmax_agreement(got, ref) >= 0.99
    assert model.sync_status() == G.GPT_OK
    with pytest.raises(G.GptError) as ex:
        model.extend(torch.zeros(B, 2, dtype=torch.int32, device="cuda"))
    assert ex.value.code == G.GPT_ESTATE
    model.close()


@pytest.mark.parametrize("dtype,page", [("bf16", 64), ("bf16", 128), ("f32", 64)])
def test_paged_cache_gives_the_contiguous_results(dtype, page):
    """gpt_create_paged: the same kernels address the KV rows through block tables, so every
    logit is bit-identical to the contiguous cache -- prefill, decode steps across page
    boundaries, a chunk appended with gpt_extend, generate, and a ragged batch."""
    shape = syn.ModelShape(2, 2, 128, 256, 300, True, dtype)
    sd = syn.make_weights(shape, seed=37, bias_std=0.05)
    B = 3
    flat = make_gpu_model(shape, sd, B)
    paged = make_gpu_model(shape, sd, B, page_size=page, n_pages=B * (256 // page))
    prompt = torch.from_numpy(syn.make_tokens(B, 70, 300, seed=2)).cuda()
    assert torch.equal(flat.prefill(prompt), paged.prefill(prompt))
    for step in range(70):  # crosses the 128 and 192 page boundaries of page 64
        tok = torch.from_numpy(syn.make_tokens(B, 1, 300, seed=100 + step)[:, 0].copy()).cuda()
        assert torch.equal(flat.decode_step(tok), paged.decode_step(tok)), step
    chunk = torch.from_numpy(syn.make_tokens(B, 20, 300, seed=9)).cuda()
    assert torch.equal(flat.extend(chunk), paged.extend(chunk))
    p40 = prompt[:, :40].contiguous()
    assert torch.equal(flat.generate(p40, 100, temperature=0.8, top_k=30, seed=5),
                       paged.generate(p40, 100, temperature=0.8, top_k=30, seed=5))
    lens = [3, 70, 33]
    assert torch.equal(flat.prefill_ragged(prompt, lens), paged.prefill_ragged(prompt, lens))
    for step in range(5):
        tok = torch.from_numpy(syn.make_tokens(B, 1, 300, seed=200 + step)[:, 0].copy()).cuda()
        assert torch.equal(flat.decode_step(tok), paged.decode_step(tok))
    assert flat.sync_status() == G.GPT_OK and paged.sync_status() == G.GPT_OK


@pytest.mark.parametrize("B", [40, 33])  # 33: chains of 16 and 17 sequences
def test_two_chain_decode_with_paged_cache(B):
    """From 32 sequences up a decode step runs as two chains of half the batch on two streams,
    the second addressing its sequences through an offset into the cache (contiguous) or into
    the block tables (paged).  Paged and contiguous caches give bit-identical logits, across
    page boundaries, through generate and a ragged batch; rows of both chains match the
    oracle."""
    shape = syn.ModelShape(2, 2, 128, 256, 300, True, "bf16")
    sd = syn.make_weights(shape, seed=41, bias_std=0.05, random_gamma=True)
    cfg, w = oracle_model(shape, sd)
    flat = make_gpu_model(shape, sd, B)
    paged = make_gpu_model(shape, sd, B, page_size=64, n_pages=B * 4)
    prompt = syn.make_tokens(B, 70, 300, seed=3)
    pd = torch.from_numpy(prompt).cuda()
    assert torch.equal(flat.prefill(pd), paged.prefill(pd))
    seqs = prompt.copy()
    for step in range(70):  # crosses the page boundary at position 128
        tok = syn.make_tokens(B, 1, 300, seed=300 + step)[:, 0].copy()
        seqs = np.concatenate([seqs, tok[:, None]], axis=1)
        a = flat.decode_step(torch.from_numpy(tok).cuda())
        assert torch.equal(a, paged.decode_step(torch.from_numpy(tok).cuda())), step
    got = a.cpu().numpy()
    for r in (0, B // 2 - 1, B // 2, B - 1):  # first and last rows of each chain
        ref = og.forward(cfg, w, seqs[r:r + 1])[0][0]
        assert np.max(np.abs(got[r] - ref)) < BF16_TOL, r
    p40 = pd[:, :40].contiguous()
    assert torch.equal(flat.generate(p40, 100, temperature=0.8, top_k=30, seed=5),
                       paged.generate(p40, 100, temperature=0.8, top_k=30, seed=5))
    lens = [1 + (7 * b) % 70 for b in range(B)]
    assert torch.equal(flat.prefill_ragged(pd, lens), paged.prefill_ragged(pd, lens))
    for step in range(5):
        tok = torch.from_numpy(syn.make_tokens(B, 1, 300, seed=400 + step)[:, 0].copy()).cuda()
        assert torch.equal(flat.decode_step(tok), paged.decode_step(tok))
    assert flat.sync_status() == G.GPT_OK and paged.sync_status() == G.GPT_OK


def test_paged_cache_reports_an_exhausted_pool():
    shape = syn.ModelShape(1, 2, 128, 256, 100, False, "bf16")
    sd = syn.make_weights(shape, seed=4)
    model = make_gpu_model(shape, sd, 3, page_size=64, n_pages=3)
    prompt = torch.from_numpy(syn.make_tokens(3, 70, 100, seed=1)).cuda()
    with pytest.raises(G.GptError) as ex:
        model.prefill(prompt)  # 3 sequences x 2 pages > 3 pages
    assert ex.value.code == G.GPT_ENOMEM
    model.prefill(prompt[:1].contiguous())  # 2 pages, and the failed call left nothing behind
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(128 - 70):
        model.decode_step(tok)  # the third page at position 128
    assert model.cache_length == 128
    model.decode_step(tok)
    with pytest.raises(G.GptError) as ex:
        model.extend(torch.zeros(1, 64, dtype=torch.int32, device="cuda"))  # a fourth page
    assert ex.value.code == G.GPT_ENOMEM
    assert model.sync_status() == G.GPT_OK


def test_model_from_an_hf_layout_checkpoint():
    """A checkpoint in the HF GPT-2 layout (Conv1D weights, mask buffers, tied lm_head, zero
    biases of a bias=False model), converted on the host, gives bit-identical logits to the
    model built from the nanoGPT-named weights."""
    from kv_cached_generation_gpt_b300 import checkpoint as ck

    shape = syn.ModelShape(2, 2, 128, 64, 300, False, "bf16")
    sd = syn.make_weights(shape, seed=51, random_gamma=True)
    config, conv = ck.from_hf_state_dict(ck.to_hf_state_dict(sd, shape.n_layer), n_head=shape.n_head,
                                         drop_zero_bias=True)
    assert config["bias"] is False and config["vocab_size"] == 300
    prompt = torch.from_numpy(syn.make_tokens(2, 20, 300, seed=52)).cuda()
    a = make_gpu_model(shape, sd, 2)
    b = make_gpu_model(shape, conv, 2)
    assert torch.equal(a.prefill(prompt), b.prefill(prompt))
    tok = prompt[:, 0].contiguous()
    assert torch.equal(a.decode_step(tok), b.decode_step(tok))
    assert a.sync_status() == G.GPT_OK and b.sync_status() == G.GPT_OK
