"""Run gpt_generate on a named workload, the last call inside an NVTX range (for ncu).

    python -m kv_cached_generation_gpt_b300.profile_generate [--workload gpt2_124m_b64_p512_d512]
        [--decode N] [--warmup W]

`--decode` caps the decode steps (default: the workload's).  ncu can restrict itself to the
range with `--nvtx --nvtx-include "profiled/"`.
"""
from __future__ import annotations

import argparse

import torch

from kv_cached_generation_gpt_b300 import gpt as G
from kv_cached_generation_gpt_b300 import synthetic as syn


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="gpt2_124m_b64_p512_d512", choices=sorted(syn.WORKLOADS))
    ap.add_argument("--decode", type=int, default=-1)
    ap.add_argument("--warmup", type=int, default=1)
    a = ap.parse_args()
    wl = syn.WORKLOADS[a.workload]
    shape = wl.model
    dt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    dev = torch.device("cuda", 0)
    sd = {k: torch.from_numpy(v).to(dt).to(dev) for k, v in syn.make_weights(shape, bias_std=wl.bias_std).items()}
    model = G.GPT(shape.n_layer, shape.n_head, shape.n_embd, shape.block_size, shape.vocab_size, shape.bias, dt,
                  wl.batch, sd)
    steps = wl.decode_steps if a.decode < 0 else min(a.decode, wl.decode_steps)
    prompt = torch.from_numpy(syn.make_tokens(wl.batch, wl.prompt, wl.token_hi)).to(dev)
    out = torch.empty(wl.batch, wl.prompt + steps + 1, dtype=torch.int32, device=dev)
    for _ in range(a.warmup):
        model.generate(prompt, steps + 1, wl.temperature, wl.top_k, 7, out)
    torch.cuda.synchronize()
    l0 = G.gpt_kernel_launches(model.handle)
    torch.cuda.nvtx.range_push("profiled")
    model.generate(prompt, steps + 1, wl.temperature, wl.top_k, 7, out)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    status = model.sync_status()
    if status != G.GPT_OK:
        raise SystemExit(f"device error word: {G.lib().gpt_strerror(status).decode()}")
    print(f"{wl.name}: prefill {wl.prompt} + {steps} decode steps, {G.gpt_kernel_launches(model.handle) - l0} "
          f"kernels in the profiled call")


if __name__ == "__main__":
    main()
