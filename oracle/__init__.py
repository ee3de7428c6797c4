"""CPU oracle for KV-cached GPT-2 generation (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(``cpu_baseline`` and ``--impl reference``) import this package.  The library's
product path (``kv_cached_generation_gpt_b300`` and its CUDA code) never does,
and this package imports nothing from it.

* ``oracle.gpt``     -- the decoder forward pass, no-cache and KV-cached, in fp64.
* ``oracle.sampler`` -- temperature / top-k / softmax / inverse-CDF sampling, with
  the Philox4x64-10 counter-based generator, in the exact integer arithmetic
  both sides follow.
"""
