"""Sampler oracle: temperature, top-k, softmax and a counter-based categorical draw.

TEST INFRASTRUCTURE: imported only by tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py.  Nothing here is shared with the CUDA path; the
CUDA sampler implements the same specification independently.

What the pages define ("原生 nanoGPT 模型服务首选", lzwjava.github.io, §2 generate();
"极速上手nanoGPT", deepseek.csdn.net, §"关键参数" temperature / top_k):
  1. divide the last-position logits by the temperature;
  2. with top_k, find v = the min(top_k, V) largest values and set every logit
     strictly below the smallest of them to -inf (ties with it survive);
  3. softmax;
  4. draw one index from the resulting categorical (torch.multinomial).

Step 4 uses torch's private random stream, which no other implementation can
reproduce.  This oracle (and the library) replace it with an exactly specified
draw so that two implementations can agree bit for bit:

  s_i  = fp32(l_i / T)                                 (IEEE fp32 division)
  tau  = the k'-th largest s (duplicates counted), k' = min(top_k, V); S = {i: s_i >= tau}
  m    = max_i s_i
  e_i  = gexp(fp32(s_i - m)) for i in S, else 0        (gexp below)
  w_i  = floor(e_i * 2^40) as an unsigned 64-bit integer
  W    = sum_i w_i                                     (exact: W < 2^57)
  r    = word 0 of Philox4x64-10(counter=(step, 0, 0, 0), key=(seed, row))
  t    = floor(r * W / 2^64)                           (exact 128-bit product)
  pick = the smallest i with w_0 + ... + w_i > t

The pick has probability w_i / W (up to the 2^-64 granularity of r), i.e. the
softmax of step 3 with each probability truncated to 40 fractional bits of the
largest term.  Temperature 0 is read as greedy argmax (lowest index on ties).

Philox4x64-10 is the counter-based generator of Salmon, Moraes, Dror and Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): ten rounds of two 64x64
-> 128-bit multiplies with the paper's multipliers, the key bumped by its two
Weyl constants between rounds.

gexp(x), x <= 0, is an fp32 exponential built only from IEEE-rounded fp32
multiplies and adds (never fused), so that any two implementations of the same
operation sequence agree bit for bit:
  n = rint(x * LOG2E);  r = (x - n*LN2_HI) - n*LN2_LO        (Cody-Waite reduction)
  p = Horner evaluation of sum_{k=0..7} r^k / k!             (Taylor series of e^r)
  gexp(x) = p * 2^n;   gexp(x) = 0 for x < -64
LN2_HI is ln 2 rounded to fp32 with its 8 low significand bits cleared (so n*LN2_HI
is exact for |n| <= 128) and LN2_LO = fp32(ln 2 - LN2_HI).
"""
from __future__ import annotations

import math

import numpy as np

MASK64 = (1 << 64) - 1

# Salmon et al., SC'11, Philox4x64: round multipliers and key-schedule (Weyl) constants.
PHILOX_M0 = 0xD2E7470EE14C6C93
PHILOX_M1 = 0xCA5A826395121157
PHILOX_W0 = 0x9E3779B97F4A7C15  # golden ratio
PHILOX_W1 = 0xBB67AE8584CAA73B  # sqrt(3) - 1
PHILOX_ROUNDS = 10


def philox4x64_10(counter, key) -> list[int]:
    """Philox4x64 with 10 rounds; counter: 4 uint64, key: 2 uint64 -> 4 uint64."""
    c = [int(x) & MASK64 for x in counter]
    k = [int(x) & MASK64 for x in key]
    for rnd in range(PHILOX_ROUNDS):
        if rnd > 0:
            k = [(k[0] + PHILOX_W0) & MASK64, (k[1] + PHILOX_W1) & MASK64]
        p0 = PHILOX_M0 * c[0]
        p1 = PHILOX_M1 * c[2]
        hi0, lo0 = p0 >> 64, p0 & MASK64
        hi1, lo1 = p1 >> 64, p1 & MASK64
        c = [hi1 ^ c[1] ^ k[0], lo1, hi0 ^ c[3] ^ k[1], lo0]
    return c


def draw_word(seed: int, row: int, step: int) -> int:
    """The 64-bit uniform word used for (row, step) under ``seed``."""
    return philox4x64_10((step, 0, 0, 0), (seed, row))[0]


# ---------------------------------------------------------------- gexp

F32 = np.float32
LOG2E = F32(1.0 / math.log(2.0))
_ln2_f32_bits = int(np.array([math.log(2.0)], dtype=np.float32).view(np.uint32)[0])
LN2_HI = np.array([_ln2_f32_bits & ~0xFF], dtype=np.uint32).view(np.float32)[0]
LN2_LO = F32(math.log(2.0) - float(LN2_HI))
TAYLOR = [F32(1.0 / math.factorial(k)) for k in range(8)]  # 1/k!, k = 0..7
GEXP_CUTOFF = F32(-64.0)
WEIGHT_BITS = 40


def gexp(x) -> np.ndarray:
    """fp32 e^x for x <= 0 by the fixed operation sequence in the module docstring."""
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        xs = np.where(x >= GEXP_CUTOFF, x, F32(0.0)).astype(np.float32)
        n = np.rint(xs * LOG2E).astype(np.float32)
        r = (xs - n * LN2_HI) - n * LN2_LO
        p = TAYLOR[7]
        for k in range(6, -1, -1):
            p = p * r + TAYLOR[k]
        scale = ((n.astype(np.int32) + 127) << 23).astype(np.int32).view(np.float32)
        e = (p * scale).astype(np.float32)
    return np.where(x >= GEXP_CUTOFF, e, F32(0.0)).astype(np.float32)


# ---------------------------------------------------------------- sampler


def scaled_logits(logits: np.ndarray, temperature: float) -> np.ndarray:
    """s = fp32(l / T)."""
    return (np.asarray(logits, dtype=np.float32) / F32(temperature)).astype(np.float32)


def topk_threshold(s: np.ndarray, top_k: int | None) -> np.float32:
    """The k'-th largest value of the row s (duplicates counted), k' = min(top_k, V).

    No top-k (None or <= 0) returns -inf, which every value passes."""
    V = s.shape[-1]
    if top_k is None or top_k <= 0:
        return F32(-np.inf)
    k = min(int(top_k), V)
    return np.sort(s)[::-1][k - 1]


def survivors(s: np.ndarray, top_k: int | None) -> np.ndarray:
    """Boolean mask of the values that top-k keeps: s >= tau."""
    return s >= topk_threshold(s, top_k)


def integer_weights(s: np.ndarray, keep: np.ndarray) -> np.ndarray:
    """w_i = floor(gexp(s_i - max s) * 2^40) for kept i, else 0 (uint64)."""
    m = s.max()
    e = gexp((s - m).astype(np.float32))
    e = np.where(keep, e, F32(0.0)).astype(np.float32)
    return (e * F32(2.0 ** WEIGHT_BITS)).astype(np.float32).astype(np.uint64)


def pick(w: np.ndarray, r: int) -> int:
    """Smallest i with w_0 + ... + w_i > floor(r * W / 2^64)."""
    total = int(w.sum(dtype=np.uint64))
    target = (int(r) * total) >> 64
    cum = np.cumsum(w, dtype=np.uint64)
    return int(np.searchsorted(cum, np.uint64(target), side="right"))


def sample_row(logits_row: np.ndarray, temperature: float, top_k: int | None, seed: int, row: int,
               step: int) -> int:
    if temperature == 0.0:
        return int(np.argmax(np.asarray(logits_row, dtype=np.float32)))
    s = scaled_logits(logits_row, temperature)
    keep = survivors(s, top_k)
    return pick(integer_weights(s, keep), draw_word(seed, row, step))


def sample(logits: np.ndarray, temperature: float, top_k: int | None, seed: int, step: int) -> np.ndarray:
    """Sample one id per row of fp32 logits (B, V); row b uses Philox key (seed, b)."""
    logits = np.asarray(logits, dtype=np.float32)
    return np.array([sample_row(logits[b], temperature, top_k, seed, b, step) for b in range(logits.shape[0])],
                    dtype=np.int32)
