// Temperature / top-k / softmax / categorical draw, one CTA per row.
//
// What the pages define ("原生 nanoGPT 模型服务首选", lzwjava.github.io, §2 generate();
// "极速上手nanoGPT", deepseek.csdn.net, §"关键参数"): divide the last-position logits by the
// temperature, keep the min(top_k, V) largest (everything equal to the k-th largest
// survives, everything strictly below it is dropped), softmax, draw one index.
//
// The draw is specified exactly so that independent implementations agree bit for bit:
//   s_i = fp32(l_i / T)                          (IEEE division)
//   tau = k'-th largest s_i (duplicates counted)  (radix select on order-preserving keys)
//   w_i = floor(gexp(s_i - max s) * 2^40) for s_i >= tau, else 0     (uint64)
//   t   = floor(r * W / 2^64), W = sum w_i, r = word 0 of Philox4x64-10(counter = (step, 0, 0, 0),
//         key = (seed, row))  (Salmon et al., SC'11, "Parallel Random Numbers: As Easy as 1, 2, 3")
//   pick the smallest i with w_0 + ... + w_i > t.
// gexp(x) (x <= 0): n = rint(x log2 e), r = (x - n LN2_HI) - n LN2_LO (Cody-Waite), the Taylor
// series of e^r to degree 7 in Horner form, times 2^n; 0 below -64.  Every operation is an
// explicitly rounded fp32 multiply or add (no contraction into FMA), so the sequence is
// reproducible on any IEEE machine.  Temperature 0 means greedy argmax (lowest index on ties).
#pragma once

#include "common.cuh"

namespace kvgpt {

constexpr int SMP_THREADS = 1024;
constexpr int SMP_WARPS = SMP_THREADS / 32;

// Philox4x64 round multipliers and Weyl key increments (Salmon et al., SC'11).
constexpr unsigned long long PHILOX_M0 = 0xD2E7470EE14C6C93ull;
constexpr unsigned long long PHILOX_M1 = 0xCA5A826395121157ull;
constexpr unsigned long long PHILOX_W0 = 0x9E3779B97F4A7C15ull;
constexpr unsigned long long PHILOX_W1 = 0xBB67AE8584CAA73Bull;

__device__ __forceinline__ unsigned long long philox_word0(unsigned long long seed, unsigned long long row,
                                                           unsigned long long step) {
  unsigned long long c0 = step, c1 = 0, c2 = 0, c3 = 0, k0 = seed, k1 = row;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    const unsigned long long lo0 = PHILOX_M0 * c0, hi0 = __umul64hi(PHILOX_M0, c0);
    const unsigned long long lo1 = PHILOX_M1 * c2, hi1 = __umul64hi(PHILOX_M1, c2);
    const unsigned long long n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return c0;
}

// fp32 e^x for x <= 0 by the fixed sequence above.  Constants are the fp32 roundings of
// 1/ln 2, ln 2 with its 8 low significand bits cleared, the remainder, and 1/k!.
__device__ __forceinline__ float gexp(float x) {
  if (!(x >= -64.0f)) return 0.0f;
  const float kLog2e = __uint_as_float(0x3fb8aa3bu);
  const float kLn2Hi = __uint_as_float(0x3f317200u);
  const float kLn2Lo = __uint_as_float(0x35bfbe8eu);
  const float n = rintf(__fmul_rn(x, kLog2e));
  const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(n, kLn2Hi)), __fmul_rn(n, kLn2Lo));
  float p = __uint_as_float(0x39500d01u);                  // 1/7!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3ab60b61u));  // 1/6!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3c088889u));  // 1/5!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3d2aaaabu));  // 1/4!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3e2aaaabu));  // 1/3!
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  return __fmul_rn(p, __int_as_float((static_cast<int>(n) + 127) << 23));
}

__device__ __forceinline__ unsigned long long weight40(float s, float m) {
  return __float2ull_rz(__fmul_rn(gexp(__fsub_rn(s, m)), 1099511627776.0f /* 2^40 */));
}

// Order-preserving map of fp32 to uint32 (ascending floats -> ascending keys) and back.
__device__ __forceinline__ unsigned int fkey(float f) {
  const unsigned int u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(unsigned int k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

struct SampleArgs {
  const float* logits;     // [B][ld]
  int ld, V;
  float temperature;       // 0: greedy
  int top_k;               // <= 0: no top-k
  unsigned long long seed;
  const int* step_dev;     // step index from device memory (nullable)
  int step;                // used when step_dev is null
  int* out;                // nullable: out[b * out_stride + out_col0 + step] = token
  int out_stride, out_col0;
  int* next_tokens;        // nullable: next_tokens[b] = token
  float* thr_out;          // nullable: the threshold tau per row (-inf: no top-k)
  unsigned long long* w_out;  // nullable: the integer weights [B][V]
};

__global__ void __launch_bounds__(SMP_THREADS) sample_kernel(SampleArgs a) {
  extern __shared__ float s_s[];  // V scaled logits
  __shared__ unsigned int s_hist[256];
  __shared__ float s_rf[SMP_WARPS];
  __shared__ int s_ri[SMP_WARPS];
  __shared__ unsigned long long s_ru[SMP_WARPS];
  __shared__ unsigned int s_prefix, s_remaining;
  __shared__ unsigned long long s_target;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* lr = a.logits + static_cast<size_t>(b) * a.ld;
  const int V = a.V;
  const int step = a.step_dev ? *a.step_dev : a.step;

  auto emit = [&](int tok, float thr) {
    if (a.out) a.out[static_cast<size_t>(b) * a.out_stride + a.out_col0 + step] = tok;
    if (a.next_tokens) a.next_tokens[b] = tok;
    if (a.thr_out) a.thr_out[b] = thr;
  };

  if (a.temperature == 0.0f) {
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = tid; i < V; i += SMP_THREADS) {
      const float v = lr[i];
      if (v > best || (v == best && i < bi)) {
        best = v;
        bi = i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, best, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (v2 > best || (v2 == best && i2 < bi)) {
        best = v2;
        bi = i2;
      }
    }
    if (lane == 0) {
      s_rf[warp] = best;
      s_ri[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < SMP_WARPS; ++w)
        if (s_rf[w] > best || (s_rf[w] == best && s_ri[w] < bi)) {
          best = s_rf[w];
          bi = s_ri[w];
        }
      emit(bi == 0x7fffffff ? 0 : bi, -INFINITY);
    }
    return;
  }

  // 1. s = l / T, its maximum and minimum
  float mx = -INFINITY, mn = INFINITY;
  for (int i = tid; i < V; i += SMP_THREADS) {
    const float s = __fdiv_rn(lr[i], a.temperature);
    s_s[i] = s;
    mx = fmaxf(mx, s);
    mn = fminf(mn, s);
  }
  mx = warp_max(mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  if (lane == 0) {
    s_rf[warp] = mx;
    s_ri[warp] = __float_as_int(mn);
  }
  __syncthreads();
  float m = s_rf[0], vmin = __int_as_float(s_ri[0]);
#pragma unroll 1
  for (int w = 1; w < SMP_WARPS; ++w) {
    m = fmaxf(m, s_rf[w]);
    vmin = fminf(vmin, __int_as_float(s_ri[w]));
  }

  // 2. tau = the k'-th largest s, k' = min(top_k, V): the minimum when top_k >= V, else a
  //    radix select, 8 bits at a time from the top
  float tau = (a.top_k > 0) ? vmin : -INFINITY;
  if (a.top_k > 0 && a.top_k < V) {
    if (tid == 0) {
      s_prefix = 0u;
      s_remaining = static_cast<unsigned int>(a.top_k);
    }
    unsigned int pmask = 0u;
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) s_hist[tid] = 0u;
      __syncthreads();
      const unsigned int prefix = s_prefix;
      for (int i = tid; i < V; i += SMP_THREADS) {
        const unsigned int k = fkey(s_s[i]);
        const bool cand = (k & pmask) == prefix;
        const unsigned int dig = (k >> shift) & 255u;
        // aggregate equal digits within the warp: one shared-memory atomic per distinct digit
        const unsigned int act = __ballot_sync(__activemask(), cand);
        if (cand) {
          const unsigned int peers = __match_any_sync(act, dig);
          if ((__ffs(peers) - 1) == lane) atomicAdd(&s_hist[dig], static_cast<unsigned int>(__popc(peers)));
        }
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 255-8l .. 248-8l (descending); find the bin holding the remaining-th
        unsigned int c[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = s_hist[255 - 8 * lane - j];
          tot += c[j];
        }
        unsigned int incl = tot;  // inclusive prefix over lanes 0..lane (descending bins)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const unsigned int rem = s_remaining;
        const unsigned int excl = incl - tot;
        if (excl < rem && rem <= incl) {
          unsigned int run = excl;
          for (int j = 0; j < 8; ++j) {
            if (run + c[j] >= rem) {
              const unsigned int dig = 255u - 8u * lane - j;
              s_remaining = rem - run;
              s_prefix = prefix | (dig << shift);
              break;
            }
            run += c[j];
          }
        }
      }
      pmask |= 255u << shift;
      __syncthreads();
    }
    tau = fkey_inv(s_prefix);
  }

  // 3. integer weights over a contiguous chunk per thread, and the block's exclusive scan
  const int chunk = (V + SMP_THREADS - 1) / SMP_THREADS;
  const int i0 = tid * chunk, i1 = min(V, i0 + chunk);
  unsigned long long local = 0;
  for (int i = i0; i < i1; ++i) {
    const float s = s_s[i];
    const unsigned long long w = (s >= tau) ? weight40(s, m) : 0ull;
    if (a.w_out) a.w_out[static_cast<size_t>(b) * V + i] = w;
    local += w;
  }
  unsigned long long incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_ru[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    unsigned long long wt = s_ru[lane];
    unsigned long long wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    s_ru[lane] = wi - wt;  // exclusive offset of each warp
    if (lane == 31) {
      const unsigned long long W = wi;
      const unsigned long long r = philox_word0(a.seed, static_cast<unsigned long long>(b),
                                                static_cast<unsigned long long>(step));
      s_target = __umul64hi(r, W);
    }
  }
  __syncthreads();
  const unsigned long long excl = s_ru[warp] + incl - local;
  const unsigned long long target = s_target;
  // 4. the thread whose range holds the target walks its chunk
  if (local > 0 && excl <= target && target < excl + local) {
    unsigned long long run = excl;
    for (int i = i0; i < i1; ++i) {
      const float s = s_s[i];
      run += (s >= tau) ? weight40(s, m) : 0ull;
      if (run > target) {
        emit(i, tau);
        break;
      }
    }
  }
}

}  // namespace kvgpt
