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
  int cand_cap;            // candidate slots after the V scaled logits in dynamic shared memory
};

struct SampleSmem {
  unsigned int hist[256];
  float rf[SMP_WARPS];
  int ri[SMP_WARPS];
  unsigned long long ru[SMP_WARPS];
  unsigned int prefix, remaining;
  unsigned long long target;
  int flag;
};

// Block-wide: the k-th largest (1-based, duplicates counted) of n order-preserving keys
// key_at(0..n-1), by a radix select 8 bits at a time from the top.
template <typename KeyAt>
__device__ unsigned int block_select_desc(KeyAt key_at, int n, unsigned int k, SampleSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __syncthreads();
  if (tid == 0) {
    sm.prefix = 0u;
    sm.remaining = k;
  }
  unsigned int pmask = 0u;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) sm.hist[tid] = 0u;
    __syncthreads();
    const unsigned int prefix = sm.prefix;
    for (int i = tid; i < n; i += SMP_THREADS) {
      const unsigned int key = key_at(i);
      const bool cand = (key & pmask) == prefix;
      const unsigned int dig = (key >> shift) & 255u;
      // aggregate equal digits within the warp: one shared-memory atomic per distinct digit
      const unsigned int act = __ballot_sync(__activemask(), cand);
      if (cand) {
        const unsigned int peers = __match_any_sync(act, dig);
        if ((__ffs(peers) - 1) == lane) atomicAdd(&sm.hist[dig], static_cast<unsigned int>(__popc(peers)));
      }
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l .. 248-8l (descending); find the bin holding the remaining-th
      unsigned int c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sm.hist[255 - 8 * lane - j];
        tot += c[j];
      }
      unsigned int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned int rem = sm.remaining;
      const unsigned int excl = incl - tot;
      if (excl < rem && rem <= incl) {
        unsigned int run = excl;
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= rem) {
            const unsigned int dig = 255u - 8u * lane - j;
            sm.remaining = rem - run;
            sm.prefix = prefix | (dig << shift);
            break;
          }
          run += c[j];
        }
      }
    }
    pmask |= 255u << shift;
    __syncthreads();
  }
  return sm.prefix;
}

// Block-wide exclusive prefix sum of one uint64 per thread (in thread order); returns the
// exclusive prefix, and the total in *total.
__device__ __forceinline__ unsigned long long block_scan_u64(unsigned long long v, unsigned long long* total,
                                                             SampleSmem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();
  if (lane == 31) sm.ru[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long wt = sm.ru[lane];
    unsigned long long wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    sm.ru[lane] = wi - wt;
    if (lane == 31) sm.target = wi;  // total, read below before the caller reuses `target`
  }
  __syncthreads();
  *total = sm.target;
  return sm.ru[warp] + incl - v;
}

// The draw over items j = 0..n-1 in ascending token order, item j being token idx(j) with
// scaled logit val(j): integer weights of the survivors (val >= tau), their total W, the
// target floor(r W / 2^64), and the first item whose running sum exceeds it.  Each thread
// takes a contiguous run of items so the block scan follows the item order.
template <typename IdxAt, typename ValAt, typename Emit>
__device__ void draw_over(int n, IdxAt idx_at, ValAt val_at, float tau, float m, unsigned long long seed, int row,
                          int step, Emit emit, SampleSmem& sm) {
  const int tid = threadIdx.x;
  const int chunk = (n + SMP_THREADS - 1) / SMP_THREADS;
  const int j0 = min(n, tid * chunk), j1 = min(n, j0 + chunk);
  unsigned long long local = 0;
  for (int j = j0; j < j1; ++j) {
    const float s = val_at(j);
    local += (s >= tau) ? weight40(s, m) : 0ull;
  }
  unsigned long long W = 0;
  const unsigned long long excl = block_scan_u64(local, &W, sm);
  const unsigned long long r =
      philox_word0(seed, static_cast<unsigned long long>(row), static_cast<unsigned long long>(step));
  const unsigned long long target = __umul64hi(r, W);
  if (local > 0 && excl <= target && target < excl + local) {
    unsigned long long run = excl;
    for (int j = j0; j < j1; ++j) {
      const float s = val_at(j);
      run += (s >= tau) ? weight40(s, m) : 0ull;
      if (run > target) {
        emit(idx_at(j), tau);
        break;
      }
    }
  }
}

// One CTA per row.  Dynamic shared memory: V scaled logits, then cand_cap int slots.
//
// The threshold tau (the k'-th largest s) is found without sorting the row: the maxima of
// 1024 disjoint groups give k' distinct elements >= L, their k'-th largest, so L <= tau and
// every survivor is a candidate with s >= L.  The candidates (usually a little over k') are
// compacted in ascending index order, tau is selected among them, and the draw runs over
// them: non-candidates have s < L <= tau and weight 0, so W and the pick are unchanged.
// When there are more candidates than slots (heavily tied rows) or k' > 1024, tau is
// selected over the whole row instead.
__global__ void __launch_bounds__(SMP_THREADS) sample_kernel(SampleArgs a) {
  extern __shared__ __align__(16) float s_s[];  // V scaled logits, then the candidate slots
  __shared__ SampleSmem sm;
  int* s_cand = reinterpret_cast<int*>(s_s + a.V);
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_wait();  // the logits come from the previous kernel
  griddep_launch();
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
      sm.rf[warp] = best;
      sm.ri[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < SMP_WARPS; ++w)
        if (sm.rf[w] > best || (sm.rf[w] == best && sm.ri[w] < bi)) {
          best = sm.rf[w];
          bi = sm.ri[w];
        }
      emit(bi == 0x7fffffff ? 0 : bi, -INFINITY);
    }
    return;
  }

  // 1. s = l / T; the row's maximum and minimum, and the maximum of group tid = {i : i % 1024 == tid}
  //    (16 loads in flight per thread; l / 1 == l exactly, so T = 1 skips the division)
  float mx = -INFINITY, mn = INFINITY;
  const bool unit_t = a.temperature == 1.0f;
  constexpr int BATCH = 16;
#pragma unroll 1
  for (int i0 = tid; i0 < V; i0 += BATCH * SMP_THREADS) {
    float l[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int i = i0 + u * SMP_THREADS;
      l[u] = i < V ? __ldg(lr + i) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int i = i0 + u * SMP_THREADS;
      if (i < V) {
        const float s = unit_t ? l[u] : __fdiv_rn(l[u], a.temperature);
        s_s[i] = s;
        mx = fmaxf(mx, s);
        mn = fminf(mn, s);
      }
    }
  }
  const float gmax = mx;
  mx = warp_max(mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  if (lane == 0) {
    sm.rf[warp] = mx;
    sm.ri[warp] = __float_as_int(mn);
  }
  __syncthreads();
  float m = sm.rf[0], vmin = __int_as_float(sm.ri[0]);
#pragma unroll 1
  for (int w = 1; w < SMP_WARPS; ++w) {
    m = fmaxf(m, sm.rf[w]);
    vmin = fminf(vmin, __int_as_float(sm.ri[w]));
  }

  auto val_row = [&](int i) { return s_s[i]; };
  auto idx_row = [&](int i) { return i; };
  const unsigned int kk = (a.top_k > 0) ? static_cast<unsigned int>(min(a.top_k, V)) : static_cast<unsigned int>(V);
  float tau = -INFINITY;
  if (a.top_k > 0 && kk >= static_cast<unsigned int>(V)) tau = vmin;  // k' = V keeps every entry
  bool done = false;
  if (a.top_k > 0 && kk < static_cast<unsigned int>(V)) {
    bool fast = kk <= static_cast<unsigned int>(SMP_THREADS) && a.cand_cap >= SMP_THREADS;
    if (fast) {
      // 2. L = the k'-th largest group maximum (groups past the row's end hold -inf)
      s_cand[tid] = static_cast<int>(fkey(gmax));
      const float L = fkey_inv(block_select_desc(
          [&](int i) { return static_cast<unsigned int>(s_cand[i]); }, SMP_THREADS, kk, sm));
      // 3. candidates {i : s_i >= L}, compacted in ascending index order; thread t scans a
      //    contiguous run whose length is a multiple of 4 (16-byte shared-memory loads)
      const int chunk = ((V + SMP_THREADS - 1) / SMP_THREADS + 3) & ~3;
      const int i0 = min(V, tid * chunk), i1 = min(V, i0 + chunk);
      unsigned int cnt = 0;
      for (int i = i0; i < i1; i += 4) {
        if (i + 4 <= i1) {
          const float4 v = *reinterpret_cast<const float4*>(s_s + i);
          cnt += (v.x >= L) + (v.y >= L) + (v.z >= L) + (v.w >= L);
        } else {
          for (int j = i; j < i1; ++j) cnt += s_s[j] >= L;
        }
      }
      unsigned long long total = 0;
      const unsigned long long off = block_scan_u64(cnt, &total, sm);
      if (total <= static_cast<unsigned long long>(a.cand_cap)) {
        int o = static_cast<int>(off);
        for (int i = i0; i < i1; i += 4) {
          if (i + 4 <= i1) {
            const float4 v = *reinterpret_cast<const float4*>(s_s + i);
            if (v.x >= L) s_cand[o++] = i;
            if (v.y >= L) s_cand[o++] = i + 1;
            if (v.z >= L) s_cand[o++] = i + 2;
            if (v.w >= L) s_cand[o++] = i + 3;
          } else {
            for (int j = i; j < i1; ++j)
              if (s_s[j] >= L) s_cand[o++] = j;
          }
        }
        __syncthreads();
        const int n = static_cast<int>(total);
        auto val_c = [&](int j) { return s_s[s_cand[j]]; };
        auto idx_c = [&](int j) { return s_cand[j]; };
        // 4. tau among the candidates, then the draw over them
        tau = fkey_inv(block_select_desc([&](int j) { return fkey(val_c(j)); }, n, kk, sm));
        draw_over(n, idx_c, val_c, tau, m, a.seed, b, step, emit, sm);
        done = true;
      }
    }
    if (!done) tau = fkey_inv(block_select_desc([&](int i) { return fkey(s_s[i]); }, V, kk, sm));
  }
  if (!done) draw_over(V, idx_row, val_row, tau, m, a.seed, b, step, emit, sm);
  if (a.w_out) {
    for (int i = tid; i < V; i += SMP_THREADS) {
      const float s = s_s[i];
      a.w_out[static_cast<size_t>(b) * V + i] = (s >= tau) ? weight40(s, m) : 0ull;
    }
  }
}

}  // namespace kvgpt
