// Token + position embedding, and LayerNorm (warp per row, one read of the row).
//
// Embedding ("第 4 章 模型构建", aiknowledge.cn, §4.5): x = wte[id] + wpe[pos], learned
// absolute positions; a new token appended to a cache of length c sits at position c.
// LayerNorm ("原生 nanoGPT 模型服务首选", §1): F.layer_norm with eps 1e-5, biased
// variance, gamma, and an optional beta (bias=False passes no beta).
#pragma once

#include "common.cuh"

namespace kvgpt {

constexpr int LN_MAX_PAIRS = 32;  // up to C = 2048 (C/64 float pairs per lane)

// rows = B*T; row r = b*T + t embeds tokens[b * tok_ld + t] at position pos0 + t (pos_rows[b] + t
// when pos_rows is given) into x[r, :] (fp32).  With lens, positions t >= lens[b] are padding:
// zero rows, no check.  A token outside [0, V) or a position >= block sets the error word and
// writes zeros.
template <typename TW>
__global__ void embed_kernel(const int* __restrict__ tokens, int tok_ld, const int* pos_rows, const int* lens,
                             int rows, int T, const int* pos0,
                             const TW* __restrict__ wte, const TW* __restrict__ wpe, int V, int block, int C,
                             float* __restrict__ x, int* err) {
  griddep_wait();
  griddep_launch();
  const int r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int t = r % T, b = r / T;
  float* xr = x + static_cast<size_t>(r) * C;
  if (lens && t >= lens[b]) {
    for (int c = lane; c < C; c += 32) xr[c] = 0.0f;
    return;
  }
  const int tok = tokens[static_cast<size_t>(b) * tok_ld + t];
  const int pos = (pos_rows ? pos_rows[b] : (pos0 ? *pos0 : 0)) + t;
  const bool bad_tok = tok < 0 || tok >= V;
  const bool bad_pos = pos >= block;
  if (bad_tok || bad_pos) {
    if (lane == 0) atomicOr(err, bad_tok ? ERR_TOKEN : ERR_POSITION);
    for (int c = lane; c < C; c += 32) xr[c] = 0.0f;
    return;
  }
  const TW* we = wte + static_cast<size_t>(tok) * C;
  const TW* pe = wpe + static_cast<size_t>(pos) * C;
  for (int c = lane * 2; c < C; c += 64) {
    float2 o;
    o.x = to_f32(we[c]) + to_f32(pe[c]);
    o.y = to_f32(we[c + 1]) + to_f32(pe[c + 1]);
    *reinterpret_cast<float2*>(xr + c) = o;
  }
}

__device__ __forceinline__ void store_pair(float* p, float a, float b) { *reinterpret_cast<float2*>(p) = make_float2(a, b); }
__device__ __forceinline__ void store_pair(__nv_bfloat16* p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}

// y[r, :] = LN(x[r * in_stride + :]) for r < rows; warp per row.  TO is bf16 or f32.
// With y_lo, also writes the rounding remainder y - bf16(y) (the lo half of a hi/lo pair).
// MAXP bounds C / 64 (the float pairs a lane holds), so small models keep few registers.
// EARLY (programmatic dependent launches of a decode step, a few rows): gamma and beta, which
// do not depend on earlier kernels, are fetched into registers before waiting for them; the
// many-row prefill form loads them at use and keeps its registers (and occupancy).
template <typename TO, int MAXP = LN_MAX_PAIRS, bool EARLY = false>
__global__ void layernorm_kernel(const float* __restrict__ x, int rows, int C, long long in_stride,
                                 const float* __restrict__ gamma, const float* __restrict__ beta,
                                 TO* __restrict__ y, TO* __restrict__ y_lo, int ldy) {
  const int lane = threadIdx.x & 31;
  const int np = C / 64;
  float2 g2[MAXP], b2[MAXP];
#pragma unroll
  for (int i = 0; i < MAXP; ++i) {
    if (EARLY && i < np) {
      const int c = i * 64 + lane * 2;
      g2[i] = *reinterpret_cast<const float2*>(gamma + c);
      b2[i] = beta ? *reinterpret_cast<const float2*>(beta + c) : make_float2(0.0f, 0.0f);
    }
  }
  griddep_wait();  // x comes from the previous kernel (a programmatic dependent launch may start early)
  griddep_launch();
  const int r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (r >= rows) return;
  const float* xr = x + static_cast<size_t>(r) * in_stride;
  float2 v[MAXP];
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < MAXP; ++i) {
    if (i < np) {
      v[i] = *reinterpret_cast<const float2*>(xr + i * 64 + lane * 2);
      s += v[i].x + v[i].y;
    }
  }
  const float mean = warp_sum(s) / static_cast<float>(C);
  float q = 0.0f;
#pragma unroll
  for (int i = 0; i < MAXP; ++i) {
    if (i < np) {
      const float a = v[i].x - mean, b = v[i].y - mean;
      q += a * a + b * b;
    }
  }
  const float var = warp_sum(q) / static_cast<float>(C);
  const float rstd = 1.0f / sqrtf(var + 1e-5f);
  TO* yr = y + static_cast<size_t>(r) * ldy;
#pragma unroll
  for (int i = 0; i < MAXP; ++i) {
    if (i < np) {
      const int c = i * 64 + lane * 2;
      if (!EARLY) {
        g2[i] = *reinterpret_cast<const float2*>(gamma + c);
        if (beta) b2[i] = *reinterpret_cast<const float2*>(beta + c);
      }
      float a = (v[i].x - mean) * rstd * g2[i].x;
      float b = (v[i].y - mean) * rstd * g2[i].y;
      if (beta) {
        a += b2[i].x;
        b += b2[i].y;
      }
      store_pair(yr + c, a, b);
      if (y_lo) {
        const float ha = to_f32(from_f32<TO>(a)), hb = to_f32(from_f32<TO>(b));
        store_pair(y_lo + static_cast<size_t>(r) * ldy + c, a - ha, b - hb);
      }
    }
  }
}

// Widen a weight vector to fp32 (LayerNorm parameters and biases are kept in fp32).
template <typename TW>
__global__ void widen_kernel(const TW* __restrict__ src, float* __restrict__ dst, long long n) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    dst[i] = to_f32(src[i]);
}

}  // namespace kvgpt
