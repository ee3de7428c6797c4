// Causal self-attention over the KV cache (head size 64).
//
// Definition ("极速上手nanoGPT", deepseek.csdn.net, §"注意力机制"; "第 4 章 模型构建",
// aiknowledge.cn, §4.5 causal mask): y = softmax(q k^T / sqrt(hs) + mask) v, where the
// query at absolute position p sees keys 0..p.  With a cache ("原生 nanoGPT 模型服务首选",
// §"一个值得做的改进") the new token's query sees every cached key, itself included.
//
// Layouts: q [B][nh][T][64]; cache [B][nh][block][64] (this layer's K or V); keys of one
// (b, h) are contiguous 128-byte rows for bf16.  Output y [B*T][C], column h*64 + d
// (heads re-concatenated in order for c_proj).
//
//   attn_decode_kernel  -- one new query per (b, h); split-KV over the keys, 8 lanes per key
//                          with 128-bit loads, warp-shuffle reductions, online softmax in
//                          fp32, splits merged by log-sum-exp in a fixed order.
//   attn_prefill_tc     -- (attention_prefill.cuh) FlashAttention-style tiles on tcgen05.
//   attn_prefill_f32    -- exact fp32 path for fp32 models (warp per query).
#pragma once

#include "common.cuh"

namespace kvgpt {

constexpr int HS = 64;
constexpr float LOG2E_F = 1.4426950408889634f;

// ------------------------------------------------------------------ decode

// Warps per CTA of the decode attention: 8 (each lane group 3 keys deep) when the grid is small
// (<= DEC_WIDE_MAX_CTAS CTAs, e.g. one 32-sequence decode chain of GPT-2 124M: 384), so that
// each SM keeps enough loads in flight; 4 (4 keys deep) for larger grids.  Measured on a B300 at
// GPT-2 124M, t = 768: 32 sequences 21.4 -> 18.2 us; the B = 64 decode step 748 -> 718 us.
constexpr int DEC_WIDE_MAX_CTAS = 512;
__host__ __device__ constexpr int dec_unroll(int nw) { return nw >= 8 ? 3 : 4; }


template <typename T>
struct Vec8;  // 8 consecutive head dims of one row
template <>
struct Vec8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { u = __ldg(reinterpret_cast<const uint4*>(p)); }
  // cached rows are read once per step: streaming (evict-first) loads
  __device__ __forceinline__ void load_stream(const __nv_bfloat16* p) { u = __ldcs(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ void to_float(float (&f)[8]) const {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
};
template <>
struct Vec8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ void load_stream(const float* p) {
    a = __ldcs(reinterpret_cast<const float4*>(p));
    b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ void to_float(float (&f)[8]) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
};

// grid (B*nh, splits).  Keys 0..t_len-1 with t_len = *pos0 + 1 (or pos_rows[b] + 1 when
// pos_rows is given: sequences of a ragged batch at their own lengths) are split in chunks of a
// multiple of 16; split s takes [s*chunk, (s+1)*chunk).  ws holds per split (m, l, acc[64])
// when splits > 1.  y_lo (nullable) receives y - bf16(y).
// HSZ = head size (32 or 64): LPK = HSZ/8 lanes per key, each holding 8 dims, so a warp
// covers 32/LPK keys per load instruction.
// PAGED: the cache rows are found through kv's block table (else kv is the contiguous layout).
template <typename T, int HSZ, bool PAGED = false, int DEC_WARPS = 4>
__global__ void __launch_bounds__(32 * DEC_WARPS) attn_decode_kernel(const T* __restrict__ q, const T* __restrict__ kc,
                                                                  const T* __restrict__ vc, KvLayout kv, int nh,
                                                                  int block,
                                                                  const int* pos0, const int* pos_rows,
                                                                  float* __restrict__ ws,
                                                                  unsigned int* __restrict__ tickets,
                                                                  T* __restrict__ y, T* __restrict__ y_lo, int C,
                                                                  int* err) {
  static_assert(HSZ == 32 || HSZ == 64, "head size 32 or 64");
  constexpr int LPK = HSZ / 8;        // lanes per key
  constexpr int KPW = 32 / LPK;       // keys per warp per load
  constexpr int KPI = DEC_WARPS * KPW;  // keys per CTA per unrolled slot
  constexpr int DEC_UNROLL = dec_unroll(DEC_WARPS);  // keys per lane group per iteration
  __shared__ float s_m[DEC_WARPS], s_l[DEC_WARPS];
  __shared__ float s_acc[DEC_WARPS][HSZ];
  __shared__ int s_last;
  const int bh = blockIdx.x, split = blockIdx.y, splits = gridDim.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = lane % LPK, g = lane / LPK;
  griddep_wait();  // q and the new key/value come from the previous kernel
  griddep_launch();
  const int t_len = (pos_rows ? pos_rows[bh / nh] : *pos0) + 1;
  if (t_len > block) {
    if (threadIdx.x == 0) atomicOr(err, ERR_POSITION);
    return;
  }
  const int chunk = ((t_len + splits - 1) / splits + 15) & ~15;
  const int kbeg = split * chunk, kend = min(t_len, kbeg + chunk);

  float qv[8];
  {
    Vec8<T> t;
    t.load(q + static_cast<size_t>(bh) * HSZ + e * 8);
    t.to_float(qv);
    const float sc = (HSZ == 64 ? 0.125f : 0.17677669529663688f) * LOG2E_F;  // 1/sqrt(hs), log2 units
#pragma unroll
    for (int i = 0; i < 8; ++i) qv[i] *= sc;
  }
  const int bq = bh / nh, hq = bh - bq * nh;
  // contiguous cache: the (b, h) rows start here; paged: each key's row through the table
  const size_t row0 = PAGED ? 0 : (static_cast<size_t>(bq) * kv.nh + hq) * kv.block;

  float m = -INFINITY, l = 0.0f, acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;

  // The loop bound is warp-uniform (the shuffles below need all 32 lanes); each lane group
  // checks its own key index.
  for (int jb = kbeg + warp * KPW; jb < kend; jb += KPI * DEC_UNROLL) {
    const int j0 = jb + g;
    Vec8<T> kr[DEC_UNROLL], vv[DEC_UNROLL];
#pragma unroll
    for (int u = 0; u < DEC_UNROLL; ++u) {
      const int j = j0 + KPI * u;
      if (j < kend) {
        const size_t row = (PAGED ? kv.row(bq, hq, j) : row0 + j) * HSZ + e * 8;
        kr[u].load_stream(kc + row);
        vv[u].load_stream(vc + row);
      }
    }
    float s[DEC_UNROLL];
#pragma unroll
    for (int u = 0; u < DEC_UNROLL; ++u) {
      float kf[8];
      kr[u].to_float(kf);
      float d = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) d = fmaf(qv[i], kf[i], d);
#pragma unroll
      for (int o = 1; o < LPK; o <<= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      s[u] = (j0 + KPI * u < kend) ? d : -INFINITY;
    }
    float mn = m;
#pragma unroll
    for (int u = 0; u < DEC_UNROLL; ++u) mn = fmaxf(mn, s[u]);
    const float corr = (mn == -INFINITY) ? 1.0f : exp2f(m - mn);  // m = -inf before the first key gives 0
    l *= corr;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] *= corr;
#pragma unroll
    for (int u = 0; u < DEC_UNROLL; ++u) {
      if (j0 + KPI * u < kend) {
        const float p = exp2f(s[u] - mn);
        l += p;
        float vf[8];
        vv[u].to_float(vf);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vf[i], acc[i]);
      }
    }
    m = mn;
  }

  // merge the lane groups of the warp (lanes e, e+LPK, e+2LPK, ... hold the same dims)
#pragma unroll
  for (int o = LPK; o <= 16; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    const float mn = fmaxf(m, m2);
    const float c1 = (m == -INFINITY) ? 0.0f : exp2f(m - mn);
    const float c2 = (m2 == -INFINITY) ? 0.0f : exp2f(m2 - mn);
    l = l * c1 + l2 * c2;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = acc[i] * c1 + __shfl_xor_sync(0xffffffffu, acc[i], o) * c2;
    m = mn;
  }
  if (g == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) s_acc[warp][e * 8 + i] = acc[i];
    if (e == 0) {
      s_m[warp] = m;
      s_l[warp] = l;
    }
  }
  __syncthreads();
  // merge the 4 warps: thread d < 64 owns output dim d
  float M = -INFINITY, L = 0.0f, A = 0.0f;
  const int d = threadIdx.x;
  if (d < HSZ) {
    for (int w = 0; w < DEC_WARPS; ++w) M = fmaxf(M, s_m[w]);
    for (int w = 0; w < DEC_WARPS; ++w) {
      const float c = (s_m[w] == -INFINITY) ? 0.0f : exp2f(s_m[w] - M);
      L += s_l[w] * c;
      A += s_acc[w][d] * c;
    }
  }
  const int b = bh / nh, h = bh - b * nh;
  const size_t yoff = static_cast<size_t>(b) * C + h * HSZ;
  if (splits == 1) {
    if (d < HSZ) {
      const float o = A / L;
      const T ho = from_f32<T>(o);
      y[yoff + d] = ho;
      if (y_lo) y_lo[yoff + d] = from_f32<T>(o - to_f32(ho));
    }
    return;
  }
  float* part = ws + (static_cast<size_t>(bh) * splits + split) * (HSZ + 2);
  if (d < HSZ) part[2 + d] = A;
  if (d == 0) {
    part[0] = M;
    part[1] = L;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&tickets[bh], 1u) == static_cast<unsigned>(splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (d < HSZ) {
    float MM = -INFINITY;
    for (int s = 0; s < splits; ++s) MM = fmaxf(MM, __ldcg(ws + (static_cast<size_t>(bh) * splits + s) * (HSZ + 2)));
    float LL = 0.0f, AA = 0.0f;
    for (int s = 0; s < splits; ++s) {
      const float* p = ws + (static_cast<size_t>(bh) * splits + s) * (HSZ + 2);
      const float ms = __ldcg(p);
      const float c = (ms == -INFINITY) ? 0.0f : exp2f(ms - MM);
      LL += __ldcg(p + 1) * c;
      AA += __ldcg(p + 2 + d) * c;
    }
    const float o = AA / LL;
    const T ho = from_f32<T>(o);
    y[yoff + d] = ho;
    if (y_lo) y_lo[yoff + d] = from_f32<T>(o - to_f32(ho));
  }
  if (threadIdx.x == 0) tickets[bh] = 0u;
}

// ------------------------------------------------------------------ prefill, fp32

// grid (T, B*nh), 32 threads: one warp per query.  Scores are kept in shared memory.
template <int HSZ>
__global__ void attn_prefill_f32(const float* __restrict__ q, const float* __restrict__ kc,
                                 const float* __restrict__ vc, KvLayout kv, int nh, int T, int block, int pos0,
                                 float* __restrict__ y, int C) {
  extern __shared__ float s_p[];  // pos0 + T scores
  const int t = blockIdx.x, bh = blockIdx.y, lane = threadIdx.x;
  const int qp = pos0 + t;
  const float* qr = q + (static_cast<size_t>(bh) * T + t) * HSZ;
  const int bq = bh / nh, hq = bh - bq * nh;
  float mx = -INFINITY;
  for (int j = lane; j <= qp; j += 32) {
    float d = 0.0f;
    const float* kr = kc + kv.row(bq, hq, j) * HSZ;
    for (int i = 0; i < HSZ; ++i) d = fmaf(qr[i], kr[i], d);
    d *= (HSZ == 64 ? 0.125f : 0.17677669529663688f);
    s_p[j] = d;
    mx = fmaxf(mx, d);
  }
  mx = warp_max(mx);
  float sum = 0.0f;
  for (int j = lane; j <= qp; j += 32) {
    const float p = expf(s_p[j] - mx);
    s_p[j] = p;
    sum += p;
  }
  sum = warp_sum(sum);
  __syncwarp();
  const int b = bh / nh, hh = bh - b * nh;
  for (int dd = lane; dd < HSZ; dd += 32) {
    float a = 0.0f;
    for (int j = 0; j <= qp; ++j) a = fmaf(s_p[j], vc[kv.row(bq, hq, j) * HSZ + dd], a);
    y[(static_cast<size_t>(b) * T + t) * C + hh * HSZ + dd] = a / sum;
  }
}

}  // namespace kvgpt
