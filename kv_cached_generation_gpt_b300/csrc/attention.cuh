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
//   attn_prefill_bf16   -- FlashAttention-style tiles: 64 queries x 64 keys per step on
//                          mma.sync m16n8k16 (bf16 in, fp32 accumulate), online softmax.
//   attn_prefill_f32    -- exact fp32 path for fp32 models (warp per query).
#pragma once

#include "common.cuh"

namespace kvgpt {

constexpr int HS = 64;
constexpr float LOG2E_F = 1.4426950408889634f;

// ------------------------------------------------------------------ decode

constexpr int DEC_THREADS = 128;  // 4 warps
constexpr int DEC_UNROLL = 4;     // keys per lane group per iteration

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
template <typename T, int HSZ, bool PAGED = false>
__global__ void __launch_bounds__(DEC_THREADS) attn_decode_kernel(const T* __restrict__ q, const T* __restrict__ kc,
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
  constexpr int KPI = 4 * KPW;        // keys per CTA per unrolled slot
  __shared__ float s_m[4], s_l[4];
  __shared__ float s_acc[4][HSZ];
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
    for (int w = 0; w < 4; ++w) M = fmaxf(M, s_m[w]);
    for (int w = 0; w < 4; ++w) {
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

// ------------------------------------------------------------------ prefill, bf16 tensor cores

constexpr int PF_BQ = 64, PF_BKEY = 64, PF_THREADS = 128;  // 4 warps x 16 query rows

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of 16-byte chunk c of row r in a 64 x 64 bf16 tile with XOR swizzle.
__device__ __forceinline__ uint32_t swz(int r, int c) { return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4)); }

// Copy ROWS consecutive rows of 64 bf16 starting at src into a swizzled tile; rows >= nvalid are zeros.
template <int ROWS>
__device__ __forceinline__ void load_tile64(uint32_t tile, const __nv_bfloat16* src, int nvalid) {
#pragma unroll
  for (int i = 0; i < ROWS * 8 / PF_THREADS; ++i) {
    const int idx = threadIdx.x + i * PF_THREADS;  // ROWS x 8 chunks of 16 B
    const int r = idx >> 3, c = idx & 7;
    const bool ok = r < nvalid;
    const __nv_bfloat16* p = src + static_cast<size_t>(ok ? r : 0) * HS + c * 8;
    cp_async16(tile + swz(r, c), p, ok);
  }
}

// grid (ceil(T/64), B*nh).  Queries t in [0, T) sit at positions pos0 + t; keys 0..pos0+T-1.
// Query blocks run heaviest (most keys) first: block qb = gridDim.x - 1 - blockIdx.x.
__global__ void __launch_bounds__(PF_THREADS) attn_prefill_bf16(const __nv_bfloat16* __restrict__ q,
                                                                const __nv_bfloat16* __restrict__ kc,
                                                                const __nv_bfloat16* __restrict__ vc, KvLayout kv,
                                                                int nh, int T,
                                                                int block, int pos0, __nv_bfloat16* __restrict__ y,
                                                                int C) {
  __shared__ __align__(128) __nv_bfloat16 sQ[PF_BQ * HS];
  __shared__ __align__(128) __nv_bfloat16 sK[2][PF_BKEY * HS];
  __shared__ __align__(128) __nv_bfloat16 sV[2][PF_BKEY * HS];
  const int qb = gridDim.x - 1 - blockIdx.x, bh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int q0 = qb * PF_BQ;
  const int n_keys = pos0 + T;
  const int last_key = min(pos0 + q0 + PF_BQ - 1, n_keys - 1);
  const int n_kb = last_key / PF_BKEY + 1;
  const __nv_bfloat16* qg = q + static_cast<size_t>(bh) * T * HS;
  const int bq = bh / nh, hq = bh - bq * nh;
  // keys r .. r+63 of this (b, h), r a multiple of 64: consecutive rows (pages hold >= 64)
  auto krows = [&](int r) { return kc + kv.row(bq, hq, r) * HS; };
  auto vrows = [&](int r) { return vc + kv.row(bq, hq, r) * HS; };
  constexpr uint32_t TILE_BYTES = PF_BKEY * HS * 2;
  const uint32_t sq = smem_u32(sQ), sk0 = smem_u32(sK[0]), sv0 = smem_u32(sV[0]);

  load_tile64<PF_BQ>(sq, qg + static_cast<size_t>(q0) * HS, T - q0);
  load_tile64<PF_BKEY>(sk0, krows(0), n_keys);
  load_tile64<PF_BKEY>(sv0, vrows(0), n_keys);
  cp_async_commit();

  uint32_t qa[4][4];  // A fragments of this warp's 16 query rows, 4 k-steps of 16 dims
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[i][j] = 0.0f;
  float row_m[2] = {-INFINITY, -INFINITY}, row_l[2] = {0.0f, 0.0f};
  const float sc = 0.125f * LOG2E_F;
  const int qpos0 = pos0 + q0 + warp * 16 + gq;  // absolute position of row gq (row gq+8 is +8)

  for (int kb = 0; kb < n_kb; ++kb) {
    const int buf = kb & 1;
    const uint32_t skb = sk0 + buf * TILE_BYTES, svb = sv0 + buf * TILE_BYTES;
    if (kb + 1 < n_kb) {
      load_tile64<PF_BKEY>(sk0 + (buf ^ 1) * TILE_BYTES, krows((kb + 1) * PF_BKEY), n_keys - (kb + 1) * PF_BKEY);
      load_tile64<PF_BKEY>(sv0 + (buf ^ 1) * TILE_BYTES, vrows((kb + 1) * PF_BKEY), n_keys - (kb + 1) * PF_BKEY);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (kb == 0) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        // matrices: rows 0-7 / 8-15 of the warp's 16 rows x dims [16ks, 16ks+8) / [16ks+8, 16ks+16)
        const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = ks * 2 + (lane >> 4);
        ldmatrix_x4(qa[ks], sq + swz(r, c));
      }
    }
    // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int j = 0; j < 4; ++j) s[nt][j] = 0.0f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t kf[4];
        const int r = nt * 8 + (lane & 7);
        const int c = half * 4 + (lane >> 3);
        ldmatrix_x4(kf, skb + swz(r, c));
        mma_bf16_16816(s[nt], qa[half * 2], kf[0], kf[1]);
        mma_bf16_16816(s[nt], qa[half * 2 + 1], kf[2], kf[3]);
      }
    }
    // scale, causal mask, online softmax (rows gq and gq+8 of the warp's 16)
    const int kbase = kb * PF_BKEY;
    const bool need_mask = kbase + PF_BKEY - 1 > pos0 + q0 + warp * 16;
    float mx[2] = {row_m[0], row_m[1]};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float v = s[nt][j] * sc;
        if (need_mask) {
          const int key = kbase + nt * 8 + tq * 2 + (j & 1);
          const int qp = qpos0 + (j >> 1) * 8;
          if (key > qp) v = -INFINITY;
        }
        s[nt][j] = v;
        mx[j >> 1] = fmaxf(mx[j >> 1], v);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
    }
    float corr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      corr[h] = (mx[h] == -INFINITY) ? 1.0f : exp2f(row_m[h] - mx[h]);
      row_m[h] = mx[h];
      row_l[h] *= corr[h];
    }
#pragma unroll
    for (int dn = 0; dn < 8; ++dn) {
      o[dn][0] *= corr[0];
      o[dn][1] *= corr[0];
      o[dn][2] *= corr[1];
      o[dn][3] *= corr[1];
    }
    uint32_t pa[4][4];  // P as A fragments, 4 k-steps of 16 keys
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      float p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float mm = row_m[j >> 1];
        p[j] = (mm == -INFINITY) ? 0.0f : exp2f(s[nt][j] - mm);
        row_l[j >> 1] += p[j];
      }
      const int ks = nt >> 1, hi = nt & 1;
      pa[ks][hi * 2 + 0] = pack_bf16x2(p[0], p[1]);
      pa[ks][hi * 2 + 1] = pack_bf16x2(p[2], p[3]);
    }
    // O += P V: 8 n-tiles of 8 dims, 4 k-steps of 16 keys
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int dp = 0; dp < 4; ++dp) {  // pairs of dim n-tiles
        uint32_t vf[4];
        const int r = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = dp * 2 + (lane >> 4);
        ldmatrix_x4_trans(vf, svb + swz(r, c));
        mma_bf16_16816(o[dp * 2], pa[ks], vf[0], vf[1]);
        mma_bf16_16816(o[dp * 2 + 1], pa[ks], vf[2], vf[3]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    row_l[h] += __shfl_xor_sync(0xffffffffu, row_l[h], 1);
    row_l[h] += __shfl_xor_sync(0xffffffffu, row_l[h], 2);
  }
  const int b = bh / nh, hh = bh - b * nh;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = q0 + warp * 16 + gq + h * 8;
    if (t < T) {
      const float inv = 1.0f / row_l[h];
      __nv_bfloat16* yr = y + (static_cast<size_t>(b) * T + t) * C + hh * HS;
#pragma unroll
      for (int dn = 0; dn < 8; ++dn) {
        *reinterpret_cast<uint32_t*>(yr + dn * 8 + tq * 2) = pack_bf16x2(o[dn][h * 2] * inv, o[dn][h * 2 + 1] * inv);
      }
    }
  }
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
