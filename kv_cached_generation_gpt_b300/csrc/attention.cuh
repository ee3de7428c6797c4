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
//   attn_prefill_tc     -- FlashAttention-style tiles on tcgen05: 128 queries x 64 keys per
//                          step, S and O accumulated in TMEM, online softmax in fp32.
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

// ------------------------------------------------------------------ prefill, tcgen05

// FlashAttention-style causal prefill on the Blackwell tensor core.  A work item is 128 query
// rows of one (b, h); a persistent CTA walks items (heaviest first, strided by the grid) and,
// for each, the key tiles of 64 it needs:
//   S = Q K^T          tcgen05.mma M=128 N=64 K=64, fp32 in TMEM columns [0, 64)
//   softmax            warps 0-3, thread = query row = TMEM lane: scale, causal mask, running
//                      max and sum (fp32); P = exp2(s - m) as bf16 into shared memory
//   O += P V           tcgen05.mma M=128 N=64 K=64 keys, V read as an MN-major operand (the
//                      cache rows are [key][dim]), fp32 in TMEM, two O buffers (items alternate)
// Q, K and V tiles arrive by TMA (128-byte swizzle) from the q buffer and the cache rows of the
// (b, h), found through KvLayout (a 64-key tile never straddles a page).  Every barrier's phase
// runs on across items, so the next item's Q and K/V loads and its first S overlap the current
// item's last tiles and output.  The MMA warp issues S for tile j+1 as soon as the softmax warps
// have read S for tile j, and P is double-buffered, so the softmax of tile j overlaps the MMAs of
// tiles j-1 and j+1; K/V run three tiles ahead; two CTAs per SM overlap further.  The running max is raised lazily: O
// (in TMEM) and the sum are rescaled only when a row's max grows by more than 2^8, so
// p = exp2(s - m) stays <= 256 and most tiles skip the TMEM round trip (y = O / l is exact for
// any m used consistently).  Keys at or past pos0 + T in the last tile are zeroed in V before
// P V (the cache may hold anything there) and masked in S.
constexpr int PT_BQ = 128;       // query rows per item (MMA M)
constexpr int PT_BK = 64;        // keys per tile
constexpr int PT_THREADS = 192;  // warps 0-3 softmax + output, warp 4 TMA, warp 5 MMA
constexpr uint32_t PT_Q_BYTES = PT_BQ * HS * 2;
constexpr uint32_t PT_KV_BYTES = PT_BK * HS * 2;
constexpr uint32_t PT_P_BYTES = PT_BQ * PT_BK * 2;
constexpr int PT_STAGES = 3;     // K/V ring
constexpr uint32_t PT_SMEM = 1024 + PT_Q_BYTES + 2 * PT_STAGES * PT_KV_BYTES + 2 * PT_P_BYTES + 256;
constexpr float PT_RESCALE_LOG2 = 8.0f;
constexpr int PT_CTAS_PER_SM = 2;

// 2^x by the SFU's approximate instruction (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Item k of n_qt * BH items (heaviest first): query tile n_qt - 1 - k / BH of (b, h) = k % BH.
struct PtItem {
  int bh, q0, nk;
};
__device__ __forceinline__ PtItem pt_item(int k, int BH, int n_qt, int T, int pos0) {
  PtItem it;
  const int qt = n_qt - 1 - k / BH;
  it.bh = k - (k / BH) * BH;
  it.q0 = qt * PT_BQ;
  const int last_q = min(it.q0 + PT_BQ, T) - 1;
  it.nk = (pos0 + last_q) / PT_BK + 1;
  return it;
}

// grid = min(items, PT_CTAS_PER_SM x SMs) persistent CTAs, PT_THREADS threads, PT_SMEM dynamic
// shared memory; items = ceil(T/128) x B*nh.  tmQ: q as [B*nh*T][64] rows; tmK / tmV: one layer's
// cache as [rows][64] (KvLayout::row numbering); 128-row (q) and 64-row (cache) boxes of 64
// columns with 128-byte swizzle.  Queries t in [0, T) sit at positions pos0 + t and see keys
// 0 .. pos0 + t.
__global__ void __launch_bounds__(PT_THREADS, PT_CTAS_PER_SM) attn_prefill_tc(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmV, KvLayout kv, int nh, int BH, int T, int pos0,
    __nv_bfloat16* __restrict__ y, int C, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + PT_Q_BYTES;                // PT_STAGES stages
  uint8_t* sV = sK + PT_STAGES * PT_KV_BYTES;   // PT_STAGES stages
  uint8_t* sP = sV + PT_STAGES * PT_KV_BYTES;   // 2 buffers (tiles alternate)
  uint64_t* bar = reinterpret_cast<uint64_t*>(sP + 2 * PT_P_BYTES);
  uint64_t* q_full = bar;                      // Q of item i landed (phase i)
  uint64_t* q_empty = bar + 1;                 // the last S of item i is done: Q may be replaced
  uint64_t* k_full = bar + 2;                  // [PT_STAGES], phases run over the tiles of all items
  uint64_t* v_full = k_full + PT_STAGES;       // [PT_STAGES]
  uint64_t* kv_empty = v_full + PT_STAGES;     // [PT_STAGES]
  uint64_t* s_full = kv_empty + PT_STAGES;     // per tile
  uint64_t* s_empty = s_full + 1;              // per tile: the softmax warps have read S
  uint64_t* p_full = s_empty + 1;              // per tile: P is written (and the V tail zeroed)
  uint64_t* p_empty = p_full + 1;              // [2] per P buffer: the P V that read it is done
  uint64_t* o_full = p_empty + 2;              // [2] per item: O buffer i%2 is complete
  uint64_t* o_empty = o_full + 2;              // [2] per item: O buffer i%2 has been read out
  uint64_t* drain = o_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (T + PT_BQ - 1) / PT_BQ;
  const int n_items = n_qt * BH;
  const int kv_len = pos0 + T;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < PT_STAGES; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 128);
    mbar_init(p_full, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_empty[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], 128);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;  // O buffers at columns 64 and 128

  if (warp == 4) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int g = 0, n_it = 0;  // tiles and items issued
      bool ok = true;
      for (int k = blockIdx.x; k < n_items && ok; k += gridDim.x, ++n_it) {
        const PtItem it = pt_item(k, BH, n_qt, T, pos0);
        const int b = it.bh / nh, h = it.bh - b * nh;
        if (n_it > 0 && !(ok = mbar_wait(q_empty, (n_it - 1) & 1, err))) break;
        mbar_arrive_expect_tx(q_full, PT_Q_BYTES);
        tma_load_2d(&tmQ, q_full, sQ, 0, it.bh * T + it.q0);
        for (int j = 0; j < it.nk; ++j, ++g) {
          const int st = g % PT_STAGES;
          if (g >= PT_STAGES && !(ok = mbar_wait(&kv_empty[st], ((g / PT_STAGES) & 1) ^ 1, err))) break;
          const int row = static_cast<int>(kv.row(b, h, j * PT_BK));
          mbar_arrive_expect_tx(&k_full[st], PT_KV_BYTES);
          tma_load_2d(&tmK, &k_full[st], sK + st * PT_KV_BYTES, 0, row);
          mbar_arrive_expect_tx(&v_full[st], PT_KV_BYTES);
          tma_load_2d(&tmV, &v_full[st], sV + st * PT_KV_BYTES, 0, row);
        }
      }
      // every load has landed before the CTA may exit
      if (n_it > 0) mbar_wait(q_full, (n_it - 1) & 1, err);
      for (int t = max(0, g - PT_STAGES); t < g; ++t) {
        mbar_wait(&k_full[t % PT_STAGES], (t / PT_STAGES) & 1, err);
        mbar_wait(&v_full[t % PT_STAGES], (t / PT_STAGES) & 1, err);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(PT_BQ, PT_BK);
      const uint32_t id_pv = idesc_bf16_f32(PT_BQ, HS) | (1u << 16);  // B (V) is MN-major
      const uint32_t aq = smem_u32(sQ), ap = smem_u32(sP);
      int g = 0, n_it = 0;
      bool ok = true;
      auto issue_s = [&](int t) {  // S = Q K^T for global tile t
        const uint32_t bk = smem_u32(sK + (t % PT_STAGES) * PT_KV_BYTES);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tS, sdesc_sw128(aq + 32 * ks), sdesc_sw128(bk + 32 * ks), id_s, ks != 0);
        umma_commit(s_full);
      };
      for (int k = blockIdx.x; k < n_items && ok; k += gridDim.x, ++n_it) {
        const PtItem it = pt_item(k, BH, n_qt, T, pos0);
        const uint32_t tO = tmem + 64 + 64 * (n_it & 1);
        // S of the item's first tile: Q landed, K landed, the previous S has been read
        if (!(ok = mbar_wait(q_full, n_it & 1, err) && mbar_wait(&k_full[g % PT_STAGES], (g / PT_STAGES) & 1, err) &&
                   (g == 0 || mbar_wait(s_empty, (g - 1) & 1, err))))
          break;
        tc_fence_after();
        issue_s(g);
        if (it.nk == 1) umma_commit(q_empty);
        // this item's O buffer has been read out (item n_it - 2)
        if (n_it >= 2 && !(ok = mbar_wait(&o_empty[n_it & 1], ((n_it >> 1) - 1) & 1, err))) break;
        for (int j = 0; j < it.nk; ++j) {
          const int t = g + j, st = t % PT_STAGES;
          if (j + 1 < it.nk) {
            const int t1 = t + 1;
            if (!(ok = mbar_wait(s_empty, t & 1, err) &&
                       mbar_wait(&k_full[t1 % PT_STAGES], (t1 / PT_STAGES) & 1, err)))
              break;
            tc_fence_after();
            issue_s(t1);
            if (j + 2 == it.nk) umma_commit(q_empty);  // the item's last S is issued
          }
          if (!(ok = mbar_wait(p_full, t & 1, err) && mbar_wait(&v_full[st], (t / PT_STAGES) & 1, err))) break;
          tc_fence_after();
          const uint32_t bv = smem_u32(sV + st * PT_KV_BYTES), bp = ap + (t & 1) * PT_P_BYTES;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)  // 16 keys per step: 2 swizzle atoms of 8 key rows
            umma_bf16(tO, sdesc_sw128(bp + 32 * ks), sdesc_sw128(bv + 2048 * ks), id_pv, (j | ks) != 0);
          umma_commit(&p_empty[t & 1]);
          umma_commit(&kv_empty[st]);
        }
        if (ok) umma_commit(&o_full[n_it & 1]);
        g += it.nk;
      }
      umma_commit(drain);  // no MMA of this CTA is in flight once it completes
      mbar_wait(drain, 0, err);
    }
  } else {
    // softmax warps: thread = query row r of the item
    const int r = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float sc = 0.125f * LOG2E_F;
    int g = 0, n_it = 0;
    bool ok = true;
    for (int k = blockIdx.x; k < n_items && ok; k += gridDim.x, ++n_it) {
      const PtItem it = pt_item(k, BH, n_qt, T, pos0);
      const uint32_t tO = tmem + 64 + 64 * (n_it & 1);
      const int qi = it.q0 + r;
      const bool valid = qi < T;
      const int qpos = pos0 + qi;
      float m_used = -INFINITY, l = 0.0f;
      for (int j = 0; j < it.nk; ++j) {
        const int t = g + j;
        if (!(ok = mbar_wait(s_full, t & 1, err))) break;
        tc_fence_after();
        float s[PT_BK];
        {
          // the four 16-column loads in flight together, one wait
          uint32_t r0[16], r1[16], r2[16], r3[16];
          tmem_ld16_raw(tS + lane_base, r0);
          tmem_ld16_raw(tS + lane_base + 16, r1);
          tmem_ld16_raw(tS + lane_base + 32, r2);
          tmem_ld16_raw(tS + lane_base + 48, r3);
          tmem_wait_ld16(r0, r1);
          tmem_wait_ld16(r2, r3);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            s[i] = __uint_as_float(r0[i]);
            s[16 + i] = __uint_as_float(r1[i]);
            s[32 + i] = __uint_as_float(r2[i]);
            s[48 + i] = __uint_as_float(r3[i]);
          }
        }
        tc_fence_before();
        mbar_arrive(s_empty);
        const int kbase = j * PT_BK;
        // causal mask (and rows past T): only tiles reaching past the warp's first query position
        if (__any_sync(0xffffffffu, !valid || kbase + PT_BK - 1 > qpos)) {
#pragma unroll
          for (int c = 0; c < PT_BK; ++c)
            if (!valid || kbase + c > qpos) s[c] = -INFINITY;
        }
        // row max of the raw scores in 8 independent chains, then scaled (sc > 0)
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
        for (int c = 8; c < PT_BK; ++c) m8[c & 7] = fmaxf(m8[c & 7], s[c]);
        const float mraw = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                 fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        const float mx = mraw * sc;
        const bool need = mx > m_used + PT_RESCALE_LOG2 || (m_used == -INFINITY && mx > -INFINITY);
        // P buffer t%2 is free once the P V of tile t-2 is done (each buffer's phases are waited in
        // order)
        if (t >= 2 && !(ok = mbar_wait(&p_empty[t & 1], ((t >> 1) - 1) & 1, err))) break;
        if (__any_sync(0xffffffffu, need && j > 0)) {
          // O *= exp2(m_used - mx) on the rows whose max moved (warp-wide TMEM round trip), once
          // the P V of tile t-1 (this item's previous tile) is done
          if (!(ok = mbar_wait(&p_empty[(t - 1) & 1], ((t - 1) >> 1) & 1, err))) break;
          const float corr = (need && j > 0) ? exp2f(m_used - mx) : 1.0f;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < HS; c += 16) {
            float v[16];
            tmem_ld16(tO + lane_base + c, v);
            uint32_t u[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(v[i] * corr);
            tmem_st16(tO + lane_base + c, u);
          }
          tmem_wait_st();
          tc_fence_before();
        }
        if (need) {
          l = (m_used == -INFINITY) ? 0.0f : l * exp2f(m_used - mx);
          m_used = mx;
        }
        // P = exp2(s * sc - m) (bf16) into row r of the 128 x 64 tile, 128-byte swizzle; the row
        // sum in 8 independent chains.  A row without any visible key so far (only rows past T)
        // gets P = 0.
        const uint32_t prow = smem_u32(sP + (t & 1) * PT_P_BYTES) + static_cast<uint32_t>(r * 128);
        const bool live = m_used != -INFINITY;
        const float neg_m = live ? -m_used : 0.0f;
        float ps8[8];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          float p[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) p[i] = live ? ex2_approx(fmaf(s[ch * 8 + i], sc, neg_m)) : 0.0f;
#pragma unroll
          for (int i = 0; i < 8; ++i) ps8[i] = ch == 0 ? p[i] : ps8[i] + p[i];
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + static_cast<uint32_t>((ch ^ (r & 7)) << 4)),
                       "r"(pack_bf16x2(p[0], p[1])), "r"(pack_bf16x2(p[2], p[3])), "r"(pack_bf16x2(p[4], p[5])),
                       "r"(pack_bf16x2(p[6], p[7]))
                       : "memory");
        }
        l += ((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) + ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7]));
        if (j == it.nk - 1 && kbase + PT_BK > kv_len) {
          // keys past the live cache: zero their V rows (0 * NaN would poison O)
          const int st = t % PT_STAGES;
          if (!(ok = mbar_wait(&v_full[st], (t / PT_STAGES) & 1, err))) break;
          const uint32_t vb = smem_u32(sV + st * PT_KV_BYTES);
          const int first = kv_len - kbase;
          for (int i = r; i < (PT_BK - first) * 8; i += 128)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vb + static_cast<uint32_t>((first + i / 8) * 128 + (i % 8) * 16)),
                         "r"(0u)
                         : "memory");
        }
        fence_proxy_async_smem();  // the MMA reads P (and V) through the async proxy
        mbar_arrive(p_full);
      }
      if (!ok) break;
      g += it.nk;
      if (!(ok = mbar_wait(&o_full[n_it & 1], (n_it >> 1) & 1, err))) break;  // the item's last P V is done
      tc_fence_after();
      const float inv = 1.0f / l;
      const int b = it.bh / nh, h = it.bh - b * nh;
      __nv_bfloat16* dst = y + (static_cast<size_t>(b) * T + qi) * C + h * HS;
#pragma unroll
      for (int c = 0; c < HS; c += 16) {
        float v[16];
        tmem_ld16(tO + lane_base + c, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= inv;
        if (valid) store16(dst + c, v);
      }
      tc_fence_before();
      mbar_arrive(&o_empty[n_it & 1]);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
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
