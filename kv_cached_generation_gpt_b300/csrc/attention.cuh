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
//   attn_decode_bulk    -- the same for bf16 / head size 64 / up to DB_MAX_SPLITS splits per
//                          (b, h) (at most 512 (b, h) pairs), the cache rows streamed through a
//                          shared-memory ring by bulk copies; in a decode step it starts on the
//                          older rows before the kernel that appends the newest key has finished.
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

// ------------------------------------------------------------------ decode, streamed through shared memory

// The same decode attention for bf16 and head size 64 (one split per (b, h), or a few for a
// few pairs), with the cache rows streamed through shared memory instead of registers: a
// producer warp issues untiled bulk
// copies of DB_KEYS consecutive K rows and the matching V rows (2 x 8 KiB) into a ring of
// DB_STAGES stages, and 8 consumer warps score and accumulate from shared memory.  A CTA then
// keeps up to 48 KiB of loads in flight however few registers its warps hold, which is what a
// grid of a few hundred CTAs (one 32-sequence decode chain) lacks with register loads; 48 KiB
// (not more) so that four CTAs fit an SM beside the kernels of the other decode chain.
// Measured on the B=64 decode step (two chains of 32 sequences): 3 stages of 64 keys 658 us per
// step, against 689 (4 x 64), 661 (2 x 96), 725 (2 x 64), 737-741 (3-4 x 32) and 720 us for the
// register-load kernel.
// Key j of a stage goes to warp (j mod 32) / 4, lane group j mod 4, as in attn_decode_kernel;
// the online softmax is rescaled once per stage.  A stage of 64 keys starts at a multiple of 64,
// so with a paged cache (pages of at least 64 positions, a power of two) it lies in one page.
constexpr int DB_WARPS = 8;                           // consumer warps
constexpr int DB_THREADS = 32 * (DB_WARPS + 1);       // + the producer warp
constexpr int DB_KEYS = 64;                           // keys per stage
constexpr int DB_STAGES = 3;
constexpr int DB_MAX_SPLITS = 8;                      // splits per (b, h), whole stages each
constexpr uint32_t DB_ROW_BYTES = HS * 2;             // one bf16 cache row
constexpr uint32_t DB_STAGE_BYTES = 2 * DB_KEYS * DB_ROW_BYTES;  // K rows, then V rows
constexpr uint32_t DB_SMEM = DB_STAGES * DB_STAGE_BYTES + 2 * DB_STAGES * 8;

// grid (B*nh, splits): keys 0..t_len-1, t_len = *pos0 + 1 (or pos_rows[b] + 1), in stages of
// DB_KEYS; split s takes stages [s*cps, (s+1)*cps), cps = ceil(stages / splits), and with
// splits > 1 leaves (m, l, acc[64]) in ws for the last split to finish (ticket) to merge in
// split order, as attn_decode_kernel does.  y [B][C] (+ y_lo).
// EARLY (a decode step's programmatic dependent launch): the cache length and every row before
// the newest key were written before the step began, so the producer reads the length and fills
// the ring with those rows before waiting for the kernel that appends the newest key; q and
// the chunk holding that key wait for it.
template <bool PAGED, bool EARLY = false>
__global__ void __launch_bounds__(DB_THREADS) attn_decode_bulk(const __nv_bfloat16* __restrict__ q,
                                                                const __nv_bfloat16* __restrict__ kc,
                                                                const __nv_bfloat16* __restrict__ vc, KvLayout kv,
                                                                int nh, int block, const int* pos0,
                                                                const int* pos_rows, float* __restrict__ ws,
                                                                unsigned int* __restrict__ tickets,
                                                                __nv_bfloat16* __restrict__ y,
                                                                __nv_bfloat16* __restrict__ y_lo, int C, int* err) {
  extern __shared__ __align__(128) uint8_t db_smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(db_smem + DB_STAGES * DB_STAGE_BYTES);
  uint64_t* empty = full + DB_STAGES;
  __shared__ float s_m[DB_WARPS], s_l[DB_WARPS];
  __shared__ float s_acc[DB_WARPS][HS];
  __shared__ int s_last;
  const int bh = blockIdx.x, split = blockIdx.y, splits = gridDim.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = lane & 7, g = lane >> 3;  // 8 lanes per key, 4 keys per warp per pass
  if (threadIdx.x == 0) {
    for (int i = 0; i < DB_STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], DB_WARPS);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const bool producer = warp == DB_WARPS;
  if (!(EARLY && producer)) griddep_wait();  // q and the new key/value come from the previous kernel
  griddep_launch();
  const int t_len = (pos_rows ? pos_rows[bh / nh] : *pos0) + 1;
  if (t_len > block) {
    if (threadIdx.x == 0) atomicOr(err, ERR_POSITION);
    return;
  }
  const int bq = bh / nh, hq = bh - bq * nh;
  const int n_all = (t_len + DB_KEYS - 1) / DB_KEYS;  // stages of the whole (b, h)
  const int cps = (n_all + splits - 1) / splits;
  const int c_beg = min(split * cps, n_all);
  const int nchunks = min(c_beg + cps, n_all) - c_beg;  // this split's stages (possibly none)

  if (producer) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();  // every cache row is read once per step
      const size_t row0 = PAGED ? 0 : (static_cast<size_t>(bq) * kv.nh + hq) * kv.block;
      // stages wholly before the newest key (t_len - 1) need not wait for the previous kernel
      const int ready = EARLY ? min(max((t_len - 1) / DB_KEYS - c_beg, 0), nchunks) : 0;
      int c = 0;
      for (; c < nchunks; ++c) {
        const int st = c % DB_STAGES;
        if (EARLY && c == min(ready, DB_STAGES)) griddep_wait();
        if (c >= DB_STAGES && !mbar_wait(&empty[st], ((c / DB_STAGES) & 1) ^ 1, err)) break;
        const int k0 = (c_beg + c) * DB_KEYS;
        const uint32_t bytes = static_cast<uint32_t>(min(DB_KEYS, t_len - k0)) * DB_ROW_BYTES;
        const size_t row = PAGED ? kv.row(bq, hq, k0) : row0 + k0;
        uint8_t* dst = db_smem + st * DB_STAGE_BYTES;
        mbar_arrive_expect_tx(&full[st], 2 * bytes);
        bulk_load(dst, kc + row * HS, bytes, &full[st], pol);
        bulk_load(dst + DB_KEYS * DB_ROW_BYTES, vc + row * HS, bytes, &full[st], pol);
      }
      // every copy issued has landed before the CTA may exit
      for (int t = max(0, c - DB_STAGES); t < c; ++t) mbar_wait(&full[t % DB_STAGES], (t / DB_STAGES) & 1, err);
    }
    return;  // the producer warp takes no part in the merge below (named barrier of the consumers)
  }

  float qv[8];
  {
    Vec8<__nv_bfloat16> t;
    t.load(q + static_cast<size_t>(bh) * HS + e * 8);
    t.to_float(qv);
#pragma unroll
    for (int i = 0; i < 8; ++i) qv[i] *= 0.125f * LOG2E_F;  // 1/sqrt(64), log2 units
  }
  float m = -INFINITY, l = 0.0f, acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  constexpr int U = DB_KEYS / 32;  // keys per lane group per stage
  for (int c = 0; c < nchunks; ++c) {
    const int st = c % DB_STAGES;
    if (!mbar_wait(&full[st], (c / DB_STAGES) & 1, err)) break;
    const uint32_t sk = smem_u32(db_smem + st * DB_STAGE_BYTES), sv = sk + DB_KEYS * DB_ROW_BYTES;
    const int k0 = (c_beg + c) * DB_KEYS;
    float sc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kk = u * 32 + warp * 4 + g;
      float d = 0.0f;
      if (k0 + kk < t_len) {
        Vec8<__nv_bfloat16> kr;
        kr.u = ld_shared_u4(sk + kk * DB_ROW_BYTES + e * 16);
        float kf[8];
        kr.to_float(kf);
#pragma unroll
        for (int i = 0; i < 8; ++i) d = fmaf(qv[i], kf[i], d);
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      sc[u] = (k0 + kk < t_len) ? d : -INFINITY;
    }
    float mn = m;
#pragma unroll
    for (int u = 0; u < U; ++u) mn = fmaxf(mn, sc[u]);
    const float corr = (mn == -INFINITY) ? 1.0f : exp2f(m - mn);
    l *= corr;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] *= corr;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kk = u * 32 + warp * 4 + g;
      if (k0 + kk < t_len) {
        const float p = exp2f(sc[u] - mn);
        l += p;
        Vec8<__nv_bfloat16> vr;
        vr.u = ld_shared_u4(sv + kk * DB_ROW_BYTES + e * 16);
        float vf[8];
        vr.to_float(vf);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vf[i], acc[i]);
      }
    }
    m = mn;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage
  }

  // merge the 4 lane groups of the warp, then the 8 warps (as attn_decode_kernel)
#pragma unroll
  for (int o = 8; o <= 16; o <<= 1) {
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
  asm volatile("bar.sync 1, %0;" ::"r"(32 * DB_WARPS) : "memory");
  const int d = threadIdx.x;
  float M = -INFINITY, L = 0.0f, A = 0.0f;
  if (d < HS) {
    for (int w = 0; w < DB_WARPS; ++w) M = fmaxf(M, s_m[w]);
    for (int w = 0; w < DB_WARPS; ++w) {
      const float cw = (s_m[w] == -INFINITY) ? 0.0f : exp2f(s_m[w] - M);
      L += s_l[w] * cw;
      A += s_acc[w][d] * cw;
    }
  }
  const size_t yoff = static_cast<size_t>(bq) * C + hq * HS;
  if (splits == 1) {
    if (d < HS) {
      const float o = A / L;
      const __nv_bfloat16 ho = __float2bfloat16_rn(o);
      y[yoff + d] = ho;
      if (y_lo) y_lo[yoff + d] = __float2bfloat16_rn(o - __bfloat162float(ho));
    }
    return;
  }
  // splits: partial (m, l, acc) to ws; the last split of the (b, h) to take the ticket merges
  float* part = ws + (static_cast<size_t>(bh) * splits + split) * (HS + 2);
  if (d < HS) part[2 + d] = A;
  if (d == 0) {
    part[0] = M;
    part[1] = L;
  }
  __threadfence();
  asm volatile("bar.sync 1, %0;" ::"r"(32 * DB_WARPS) : "memory");
  if (threadIdx.x == 0) s_last = atomicAdd(&tickets[bh], 1u) == static_cast<unsigned>(splits - 1);
  asm volatile("bar.sync 1, %0;" ::"r"(32 * DB_WARPS) : "memory");
  if (!s_last) return;
  __threadfence();
  if (d < HS) {
    float MM = -INFINITY;
    for (int sp = 0; sp < splits; ++sp) MM = fmaxf(MM, __ldcg(ws + (static_cast<size_t>(bh) * splits + sp) * (HS + 2)));
    float LL = 0.0f, AA = 0.0f;
    for (int sp = 0; sp < splits; ++sp) {
      const float* p = ws + (static_cast<size_t>(bh) * splits + sp) * (HS + 2);
      const float ms = __ldcg(p);
      const float cw = (ms == -INFINITY) ? 0.0f : exp2f(ms - MM);
      LL += __ldcg(p + 1) * cw;
      AA += __ldcg(p + 2 + d) * cw;
    }
    const float o = AA / LL;
    const __nv_bfloat16 ho = __float2bfloat16_rn(o);
    y[yoff + d] = ho;
    if (y_lo) y_lo[yoff + d] = __float2bfloat16_rn(o - __bfloat162float(ho));
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
