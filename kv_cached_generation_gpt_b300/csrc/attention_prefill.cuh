// Causal prefill attention on the Blackwell tensor core (head size 64, bf16).
//
// Definition ("极速上手nanoGPT", deepseek.csdn.net, §"注意力机制"; "第 4 章 模型构建",
// aiknowledge.cn, §4.5 causal mask): y = softmax(q k^T / sqrt(hs) + mask) v, where the
// query at absolute position p sees keys 0..p; a chunk appended to a cache of length pos0
// ("原生 nanoGPT 模型服务首选", §"一个值得做的改进") sits at positions pos0 .. pos0+T-1.
// Layouts as in attention.cuh: q [B][nh][T][64], cache rows through KvLayout, y [B*T][C].
#pragma once

#include "attention.cuh"
#include "common.cuh"

namespace kvgpt {

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

}  // namespace kvgpt
