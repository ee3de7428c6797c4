// Linear layers of a decode step: out[b, n] = sum_k a[b, k] W[n, k] (+ fused epilogue) for
// up to 128 new tokens b, with the activation given as a hi/lo pair of bf16 rows
// (a = hi + lo; hi rows 0..M-1, lo rows M..2M-1).
//
// These are the same four per-layer Linear layers and the tied lm_head as in gemm.cuh
// ("nanoGPT 架构分析", wangbinyq.github.io, §4.1), at the shapes a KV-cached step gives them:
// one new row per sequence ("原生 nanoGPT 模型服务首选", §"一个值得做的改进": only the new
// token is fed), so the work is a stream over the weights with very few rows.
//
// Swap-AB on tcgen05: the weight rows (output features) are the MMA's M = 128 side and the
// token rows its N side, hi rows then lo rows (N = 2 * Bp, Bp = M rounded up to 8).  One
// 128-feature tile is split along K across the S CTAs of a thread-block cluster (S <= 16).
// CTA r owns features [r*128/S, (r+1)*128/S) of the tile.  TMEM lane f holds feature f for
// every token row; the thread reading it adds the hi and lo halves and stores the column
// straight into the owner's shared memory (st.async, counted on the owner's mbarrier; its own
// slice with plain stores), once a cluster barrier has shown that every CTA's MMAs are done
// with the ring the receive slots overlay.  The owner sums the S slices in split order -- a
// fixed order, so results do not depend on timing -- and applies the epilogue.  No global
// scratch is used.
//
// Programmatic dependent launch: weight tiles do not depend on earlier kernels, so they are
// requested before griddepcontrol.wait; activations, residual and outputs come after it.
//
// Up to 8 token rows, the LayerNorm before c_attn, c_fc and the lm_head runs inside this
// kernel: every CTA reads the whole fp32 rows (a few KiB), takes their statistics exactly as
// layernorm_kernel does, and writes its K-slice of LN(x) as the bf16 hi/lo operand straight
// into the swizzled shared-memory tile the MMA reads, so no LayerNorm launch is needed.
#pragma once

#include "common.cuh"
#include "gemm.cuh"
#include "norm.cuh"

namespace kvgpt {

constexpr int DL_THREADS = 192;  // warps 0-3: TMEM -> partial; warp 4: TMA; warp 5: MMA; all: reduce
constexpr int DL_MAX_STAGES = 3;
constexpr int DL_MAX_ROWS = 128;
constexpr int DL_MAX_SPLITS = 16;
constexpr int DL_LN_MAX_ROWS = 8;   // in-kernel LayerNorm operand up to this many token rows
constexpr uint32_t DL_W_BYTES = 128u * TC_BK * 2u;

__host__ __device__ constexpr int dl_bp(int rows) { return (rows + 7) & ~7; }
__host__ __device__ constexpr uint32_t dl_stage_bytes(int bp) { return DL_W_BYTES + 2u * bp * 128u; }
// Once the MMAs are done the ring holds the receive slots: [S][R][bp] floats (sender, feature
// of the owner's slice, token row), bp x 128 floats in all.  Within a column the 16-byte
// chunks of 4 rows are XOR-swizzled by the feature (dl_chunk), so that the stores of 8
// consecutive features fall in distinct banks, and the reduce's reads (a warp covers a few
// rows x several 8-feature groups) conflict at most 2-way.
__host__ __device__ constexpr uint32_t dl_recv_bytes(int bp) { return static_cast<uint32_t>(bp * 512); }
__host__ __device__ constexpr uint32_t dl_ring_bytes(int bp, int stages) {
  return stages * dl_stage_bytes(bp) > dl_recv_bytes(bp) ? stages * dl_stage_bytes(bp) : dl_recv_bytes(bp);
}
__host__ __device__ constexpr uint32_t dl_smem_bytes(int bp, int stages) {
  return 1024u + dl_ring_bytes(bp, stages) + 256u;
}

// Position of 4-row chunk q in the receive column of feature fr: q ^ ((fr ^ fr / 8) mod g), g
// the largest power of two <= 8 dividing the chunk count bp / 4 (so the swizzle stays inside
// the column).
__device__ __forceinline__ int dl_chunk(int q, int fr, int bp) {
  const int n = bp >> 2;
  return q ^ ((fr ^ (fr >> 3)) & (min(8, n & -n) - 1));
}

// Apply the epilogue to 8 consecutive features n0..n0+7 of token row r (n0 % 8 == 0); qpos is
// the position of the new token (EPI_QKV).
template <int EPI>
__device__ __forceinline__ void dl_epilogue8(const Epi<__nv_bfloat16>& e, int r, int n0, float (&v)[8], int qpos) {
  if (EPI == EPI_F32) {
    float* dst = e.x + static_cast<size_t>(r) * e.ldx + n0;
    if (n0 + 8 <= e.N && (e.ldx & 3) == 0) {
      if (e.bias) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] += e.bias[n0 + j];
      }
      reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      for (int j = 0; j < 8 && n0 + j < e.N; ++j) dst[j] = v[j] + (e.bias ? e.bias[n0 + j] : 0.0f);
    }
    return;
  }
  if (e.bias) {
    const float4 b0 = reinterpret_cast<const float4*>(e.bias + n0)[0];
    const float4 b1 = reinterpret_cast<const float4*>(e.bias + n0)[1];
    v[0] += b0.x; v[1] += b0.y; v[2] += b0.z; v[3] += b0.w;
    v[4] += b1.x; v[5] += b1.y; v[6] += b1.z; v[7] += b1.w;
  }
  if (EPI == EPI_RESID) {
    float4* dst = reinterpret_cast<float4*>(e.x + static_cast<size_t>(r) * e.ldx + n0);
    const float4 o0 = dst[0], o1 = dst[1];
    dst[0] = make_float4(v[0] + o0.x, v[1] + o0.y, v[2] + o0.z, v[3] + o0.w);
    dst[1] = make_float4(v[4] + o1.x, v[5] + o1.y, v[6] + o1.z, v[7] + o1.w);
  } else if (EPI == EPI_GELU) {
    uint4 hi, lo;
    float g[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) g[j] = gelu_erf(v[j]);
    hi.x = pack_bf16x2(g[0], g[1]);
    hi.y = pack_bf16x2(g[2], g[3]);
    hi.z = pack_bf16x2(g[4], g[5]);
    hi.w = pack_bf16x2(g[6], g[7]);
    const size_t off = static_cast<size_t>(r) * e.ldo + n0;
    *reinterpret_cast<uint4*>(e.out + off) = hi;
    if (e.out_lo) {
      const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&hi);
      float l[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) l[j] = g[j] - __bfloat162float(h[j]);
      lo.x = pack_bf16x2(l[0], l[1]);
      lo.y = pack_bf16x2(l[2], l[3]);
      lo.z = pack_bf16x2(l[4], l[5]);
      lo.w = pack_bf16x2(l[6], l[7]);
      *reinterpret_cast<uint4*>(e.out_lo + off) = lo;
    }
  } else if (EPI == EPI_QKV) {
    // one new token per sequence: row r is sequence r, at position *pos0
    const int part = n0 / e.C;
    const int hn = n0 - part * e.C;
    const int h = hn / e.hs, d0 = hn - h * e.hs;
    __nv_bfloat16* dst;
    if (part == 0) {
      dst = e.q + (static_cast<size_t>(r) * e.nh + h) * e.hs + d0;
    } else {
      const int pos = e.pos_rows ? e.pos_rows[r] : qpos;  // the cache length before this token
      if (pos >= e.block) {
        atomicOr(e.err, ERR_POSITION);
        return;
      }
      __nv_bfloat16* base = part == 1 ? e.kc : e.vc;
      dst = base + e.kv.row(r, h, pos) * e.hs + d0;
    }
    uint4 o;
    o.x = pack_bf16x2(v[0], v[1]);
    o.y = pack_bf16x2(v[2], v[3]);
    o.z = pack_bf16x2(v[4], v[5]);
    o.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(dst) = o;
  }
}

// Bring the global operands of dl_epilogue8 for (row r, features n0..n0+7) that earlier kernels
// write into L1 (the bias is fetched at the start).
template <int EPI>
__device__ __forceinline__ void dl_prefetch_epilogue(const Epi<__nv_bfloat16>& e, int r, int n0) {
  if (EPI == EPI_RESID) prefetch_l1(e.x + static_cast<size_t>(r) * e.ldx + n0);
  if (EPI == EPI_QKV && e.pos_rows) prefetch_l1(e.pos_rows + r);
}

// grid.x = n_tiles * splits, cluster (splits, 1, 1); CTA rank r of cluster c works on
// feature tile c and k-blocks [r*kb_total/splits, (r+1)*kb_total/splits) (splits <= kb_total),
// through a ring of `stages` (1..3) shared-memory stages.
// e.M = token rows (<= 128), e.N = output features.
template <int EPI>
__global__ void __launch_bounds__(DL_THREADS) dec_linear_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                 const __grid_constant__ CUtensorMap tmX,
                                                                 int kb_total, int splits, int stages,
                                                                 Epi<__nv_bfloat16> e) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int bp = dl_bp(e.M);
  const uint32_t stage_bytes = dl_stage_bytes(bp);
  const uint32_t x_bytes = 2u * bp * 128u;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + dl_ring_bytes(bp, stages));
  uint64_t* empty = full + DL_MAX_STAGES;
  uint64_t* acc_full = empty + DL_MAX_STAGES;
  uint64_t* recv_full = acc_full + 1;
  uint64_t* x_full = recv_full + 1;  // [DL_MAX_STAGES]: operand written by warps 0-3 (LayerNorm)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(x_full + DL_MAX_STAGES);
  const bool lnx = e.ln_x != nullptr;  // callers pass LayerNorm inputs only for M <= DL_LN_MAX_ROWS
  __shared__ float s_mean[DL_LN_MAX_ROWS], s_rstd[DL_LN_MAX_ROWS];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = splits > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int tile = blockIdx.x / splits;
  const int kb0 = (rank * kb_total) / splits, kb1 = ((rank + 1) * kb_total) / splits;
  const int nkb = kb1 - kb0;
  const int R = 128 / splits;                  // features owned by each CTA of the cluster
  const uint32_t slice_bytes = static_cast<uint32_t>(bp * R * 4);
  float* recv = reinterpret_cast<float*>(smem);  // [S][R][bp], over the ring
  uint32_t tcols = 32;
  while (tcols < static_cast<uint32_t>(2 * bp)) tcols <<= 1;

  // the bias of this CTA's R features does not depend on earlier kernels: into L1 now
  if (e.bias && threadIdx.x * 32 < R && tile * 128 + rank * R + static_cast<int>(threadIdx.x) * 32 < e.N)
    prefetch_l1(e.bias + tile * 128 + rank * R + threadIdx.x * 32);

  auto w_tile = [&](int s) { return smem + s * stage_bytes; };
  auto x_tile = [&](int s) { return smem + s * stage_bytes + DL_W_BYTES; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(recv_full, 1);
    for (int s = 0; s < stages; ++s) mbar_init(&x_full[s], 128);
    fence_mbar_init();
    // the S - 1 peers' slices for this CTA complete on recv_full
    if (splits > 1) mbar_arrive_expect_tx(recv_full, static_cast<uint32_t>(splits - 1) * slice_bytes);
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch();  // this CTA holds its TMEM: the next kernel may begin its own prologue

  if (warp == 4) {
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      const int pre = min(nkb, stages);
      const uint32_t tx = lnx ? DL_W_BYTES : DL_W_BYTES + x_bytes;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], tx);
        tma_load_2d(&tmW, &full[i], w_tile(i), (kb0 + i) * TC_BK, tile * 128);
      }
      griddep_wait();  // activations come from the previous kernel
      if (!lnx) {
        for (int i = 0; i < pre; ++i) {
          tma_load_2d(&tmX, &full[i], x_tile(i), (kb0 + i) * TC_BK, 0);
          tma_load_2d(&tmX, &full[i], x_tile(i) + bp * 128, (kb0 + i) * TC_BK, e.M);
        }
      }
      int issued = pre;
      for (int i = pre; i < nkb; ++i) {
        const int s = i % stages;
        if (!mbar_wait(&empty[s], ((i / stages) & 1) ^ 1, e.err)) break;
        mbar_arrive_expect_tx(&full[s], tx);
        const int kx = (kb0 + i) * TC_BK;
        tma_load_2d(&tmW, &full[s], w_tile(s), kx, tile * 128);
        if (!lnx) {
          tma_load_2d(&tmX, &full[s], x_tile(s), kx, 0);
          tma_load_2d(&tmX, &full[s], x_tile(s) + bp * 128, kx, e.M);
        }
        issued = i + 1;
      }
      // Drain: the most recent load into each stage has landed before shared memory is reused.
      for (int i = max(0, issued - stages); i < issued; ++i) mbar_wait(&full[i % stages], (i / stages) & 1, e.err);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 2 * bp);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % stages;
        if (!mbar_wait(&full[s], (i / stages) & 1, e.err)) break;
        if (lnx && !mbar_wait(&x_full[s], (i / stages) & 1, e.err)) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(w_tile(s)), b0 = smem_u32(x_tile(s));
#pragma unroll
        for (int k = 0; k < TC_BK / 16; ++k)
          umma_bf16(tmem, sdesc_sw128(a0 + 32 * k), sdesc_sw128(b0 + 32 * k), idesc, (i | k) != 0);
        umma_commit(&empty[s]);
      }
      umma_commit(acc_full);
      mbar_wait(acc_full, 0, e.err);  // no MMA in flight once this returns
    }
  } else {
    if (lnx) {
      // Warps 0-3 first build the operand: LayerNorm statistics of every token row (warp w
      // takes rows w, w+4: lanes hold column pairs i*64 + 2*lane, as layernorm_kernel does) ...
      griddep_wait();  // the residual rows come from the previous kernel
      const int C = kb_total * TC_BK;
      const int np = C / 64;
      for (int r = warp; r < e.M; r += 4) {
        const float* xr = e.ln_x + r * e.ln_ldx;
        float2 v[LN_MAX_PAIRS];
#pragma unroll
        for (int i = 0; i < LN_MAX_PAIRS; ++i)
          if (i < np) v[i] = *reinterpret_cast<const float2*>(xr + i * 64 + lane * 2);
        float sm = 0.0f;
#pragma unroll
        for (int i = 0; i < LN_MAX_PAIRS; ++i)
          if (i < np) sm += v[i].x + v[i].y;
        const float mean = warp_sum(sm) / static_cast<float>(C);
        float q = 0.0f;
#pragma unroll
        for (int i = 0; i < LN_MAX_PAIRS; ++i) {
          if (i < np) {
            const float a = v[i].x - mean, b = v[i].y - mean;
            q += a * a + b * b;
          }
        }
        const float var = warp_sum(q) / static_cast<float>(C);
        if (lane == 0) {
          s_mean[r] = mean;
          s_rstd[r] = 1.0f / sqrtf(var + 1e-5f);
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      // ... then, per k-block, its 64 columns of LN(x) as hi (rows 0..bp-1) and lo (rows
      // bp..2bp-1) in the 128-byte-swizzled layout a TMA load would have written.
      // Thread t writes the 8-column piece c = t % 8 of row t / 8 (rows past e.M are zeros).
      const int tid = threadIdx.x;
      const int c = tid & 7;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % stages;
        if (i >= stages && !mbar_wait(&empty[s], ((i / stages) & 1) ^ 1, e.err)) break;
        const uint32_t xt = smem_u32(x_tile(s));
        const int k = (kb0 + i) * TC_BK + c * 8;
        float gm[8], bt[8];
        {
          const float4 g0 = reinterpret_cast<const float4*>(e.ln_g + k)[0];
          const float4 g1 = reinterpret_cast<const float4*>(e.ln_g + k)[1];
          gm[0] = g0.x; gm[1] = g0.y; gm[2] = g0.z; gm[3] = g0.w;
          gm[4] = g1.x; gm[5] = g1.y; gm[6] = g1.z; gm[7] = g1.w;
          float4 b0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), b1 = b0;
          if (e.ln_b) {
            b0 = reinterpret_cast<const float4*>(e.ln_b + k)[0];
            b1 = reinterpret_cast<const float4*>(e.ln_b + k)[1];
          }
          bt[0] = b0.x; bt[1] = b0.y; bt[2] = b0.z; bt[3] = b0.w;
          bt[4] = b1.x; bt[5] = b1.y; bt[6] = b1.z; bt[7] = b1.w;
        }
        const int r = tid >> 3;
        if (r < bp) {  // bp <= DL_LN_MAX_ROWS: one row per thread
          uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
          if (r < e.M) {
            const float4* xp = reinterpret_cast<const float4*>(e.ln_x + static_cast<size_t>(r) * e.ln_ldx + k);
            const float4 x0 = xp[0], x1 = xp[1];
            float y[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const float mean = s_mean[r], rstd = s_rstd[r];
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] = (y[j] - mean) * rstd * gm[j] + bt[j];
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const __nv_bfloat162 h = __floats2bfloat162_rn(y[2 * j], y[2 * j + 1]);
              const float2 hf = __bfloat1622float2(h);
              hw[j] = *reinterpret_cast<const uint32_t*>(&h);
              lw[j] = pack_bf16x2(y[2 * j] - hf.x, y[2 * j + 1] - hf.y);
            }
            hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
          const uint32_t off_hi = static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
          const uint32_t off_lo = static_cast<uint32_t>((bp + r) * 128 + ((c ^ (r & 7)) << 4));  // bp % 8 == 0
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(xt + off_hi), "r"(hi.x), "r"(hi.y), "r"(hi.z),
                       "r"(hi.w)
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(xt + off_lo), "r"(lo.x), "r"(lo.y), "r"(lo.z),
                       "r"(lo.w)
                       : "memory");
        }
        fence_proxy_async_smem();  // the MMA reads the operand through the async proxy
        mbar_arrive(&x_full[s]);
      }
    }
    // Warps 0-3: TMEM lane f = feature f of the tile, for token rows 0..bp-1 (hi columns, then
    // lo).  The column goes to recv[rank][f % R][:] of owner o = f / R.
    const bool ok = mbar_wait(acc_full, 0, e.err);
    tc_fence_after();
    // This CTA's MMAs are done: its ring may take the peers' slices.  The wait below overlaps
    // the first TMEM load.
    if (splits > 1) cluster_arrive();
    const int f = warp * 32 + lane;
    const uint32_t o = static_cast<uint32_t>(f / R);
    const int fr = f % R;
    const uint32_t col = smem_u32(recv + (rank * R + fr) * bp);
    const uint32_t dst = splits > 1 ? mapa_shared(col, o) : col;
    const uint32_t bar = splits > 1 ? mapa_shared(smem_u32(recv_full), o) : 0u;
    const bool local = static_cast<int>(o) == rank;
    const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
    for (int c = 0; c < bp; c += 16) {
      uint32_t hi[16], lo[16];
      const bool two = c + 8 < bp;  // bp is a multiple of 8: 16 columns, or the last 8
      if (two) {
        tmem_ld16_raw(t_row + c, hi);
        tmem_ld16_raw(t_row + bp + c, lo);
      } else {
        tmem_ld8_raw(t_row + c, hi);
        tmem_ld8_raw(t_row + bp + c, lo);
      }
      tmem_wait_ld16(hi, lo);
      if (c == 0 && splits > 1) cluster_wait();  // every CTA of the cluster is past its MMAs
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = ok ? __uint_as_float(hi[j]) + __uint_as_float(lo[j]) : 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q < 2 || two) {
          const uint32_t a = dst + static_cast<uint32_t>(dl_chunk((c >> 2) + q, fr, bp) * 16);
          if (local)
            st_shared_f4(a, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          else
            st_async_f4(a, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3], bar);
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  if (splits > 1 && warp >= 4) cluster_sync();  // warps 0-3 met the barrier before sending
  __syncthreads();                              // this CTA's own slice is written

  // Reduce: this CTA's R features of the tile, for every token row, in split order.  Unit u
  // is token row u / (R/8) and features fl .. fl+7, fl = 8 (u mod R/8): consecutive threads
  // cover consecutive features of a row, so the epilogue's stores coalesce.  Its global
  // operands are fetched into L1 while the peers' slices are still arriving.
  griddep_wait();
  const int upr = R / 8;
  const int units = e.M * upr;
#pragma unroll 1
  for (int u = threadIdx.x; u < units; u += DL_THREADS) {
    const int r = u / upr, fl = (u - r * upr) * 8;
    const int n0 = tile * 128 + rank * R + fl;
    if (n0 < e.N) dl_prefetch_epilogue<EPI>(e, r, n0);
  }
  int qpos = 0;
  if (EPI == EPI_QKV && e.pos0) qpos = *e.pos0;
  if (splits > 1) mbar_wait(recv_full, 0, e.err);
#pragma unroll 1
  for (int u = threadIdx.x; u < units; u += DL_THREADS) {
    const int r = u / upr, fl = (u - r * upr) * 8;
    const int n0 = tile * 128 + rank * R + fl;
    if (n0 >= e.N) continue;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.0f;
#pragma unroll 1
    for (int s = 0; s < splits; ++s) {
      const float* src = recv + (s * R + fl) * bp + (r & 3);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] += src[j * bp + 4 * dl_chunk(r >> 2, fl + j, bp)];
    }
    dl_epilogue8<EPI>(e, r, n0, v, qpos);
  }
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

}  // namespace kvgpt
