// Linear layers y = x W^T (+ b) with fused epilogues.
//
// nanoGPT's four per-layer Linear layers and the tied lm_head ("nanoGPT 架构分析",
// wangbinyq.github.io, §4.1; "原生 nanoGPT 模型服务首选", §"一个值得做的改进" for the
// fused c_attn split into q|k|v) are the only dense contractions of the decoder.  W is
// kept in nn.Linear's (out_features, in_features) row-major layout, which is already
// K-major for both tensor-core operands.
//
//   bf16 models: gemm_tc_kernel -- tcgen05.mma (kind::f16, M=128, N=BN, fp32 accumulator
//                in TMEM) fed by TMA (128-byte swizzle) through an mbarrier ring;
//                warp-specialised: warp 4 issues TMA, warp 5 issues MMAs and owns TMEM,
//                warps 0-3 run the epilogue (TMEM -> registers -> global).
//   f32 models:  gemm_f32_kernel -- exact fp32 FMA tiles, same epilogues.
//
// Epilogues (rows r are tokens b*T+t, columns n are output features):
//   EPI_F32   out[r, n] = acc + b[n]                   (fp32; lm_head logits, tests)
//   EPI_RESID x[r, n] += acc + b[n]                    (fp32 residual; attn c_proj, mlp c_proj)
//   EPI_GELU  h[r, n]  = gelu_erf(acc + b[n])          (mlp c_fc)
//   EPI_QKV   acc + b[n] split at C and 2C, head h = columns [h*hs, (h+1)*hs) of each part:
//             q -> q[b, h, t, :], k/v -> cache[b, h, pos0+t, :]
//             (the KV-cache append of the sketch, done in place instead of a cat)
//
// HILO: the A operand is given as two bf16 row blocks, hi = bf16(a) (rows 0..M-1) and
// lo = bf16(a - hi) (rows M..2M-1); both are multiplied into the same accumulator, so
// the contraction sees a with ~16 significant bits instead of 8.
//
// Split-K: grid.z CTAs share one output tile; each writes its fp32 partial to a workspace,
// and the last CTA to take a ticket sums the partials in split order (deterministic) and
// runs the epilogue, then resets the ticket.
#pragma once

#include "common.cuh"

namespace kvgpt {

enum EpiKind : int { EPI_F32 = 0, EPI_RESID = 1, EPI_GELU = 2, EPI_QKV = 3 };

template <typename TE>
struct Epi {
  int M = 0, N = 0;               // rows (tokens) and columns (features) of the output
  const float* bias = nullptr;    // [N] or null
  float* x = nullptr;             // EPI_F32 output / EPI_RESID residual, row stride ldx
  int ldx = 0;
  TE* out = nullptr;              // EPI_GELU output, row stride ldo
  TE* out_lo = nullptr;           // optional: also write lo = out - bf16(out) (same layout)
  int ldo = 0;
  TE* q = nullptr;                // EPI_QKV: q [B][nh][T][hs]
  TE* kc = nullptr;               // EPI_QKV: this layer's K cache [B][nh][block][hs]
  TE* vc = nullptr;               //          and V cache
  int C = 0, nh = 0, hs = 64, T = 1, block = 0;
  const int* pos0 = nullptr;      // device cache length before the append (null: 0)
  const int* pos_rows = nullptr;  // or per sequence b: its own cache length (ragged batches)
  KvLayout kv;                    // EPI_QKV: where (b, h, pos) lives in kc / vc
  float* ws = nullptr;            // split-K partials [splits][M][N]
  unsigned int* tickets = nullptr;
  int splits = 1;
  int* err = nullptr;
  // Decode-step kernel only: the activation operand is LayerNorm(ln_x rows) (ln_g, ln_b
  // nullable; row r at ln_x + r * ln_ldx, fp32), computed in the kernel, instead of a bf16 hi/lo
  // operand read by TMA (M <= DL_LN_MAX_ROWS).
  const float* ln_x = nullptr;
  long long ln_ldx = 0;
  const float* ln_g = nullptr;
  const float* ln_b = nullptr;
};

// Apply the epilogue to 16 consecutive columns n0..n0+15 of row r (n0 % 16 == 0).
template <int EPI, typename TE>
__device__ __forceinline__ void epi_apply16(const Epi<TE>& e, int r, int n0, float (&v)[16]) {
  if (r >= e.M || n0 >= e.N) return;
  if (EPI == EPI_F32) {
    float* dst = e.x + static_cast<size_t>(r) * e.ldx + n0;
    if (n0 + 16 <= e.N && (e.ldx & 3) == 0) {
      if (e.bias) {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] += e.bias[n0 + j];
      }
      store16(dst, v);
    } else {
      for (int j = 0; j < 16 && n0 + j < e.N; ++j) dst[j] = v[j] + (e.bias ? e.bias[n0 + j] : 0.0f);
    }
    return;
  }
  if (e.bias) {
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
      float4 b = *reinterpret_cast<const float4*>(e.bias + n0 + j);
      v[j] += b.x;
      v[j + 1] += b.y;
      v[j + 2] += b.z;
      v[j + 3] += b.w;
    }
  }
  if (EPI == EPI_RESID) {
    float* dst = e.x + static_cast<size_t>(r) * e.ldx + n0;
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
      float4 o = reinterpret_cast<const float4*>(dst)[j / 4];
      v[j] += o.x;
      v[j + 1] += o.y;
      v[j + 2] += o.z;
      v[j + 3] += o.w;
    }
    store16(dst, v);
  } else if (EPI == EPI_GELU) {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = gelu_erf(v[j]);
    TE* dst = e.out + static_cast<size_t>(r) * e.ldo + n0;
    store16(dst, v);
    if (e.out_lo) {
      float lo[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) lo[j] = v[j] - to_f32(from_f32<TE>(v[j]));
      store16(e.out_lo + static_cast<size_t>(r) * e.ldo + n0, lo);
    }
  } else if (EPI == EPI_QKV) {
    const int part = n0 / e.C;
    const int hn = n0 - part * e.C;
    const int h = hn / e.hs, d0 = hn - h * e.hs;
    const int b = r / e.T, t = r - b * e.T;
    TE* dst;
    if (part == 0) {
      dst = e.q + ((static_cast<size_t>(b) * e.nh + h) * e.T + t) * e.hs + d0;
    } else {
      const int pos = (e.pos_rows ? e.pos_rows[b] : (e.pos0 ? *e.pos0 : 0)) + t;
      if (pos >= e.block) {
        atomicOr(e.err, ERR_POSITION);
        return;
      }
      TE* base = part == 1 ? e.kc : e.vc;
      dst = base + e.kv.row(b, h, pos) * e.hs + d0;
    }
    store16(dst, v);
  }
}

// ------------------------------------------------------------------ tcgen05 kernel

constexpr int TC_BM = 128;
constexpr int TC_BK = 64;  // bf16 elements in one 128-byte swizzle row
constexpr int TC_THREADS = 192;
constexpr uint32_t TC_A_BYTES = TC_BM * TC_BK * 2;

template <int BN, int STAGES, bool HILO>
struct TcSmem {
  static constexpr int A_TILES = HILO ? 2 : 1;
  static constexpr uint32_t B_BYTES = BN * TC_BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_TILES * TC_A_BYTES + B_BYTES;
  static constexpr uint32_t TILES_BYTES = STAGES * STAGE_BYTES;
  static constexpr uint32_t TOTAL = 1024 /*alignment slack*/ + TILES_BYTES + 256 /*barriers*/;
};

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int BN, int STAGES, bool HILO, int EPI>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int kb_total,
                   int kb_per_split, Epi<__nv_bfloat16> e) {
  using S = TcSmem<BN, STAGES, HILO>;
  static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256 && (BN & (BN - 1)) == 0, "BN: power of two in [32, 256]");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::TILES_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = blockIdx.x, tile_m = blockIdx.y, split = blockIdx.z;
  const int kb0 = split * kb_per_split;
  const int nkb = min(kb_per_split, kb_total - kb0);

  auto a_tile = [&](int s, int h) { return smem + s * S::STAGE_BYTES + h * TC_A_BYTES; };
  auto b_tile = [&](int s) { return smem + s * S::STAGE_BYTES + S::A_TILES * TC_A_BYTES; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES && !mbar_wait(&empty[s], ((i / STAGES) & 1) ^ 1, e.err)) break;
        mbar_arrive_expect_tx(&full[s], S::STAGE_BYTES);
        const int kx = (kb0 + i) * TC_BK;
        tma_load_2d(&tmA, &full[s], a_tile(s, 0), kx, tile_m * TC_BM);
        if (HILO) tma_load_2d(&tmA, &full[s], a_tile(s, 1), kx, e.M + tile_m * TC_BM);
        tma_load_2d(&tmB, &full[s], b_tile(s), kx, tile_n * BN);
        issued = i + 1;
      }
      // Drain: the most recent load into each stage has landed before shared memory is released.
      for (int i = max(0, issued - STAGES); i < issued; ++i) mbar_wait(&full[i % STAGES], (i / STAGES) & 1, e.err);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(TC_BM, BN);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(&full[s], (i / STAGES) & 1, e.err)) break;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < S::A_TILES; ++h) {
          const uint32_t a0 = smem_u32(a_tile(s, h)), b0 = smem_u32(b_tile(s));
#pragma unroll
          for (int k = 0; k < TC_BK / 16; ++k)
            umma_bf16(tmem, sdesc_sw128(a0 + 32 * k), sdesc_sw128(b0 + 32 * k), idesc, (i | h | k) != 0);
        }
        umma_commit(&empty[s]);
      }
      umma_commit(acc_full);
      mbar_wait(acc_full, 0, e.err);  // drain: no MMA in flight when TMEM is released
    }
  } else {
    // Epilogue warps 0..3: warp w owns TMEM lanes 32w..32w+31 (accumulator rows).
    const int row = tile_m * TC_BM + warp * 32 + lane;
    const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const bool ok = mbar_wait(acc_full, 0, e.err);
    tc_fence_after();
    if (e.splits == 1) {
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        tmem_ld16(t_row + c, v);
        if (ok) epi_apply16<EPI>(e, row, tile_n * BN + c, v);
      }
    } else {
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        tmem_ld16(t_row + c, v);
        const int n0 = tile_n * BN + c;
        if (row < e.M && n0 < e.N) store16(e.ws + (static_cast<size_t>(split) * e.M + row) * e.N + n0, v);
      }
      __threadfence();
      epi_bar_sync();
      const unsigned int tile_id = tile_m * gridDim.x + tile_n;
      if (threadIdx.x == 0) s_last = atomicAdd(&e.tickets[tile_id], 1u) == static_cast<unsigned>(e.splits - 1);
      epi_bar_sync();
      if (s_last) {
        __threadfence();
        if (row < e.M) {
          for (int c = 0; c < BN; c += 16) {
            const int n0 = tile_n * BN + c;
            if (n0 >= e.N) break;
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.0f;
            for (int s = 0; s < e.splits; ++s) {
              const float4* p = reinterpret_cast<const float4*>(e.ws + (static_cast<size_t>(s) * e.M + row) * e.N + n0);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                float4 t = __ldcg(p + j);
                v[4 * j] += t.x;
                v[4 * j + 1] += t.y;
                v[4 * j + 2] += t.z;
                v[4 * j + 3] += t.w;
              }
            }
            epi_apply16<EPI>(e, row, n0, v);
          }
        }
        if (threadIdx.x == 0) e.tickets[tile_id] = 0u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, BN);
  }
}

// ------------------------------------------------------------------ persistent tcgen05 kernel

// Persistent form for large M (prefill): one CTA per SM walks the output tiles
// t = blockIdx.x, blockIdx.x + gridDim.x, ... (row-block major, so the CTAs in flight share
// A row blocks in L2).  Two TMEM accumulators of BN columns: the MMA warp fills one while
// the epilogue warps drain the other, so the epilogue's global traffic overlaps the next
// tile's mainloop.  The shared-memory ring's phase runs on across tiles.
// No split-K, no hi/lo operand.
template <int BN, int STAGES>
struct TcPersistSmem {
  static constexpr uint32_t B_BYTES = BN * TC_BK * 2;
  static constexpr uint32_t STAGE_BYTES = TC_A_BYTES + B_BYTES;
  static constexpr uint32_t TILES_BYTES = STAGES * STAGE_BYTES;
  static constexpr uint32_t STAGE_OFFSET = TILES_BYTES + 256;  // after the ring and the barriers
  static constexpr uint32_t TOTAL = 1024 + STAGE_OFFSET + 8 * 32 * 20 * 4;  // + a 32 x 20-float buffer per epilogue warp
};

// The fp32 residual add of one warp's 32 accumulator rows (row0 .. row0+31) over the ncols
// (multiple of 32) columns starting at n0, TMEM column t_warp.  Thread = row in TMEM, so each
// 16-column chunk is restaged through this warp's 32 x 20-float shared buffer: afterwards lane
// l handles rows l/4 + 8i and columns 4*(l%4) .. +3, and the read-modify-write of x goes out
// in 64-byte runs per row.  The residual of the next 32-column group is in flight while this
// group is added.
constexpr int RESID_STAGE_FLOATS = 32 * 20;
constexpr int PERSIST_THREADS = 320;  // warps 0-7 epilogue (two per TMEM lane quadrant), 8 TMA, 9 MMA

__device__ __forceinline__ void persist_resid_warp(const Epi<__nv_bfloat16>& e, int row0, int n0, int ncols,
                                                   uint32_t t_warp, float* stage) {
  const int lane = threadIdx.x & 31;
  const int sr = lane >> 2, sc = (lane & 3) * 4;
  const int G = ncols / 32;
  float4 cur[8], nxt[8];
  auto load = [&](float4 (&dst)[8], int g) {
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = row0 + sr + 8 * i, c = n0 + g * 32 + q * 16 + sc;
        dst[q * 4 + i] = (r < e.M && c < e.N) ? *reinterpret_cast<const float4*>(e.x + static_cast<size_t>(r) * e.ldx + c)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
      }
  };
  load(cur, 0);
#pragma unroll 1
  for (int g = 0; g < G; ++g) {
    if (g + 1 < G) load(nxt, g + 1);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float v[16];
      tmem_ld16(t_warp + g * 32 + q * 16, v);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        reinterpret_cast<float4*>(stage + lane * 20)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = row0 + sr + 8 * i, c = n0 + g * 32 + q * 16 + sc;
        if (r < e.M && c < e.N) {
          const float4 a = *reinterpret_cast<const float4*>(stage + (sr + 8 * i) * 20 + sc);
          const float4 b = e.bias ? *reinterpret_cast<const float4*>(e.bias + c) : make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 o = cur[q * 4 + i];
          *reinterpret_cast<float4*>(e.x + static_cast<size_t>(r) * e.ldx + c) =
              make_float4(a.x + b.x + o.x, a.y + b.y + o.y, a.z + b.z + o.z, a.w + b.w + o.w);
        }
      }
      __syncwarp();
    }
    if (g + 1 < G) {
#pragma unroll
      for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
    }
  }
}

template <int BN, int STAGES, int EPI>
__global__ void __launch_bounds__(PERSIST_THREADS, 1)
    gemm_tc_persistent(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int kb_total,
                       Epi<__nv_bfloat16> e) {
  using S = TcPersistSmem<BN, STAGES>;
  static_assert(2 * BN <= 512, "two accumulators must fit in TMEM");
  constexpr uint32_t TCOLS = 2 * BN <= 256 ? 256 : 512;  // allocation: a power of two
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::TILES_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tm_full = empty + STAGES;   // [2] MMA -> epilogue
  uint64_t* tm_empty = tm_full + 2;     // [2] epilogue -> MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tm_empty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles_n = (e.N + BN - 1) / BN;
  const int n_tiles = ((e.M + TC_BM - 1) / TC_BM) * n_tiles_n;

  auto a_tile = [&](int s) { return smem + s * S::STAGE_BYTES; };
  auto b_tile = [&](int s) { return smem + s * S::STAGE_BYTES + TC_A_BYTES; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tm_full[b], 1);
      mbar_init(&tm_empty[b], 256);
    }
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // A comes from the previous kernel

  if (warp == 8) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        const int m_blk = t / n_tiles_n, n_blk = t - m_blk * n_tiles_n;
        for (int kb = 0; kb < kb_total; ++kb, ++it) {
          const int s = it % STAGES;
          if (it >= STAGES && !mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, e.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], S::STAGE_BYTES);
          tma_load_2d(&tmA, &full[s], a_tile(s), kb * TC_BK, m_blk * TC_BM);
          tma_load_2d(&tmB, &full[s], b_tile(s), kb * TC_BK, n_blk * BN);
        }
      }
      // Drain: the most recent load into each stage has landed before shared memory is released.
      for (int i = max(0, it - STAGES); i < it; ++i) mbar_wait(&full[i % STAGES], (i / STAGES) & 1, e.err);
    }
  } else if (warp == 9) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(TC_BM, BN);
      int it = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++lt) {
        const int buf = lt & 1, use = lt >> 1;
        if (use > 0 && !mbar_wait(&tm_empty[buf], (use & 1) ^ 1, e.err)) break;
        tc_fence_after();
        const uint32_t acc = tmem + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < kb_total; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&full[s], (it / STAGES) & 1, e.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(a_tile(s)), b0 = smem_u32(b_tile(s));
#pragma unroll
          for (int k = 0; k < TC_BK / 16; ++k)
            umma_bf16(acc, sdesc_sw128(a0 + 32 * k), sdesc_sw128(b0 + 32 * k), idesc, (kb | k) != 0);
          umma_commit(&empty[s]);
        }
        umma_commit(&tm_full[buf]);
      }
    }
  } else {
    // Epilogue warps 0..7: warp w owns TMEM lanes 32(w%4) .. +31 (accumulator rows) and
    // columns [(w/4) BN/2, (w/4 + 1) BN/2) of the tile.
    const int quad = warp & 3, half = warp >> 2;
    constexpr int HALF = BN / 2;
    int lt = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++lt) {
      const int m_blk = t / n_tiles_n, n_blk = t - m_blk * n_tiles_n;
      const int buf = lt & 1, use = lt >> 1;
      const bool ok = mbar_wait(&tm_full[buf], use & 1, e.err);
      tc_fence_after();
      const int row = m_blk * TC_BM + quad * 32 + lane;
      const uint32_t t_row =
          tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(buf * BN + half * HALF);
      if (EPI == EPI_RESID && ok) {
        persist_resid_warp(e, m_blk * TC_BM + quad * 32, n_blk * BN + half * HALF, HALF, t_row,
                           reinterpret_cast<float*>(smem + S::STAGE_OFFSET) + warp * RESID_STAGE_FLOATS);
      } else {
#pragma unroll 1
        for (int c = 0; c < HALF; c += 16) {
          float v[16];
          tmem_ld16(t_row + c, v);
          if (ok) epi_apply16<EPI>(e, row, n_blk * BN + half * HALF + c, v);
        }
      }
      tc_fence_before();
      mbar_arrive(&tm_empty[buf]);
      if (!ok) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, TCOLS);
  }
}

// ------------------------------------------------------------------ fp32 kernel

// 64x64 output tile, 256 threads, 4x4 outputs per thread, K in steps of 16.
// Produces 16-column chunks through the same epilogue (each thread row-group owns them).
constexpr int F32_BM = 64, F32_BN = 64, F32_BK = 16;

template <int EPI>
__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, const float* __restrict__ W, int K,
                                                        Epi<float> e) {
  __shared__ float As[F32_BK][F32_BM + 4];
  __shared__ float Ws[F32_BK][F32_BN + 4];
  __shared__ float Cs[F32_BM][F32_BN + 1];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * F32_BM, n0 = blockIdx.x * F32_BN;
  const int tr = tid / 16, tc = tid % 16;  // 16 x 16 threads, 4 x 4 each
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += F32_BK) {
    for (int i = tid; i < F32_BM * F32_BK; i += 256) {
      const int r = i / F32_BK, k = i % F32_BK;
      As[k][r] = (m0 + r < e.M && k0 + k < K) ? A[static_cast<size_t>(m0 + r) * K + k0 + k] : 0.0f;
      Ws[k][r] = (n0 + r < e.N && k0 + k < K) ? W[static_cast<size_t>(n0 + r) * K + k0 + k] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < F32_BK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[k][tr * 4 + i];
        b[i] = Ws[k][tc * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) Cs[tr * 4 + i][tc * 4 + j] = acc[i][j];
  __syncthreads();
  // 64 rows x 4 chunks of 16 columns = 256 (row, chunk) pairs, one per thread.
  const int r = tid / 4, c = (tid % 4) * 16;
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = Cs[r][c + j];
  epi_apply16<EPI>(e, m0 + r, n0 + c, v);
}

}  // namespace kvgpt
