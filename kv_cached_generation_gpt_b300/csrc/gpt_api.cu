// libgpt_b300: runtime and C ABI for KV-cached GPT-2 generation on sm_103a.
//
// One model = library-owned weights (nn.Linear layout), a contiguous KV cache
// [layer][k|v][batch][head][position][64], activation buffers sized for max_batch x
// block_size tokens, a device error word and a device-resident cache length.
//
// A forward pass over B x T new tokens (prefill: T = prompt length from an empty cache;
// decode: T = 1 at position = cache length) enqueues:
//   embed -> per layer [ln_1 -> c_attn GEMM (+ KV append) -> attention -> c_proj GEMM
//   (+ residual) -> ln_2 -> c_fc GEMM (+ GELU) -> mlp c_proj GEMM (+ residual)] ->
//   ln_f on each sequence's last position -> lm_head GEMM (tied wte) -> fp32 logits
// ("nanoGPT 架构分析", wangbinyq.github.io, §4.1; "原生 nanoGPT 模型服务首选", §"一个值得做的改进").
// gpt_generate captures one decode step plus its draw as a CUDA graph and replays it.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <atomic>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/gpt.h"
#include "attention.cuh"
#include "attention_prefill.cuh"
#include "common.cuh"
#include "decode_linear.cuh"
#include "gemm.cuh"
#include "norm.cuh"
#include "sampler.cuh"

using namespace kvgpt;
using bf16 = __nv_bfloat16;

namespace {

thread_local std::string g_detail;

// gpt_create_paged's request, read by gpt_create on the same thread
struct PagedRequest {
  bool paged = false;
  int page_size = 0, n_pages = 0;
};
thread_local PagedRequest g_paged_request;

// Failure injection for tests (gpt_debug_fail_allocation): when positive, the allocation that
// brings it to zero fails as if the device were out of memory.
std::atomic<int> g_fail_alloc_countdown{0};

bool fail_this_allocation() {
  int c = g_fail_alloc_countdown.load();
  while (c > 0) {
    if (g_fail_alloc_countdown.compare_exchange_weak(c, c - 1)) return c == 1;
  }
  return false;
}

int cuda_fail(cudaError_t e, const char* what) {
  g_detail = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return e == cudaErrorMemoryAllocation ? GPT_ENOMEM : GPT_ECUDA;
}

#define CK(call)                                                        \
  do {                                                                  \
    cudaError_t e_ = (call);                                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);                 \
  } while (0)

inline int cdiv(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// ------------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encode() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// Row-major bf16 matrix [rows][cols] read in boxes of box_rows x 64 with 128-byte swizzle.
int make_tmap(CUtensorMap* map, const void* ptr, long long rows, long long cols, int box_rows) {
  if (!load_encode()) {
    g_detail = "cuTensorMapEncodeTiled unavailable";
    return GPT_EUNSUPPORTED;
  }
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(TC_BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_detail = "cuTensorMapEncodeTiled failed (" + std::to_string(static_cast<int>(r)) + ")";
    return GPT_ECUDA;
  }
  return GPT_OK;
}

// ------------------------------------------------------------------ GEMM launch

unsigned long long g_attr_mask[64] = {};  // per kernel slot: devices whose smem attribute is set
std::mutex g_attr_mu;

constexpr int TC_STAGES = 4;

template <int BN, bool HILO, int EPI>
cudaError_t attr_tc(int slot, int dev) {
  using S = TcSmem<BN, TC_STAGES, HILO>;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (!(g_attr_mask[slot] & (1ull << dev))) {
    cudaError_t r = cudaFuncSetAttribute(gemm_tc_kernel<BN, TC_STAGES, HILO, EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::TOTAL);
    if (r != cudaSuccess) return r;
    g_attr_mask[slot] |= 1ull << dev;
  }
  return cudaSuccess;
}

template <int BN, bool HILO, int EPI>
cudaError_t launch_tc(int slot, int dev, const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K,
                      int splits, const Epi<bf16>& e, cudaStream_t st) {
  constexpr int STAGES = TC_STAGES;
  using S = TcSmem<BN, STAGES, HILO>;
  auto kern = gemm_tc_kernel<BN, STAGES, HILO, EPI>;
  cudaError_t r = attr_tc<BN, HILO, EPI>(slot, dev);
  if (r != cudaSuccess) return r;
  const int kb = K / TC_BK;
  const int kbps = cdiv(kb, splits);
  dim3 grid(cdiv(N, BN), cdiv(M, TC_BM), splits);
  kern<<<grid, TC_THREADS, S::TOTAL, st>>>(ta, tb, kb, kbps, e);
  return cudaGetLastError();
}

cudaError_t dispatch_tc(int bn, bool hilo, int epi, int dev, const CUtensorMap& ta, const CUtensorMap& tb, int M,
                        int N, int K, int splits, const Epi<bf16>& e, cudaStream_t st) {
#define KVGPT_TC_CASE(BN, H, E, SLOT) \
  if (bn == BN && hilo == H && epi == E) return launch_tc<BN, H, E>(SLOT, dev, ta, tb, M, N, K, splits, e, st);
  KVGPT_TC_CASE(64, false, EPI_F32, 0)
  KVGPT_TC_CASE(64, false, EPI_RESID, 1)
  KVGPT_TC_CASE(64, false, EPI_GELU, 2)
  KVGPT_TC_CASE(64, false, EPI_QKV, 3)
  KVGPT_TC_CASE(64, true, EPI_F32, 4)
  KVGPT_TC_CASE(64, true, EPI_RESID, 5)
  KVGPT_TC_CASE(64, true, EPI_GELU, 6)
  KVGPT_TC_CASE(64, true, EPI_QKV, 7)
  KVGPT_TC_CASE(128, false, EPI_F32, 8)
  KVGPT_TC_CASE(128, false, EPI_RESID, 9)
  KVGPT_TC_CASE(128, false, EPI_GELU, 10)
  KVGPT_TC_CASE(128, false, EPI_QKV, 11)
  KVGPT_TC_CASE(128, true, EPI_F32, 12)
  KVGPT_TC_CASE(128, true, EPI_RESID, 13)
  KVGPT_TC_CASE(128, true, EPI_GELU, 14)
  KVGPT_TC_CASE(128, true, EPI_QKV, 15)
  KVGPT_TC_CASE(256, false, EPI_F32, 16)
  KVGPT_TC_CASE(256, false, EPI_RESID, 17)
  KVGPT_TC_CASE(256, false, EPI_GELU, 18)
  KVGPT_TC_CASE(256, false, EPI_QKV, 19)
#undef KVGPT_TC_CASE
  return cudaErrorInvalidValue;
}

// Persistent prefill GEMMs: BN 256 with 4 stages or BN 128 with 6 (192 KiB of ring either way).
template <int BN>
constexpr int persist_stages() {
  return BN == 256 ? 4 : BN == 192 ? 5 : 6;
}

// Tile width of a persistent GEMM: among 256, 192 and 128 (dividing N), the one whose tile
// count fills the last wave of num_sms CTAs best (ties: the wider tile); 0 if none applies
// or there are fewer tiles than SMs.
int persist_bn(int M, int N, int num_sms) {
  int best = 0;
  double best_eff = 0.0;
  for (int bn : {256, 192, 128}) {
    if (N % bn != 0) continue;
    const long long tiles = static_cast<long long>(cdiv(M, TC_BM)) * (N / bn);
    if (tiles < num_sms) continue;
    const double eff = static_cast<double>(tiles) / (static_cast<double>(cdiv(tiles, num_sms)) * num_sms);
    if (eff > best_eff + 1e-3) {
      best = bn;
      best_eff = eff;
    }
  }
  return best;
}

template <int BN, int EPI>
cudaError_t attr_persist() {
  using S = TcPersistSmem<BN, persist_stages<BN>()>;
  return cudaFuncSetAttribute(gemm_tc_persistent<BN, persist_stages<BN>(), EPI>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, S::TOTAL);
}

cudaError_t init_persist_attrs_once();

cudaError_t init_persist_attrs() {
  cudaError_t r;
  if ((r = attr_persist<256, EPI_F32>()) != cudaSuccess) return r;
  if ((r = attr_persist<256, EPI_RESID>()) != cudaSuccess) return r;
  if ((r = attr_persist<256, EPI_GELU>()) != cudaSuccess) return r;
  if ((r = attr_persist<256, EPI_QKV>()) != cudaSuccess) return r;
  if ((r = attr_persist<192, EPI_F32>()) != cudaSuccess) return r;
  if ((r = attr_persist<192, EPI_RESID>()) != cudaSuccess) return r;
  if ((r = attr_persist<192, EPI_GELU>()) != cudaSuccess) return r;
  if ((r = attr_persist<192, EPI_QKV>()) != cudaSuccess) return r;
  if ((r = attr_persist<128, EPI_F32>()) != cudaSuccess) return r;
  if ((r = attr_persist<128, EPI_RESID>()) != cudaSuccess) return r;
  if ((r = attr_persist<128, EPI_GELU>()) != cudaSuccess) return r;
  return attr_persist<128, EPI_QKV>();
}

// Once per device (the stand-alone operations have no gpt_create to do it).
cudaError_t init_persist_attrs_once() {
  static unsigned long long mask = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t r = cudaGetDevice(&dev);
  if (r != cudaSuccess) return r;
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 64 && (mask & (1ull << dev))) return cudaSuccess;
  if ((r = init_persist_attrs()) != cudaSuccess) return r;
  if (dev < 64) mask |= 1ull << dev;
  return cudaSuccess;
}

// The tcgen05 prefill attention's shared-memory limit, once per device (for the stand-alone
// operation; gpt_create sets it with the other kernels').
cudaError_t init_attn_tc_once() {
  static unsigned long long mask = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t r = cudaGetDevice(&dev);
  if (r != cudaSuccess) return r;
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 64 && (mask & (1ull << dev))) return cudaSuccess;
  r = cudaFuncSetAttribute(attn_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(PT_SMEM));
  if (r != cudaSuccess) return r;
  if (dev < 64) mask |= 1ull << dev;
  return cudaSuccess;
}

template <int BN, int EPI>
cudaError_t launch_persist_epi(const CUtensorMap& ta, const CUtensorMap& tb, int K, int grid, const Epi<bf16>& e,
                               cudaStream_t st) {
  constexpr int STAGES = persist_stages<BN>();
  using S = TcPersistSmem<BN, STAGES>;
  gemm_tc_persistent<BN, STAGES, EPI><<<grid, PERSIST_THREADS, S::TOTAL, st>>>(ta, tb, K / TC_BK, e);
  return cudaGetLastError();
}

cudaError_t launch_persist(int bn, int epi, const CUtensorMap& ta, const CUtensorMap& tb, int K, int grid,
                           const Epi<bf16>& e, cudaStream_t st) {
#define KVGPT_PERSIST_CASE(BN, E) \
  if (bn == BN && epi == E) return launch_persist_epi<BN, E>(ta, tb, K, grid, e, st);
  KVGPT_PERSIST_CASE(256, EPI_F32)
  KVGPT_PERSIST_CASE(256, EPI_RESID)
  KVGPT_PERSIST_CASE(256, EPI_GELU)
  KVGPT_PERSIST_CASE(256, EPI_QKV)
  KVGPT_PERSIST_CASE(192, EPI_F32)
  KVGPT_PERSIST_CASE(192, EPI_RESID)
  KVGPT_PERSIST_CASE(192, EPI_GELU)
  KVGPT_PERSIST_CASE(192, EPI_QKV)
  KVGPT_PERSIST_CASE(128, EPI_F32)
  KVGPT_PERSIST_CASE(128, EPI_RESID)
  KVGPT_PERSIST_CASE(128, EPI_GELU)
  KVGPT_PERSIST_CASE(128, EPI_QKV)
#undef KVGPT_PERSIST_CASE
  return cudaErrorInvalidValue;
}

cudaError_t set_tc_attr(int bn, bool hilo, int epi, int dev) {
#define KVGPT_TC_ATTR(BN, H, E, SLOT) \
  if (bn == BN && hilo == H && epi == E) return attr_tc<BN, H, E>(SLOT, dev);
  KVGPT_TC_ATTR(64, false, EPI_F32, 0)
  KVGPT_TC_ATTR(64, false, EPI_RESID, 1)
  KVGPT_TC_ATTR(64, false, EPI_GELU, 2)
  KVGPT_TC_ATTR(64, false, EPI_QKV, 3)
  KVGPT_TC_ATTR(64, true, EPI_F32, 4)
  KVGPT_TC_ATTR(64, true, EPI_RESID, 5)
  KVGPT_TC_ATTR(64, true, EPI_GELU, 6)
  KVGPT_TC_ATTR(64, true, EPI_QKV, 7)
  KVGPT_TC_ATTR(128, false, EPI_F32, 8)
  KVGPT_TC_ATTR(128, false, EPI_RESID, 9)
  KVGPT_TC_ATTR(128, false, EPI_GELU, 10)
  KVGPT_TC_ATTR(128, false, EPI_QKV, 11)
  KVGPT_TC_ATTR(128, true, EPI_F32, 12)
  KVGPT_TC_ATTR(128, true, EPI_RESID, 13)
  KVGPT_TC_ATTR(128, true, EPI_GELU, 14)
  KVGPT_TC_ATTR(128, true, EPI_QKV, 15)
  KVGPT_TC_ATTR(256, false, EPI_F32, 16)
  KVGPT_TC_ATTR(256, false, EPI_RESID, 17)
  KVGPT_TC_ATTR(256, false, EPI_GELU, 18)
  KVGPT_TC_ATTR(256, false, EPI_QKV, 19)
#undef KVGPT_TC_ATTR
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ decode-shape linear layers

// Per device: how many clusters of the decode linear kernel can be resident at once, for
// each cluster size (2, 4, 8, 16), token-row class (bp = 8 .. 128) and stage count (1 .. 3).
// Filled once per device (outside any stream capture); plans keep a launch within one wave.
int g_dl_max_clusters[64][5][DL_MAX_ROWS / 8][DL_MAX_STAGES] = {};
unsigned long long g_dl_attr_mask = 0;
std::mutex g_dl_mu;

template <int EPI>
cudaError_t dl_attr() {
  auto kern = dec_linear_kernel<EPI>;
  cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(dl_smem_bytes(DL_MAX_ROWS, DL_MAX_STAGES)));
  if (r != cudaSuccess) return r;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

int dl_max_clusters(int dev, int splits, int bp, int stages) {
  int si = 0;
  while ((2 << si) < splits) ++si;
  return g_dl_max_clusters[dev][si][bp / 8 - 1][stages - 1];
}

cudaError_t init_dl_attrs(int dev) {
  std::lock_guard<std::mutex> lk(g_dl_mu);
  if (g_dl_attr_mask & (1ull << dev)) return cudaSuccess;
  cudaError_t r;
  if ((r = dl_attr<EPI_F32>()) != cudaSuccess) return r;
  if ((r = dl_attr<EPI_RESID>()) != cudaSuccess) return r;
  if ((r = dl_attr<EPI_GELU>()) != cudaSuccess) return r;
  if ((r = dl_attr<EPI_QKV>()) != cudaSuccess) return r;
  for (int si = 0; si < 5; ++si)
    for (int bi = 0; bi < DL_MAX_ROWS / 8; ++bi)
      for (int st = 1; st <= DL_MAX_STAGES; ++st) {
        const int splits = 2 << si;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3(splits * 16);
        cfg.blockDim = dim3(DL_THREADS);
        cfg.dynamicSmemBytes = dl_smem_bytes(8 * (bi + 1), st);
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = splits;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (splits > DL_MAX_SPLITS || cudaOccupancyMaxActiveClusters(&n, dec_linear_kernel<EPI_RESID>, &cfg) != cudaSuccess) {
          cudaGetLastError();
          n = 0;
        }
        g_dl_max_clusters[dev][si][bi][st - 1] = n;
      }
  g_dl_attr_mask |= 1ull << dev;
  return cudaSuccess;
}

int dl_stages(int kb, int splits) { return std::min(DL_MAX_STAGES, cdiv(kb, splits)); }


// Split-K factor (= cluster size): the largest power of two <= 16 and <= the k-block count
// that keeps the grid within 2/3 of the SMs and all clusters resident in one wave.  (Fewer,
// larger CTAs measure faster than one CTA per SM here: the cost is latency, not bandwidth.)
int plan_dl_splits(int n_tiles, int kb, int rows, int num_sms, int dev) {
  const int bp = dl_bp(rows);
  int s = 1;
  for (int c = 2; c <= DL_MAX_SPLITS && c <= kb; c *= 2) {
    if (static_cast<long long>(n_tiles) * c * 3 > 2LL * num_sms) break;
    if (dl_max_clusters(dev, c, bp, dl_stages(kb, c)) < n_tiles) break;
    s = c;
  }
  return s;
}

cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Launch `kern` on `st`, as a programmatic dependent of the previous kernel when pdl is set
// (the kernel must call griddep_wait before touching data that earlier kernels produce).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Decode attention over a grid of (rows x splits) CTAs: the 8-warp form for small grids, the
// 4-warp form otherwise (DEC_WIDE_MAX_CTAS).  The choice depends on the shapes only, so every
// entry point gives the same results for the same inputs.
constexpr int DB_FEW_PAIRS = 32;  // the streamed decode attention takes splits up to this many (b, h)

unsigned long long g_db_attr_mask[2] = {};  // per paged flag: devices whose smem attribute is set
std::mutex g_db_mu;

template <bool PAGED>
cudaError_t db_attr(int dev) {
  std::lock_guard<std::mutex> lk(g_db_mu);
  if (g_db_attr_mask[PAGED] & (1ull << dev)) return cudaSuccess;
  cudaError_t r = cudaFuncSetAttribute(attn_decode_bulk<PAGED, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(DB_SMEM));
  if (r == cudaSuccess)
    r = cudaFuncSetAttribute(attn_decode_bulk<PAGED, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(DB_SMEM));
  if (r == cudaSuccess) g_db_attr_mask[PAGED] |= 1ull << dev;
  return r;
}

template <typename T, int HSZ, bool PAGED>
cudaError_t launch_dec_attn(int rows, int splits, cudaStream_t st, const T* q, const T* kc, const T* vc,
                            const KvLayout& kv, int nh, int block, const int* pos0, const int* pos_rows, float* ws,
                            unsigned int* tickets, T* y, T* y_lo, int C, int* err, bool step = false) {
  if constexpr (std::is_same<T, bf16>::value && HSZ == 64) {
    // the cache rows streamed through shared memory -- one split per (b, h) for up to 512 pairs
    // (a decode chain), or up to DB_MAX_SPLITS splits for a few pairs (B = 1); within a decode
    // step (step) as a programmatic dependent that streams the older rows before the c_attn
    // kernel that appends the newest one has finished.  In between (the 350M shape at B = 8,
    // 128 pairs) the register-load kernel measured faster: 1022 against 1058 / 1095 us per step
    // with 2 / 3 streamed splits.
    if ((splits == 1 && rows <= DEC_WIDE_MAX_CTAS) || (splits <= DB_MAX_SPLITS && rows <= DB_FEW_PAIRS)) {
      int dev = 0;
      cudaError_t r = cudaGetDevice(&dev);
      if (r == cudaSuccess) r = db_attr<PAGED>(dev);
      if (r != cudaSuccess) return r;
      if (step)
        return launch_k(attn_decode_bulk<PAGED, true>, dim3(rows, splits), dim3(DB_THREADS), DB_SMEM, st, true, q, kc,
                        vc, kv, nh, block, pos0, pos_rows, ws, tickets, y, y_lo, C, err);
      return launch_k(attn_decode_bulk<PAGED, false>, dim3(rows, splits), dim3(DB_THREADS), DB_SMEM, st, false, q, kc,
                      vc, kv, nh, block, pos0, pos_rows, ws, tickets, y, y_lo, C, err);
    }
  }
  if (static_cast<long long>(rows) * splits <= DEC_WIDE_MAX_CTAS)
    return launch_k(attn_decode_kernel<T, HSZ, PAGED, 8>, dim3(rows, splits), dim3(256), 0, st, false, q, kc, vc, kv,
                    nh, block, pos0, pos_rows, ws, tickets, y, y_lo, C, err);
  return launch_k(attn_decode_kernel<T, HSZ, PAGED, 4>, dim3(rows, splits), dim3(128), 0, st, false, q, kc, vc, kv, nh,
                  block, pos0, pos_rows, ws, tickets, y, y_lo, C, err);
}

template <int EPI>
cudaError_t launch_dl_epi(const CUtensorMap& tw, const CUtensorMap& tx, int kb, int splits, int stages, int n_tiles,
                          const Epi<bf16>& e, bool pdl, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  cfg.gridDim = dim3(n_tiles * splits);
  cfg.blockDim = dim3(DL_THREADS);
  cfg.dynamicSmemBytes = dl_smem_bytes(dl_bp(e.M), stages);
  cfg.stream = st;
  if (splits > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = splits;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) attr[na++] = pdl_attr();
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, dec_linear_kernel<EPI>, tw, tx, kb, splits, stages, e);
}

cudaError_t launch_dl(int epi, const CUtensorMap& tw, const CUtensorMap& tx, int kb, int splits, int stages,
                      int n_tiles, const Epi<bf16>& e, bool pdl, cudaStream_t st) {
  switch (epi) {
    case EPI_F32: return launch_dl_epi<EPI_F32>(tw, tx, kb, splits, stages, n_tiles, e, pdl, st);
    case EPI_RESID: return launch_dl_epi<EPI_RESID>(tw, tx, kb, splits, stages, n_tiles, e, pdl, st);
    case EPI_GELU: return launch_dl_epi<EPI_GELU>(tw, tx, kb, splits, stages, n_tiles, e, pdl, st);
    case EPI_QKV: return launch_dl_epi<EPI_QKV>(tw, tx, kb, splits, stages, n_tiles, e, pdl, st);
    default: return cudaErrorInvalidValue;
  }
}

// Raise the dynamic shared memory limit of every tensor-core GEMM instantiation and of
// the sampler once per device, before any stream capture can need them.
cudaError_t init_kernel_attrs(int dev) {
  static const int bns[3] = {64, 128, 256};
  for (int bi = 0; bi < 3; ++bi)
    for (int h = 0; h < 2; ++h)
      for (int epi = 0; epi < 4; ++epi) {
        if (bns[bi] == 256 && h) continue;
        cudaError_t r = set_tc_attr(bns[bi], h != 0, epi, dev);
        if (r != cudaSuccess) return r;
      }
  cudaError_t r = init_persist_attrs();
  if (r != cudaSuccess) return r;
  r = cudaFuncSetAttribute(attn_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(PT_SMEM));
  if (r != cudaSuccess) return r;
  return init_dl_attrs(dev);
}

struct GemmPlan {
  int bn = 64;
  int splits = 1;
};

// Output tile width and split-K count: wide tiles when there are enough tiles to fill the
// GPU, otherwise 64-wide tiles with the K range split until about one wave of CTAs.
GemmPlan plan_gemm(int M, int N, int K, int num_sms, bool hilo, size_t ws_bytes) {
  GemmPlan p;
  const int mt = cdiv(M, TC_BM), kb = K / TC_BK;
  if (!hilo && N % 256 == 0 && mt * (N / 256) >= num_sms) {
    p.bn = 256;
  } else if (N % 128 == 0 && mt * (N / 128) >= num_sms) {
    p.bn = 128;
  } else {
    p.bn = 64;
    if (N % 16 == 0) {
      const int tiles = mt * cdiv(N, 64);
      int s = std::max(1, std::min(kb, num_sms / std::max(1, tiles)));
      while (s > 1 && static_cast<size_t>(s) * M * N * sizeof(float) > ws_bytes) --s;
      const int kbps = cdiv(kb, s);
      p.splits = cdiv(kb, kbps);
    }
  }
  return p;
}

// ------------------------------------------------------------------ small kernels

__global__ void set_ints_kernel(int* a, int va, int* b, int vb) {
  if (a) *a = va;
  if (b) *b = vb;
}
// x_last[b, :] = x[b * T + lens[b] - 1, :] (each sequence's last prompt row, ragged prefill)
__global__ void gather_last_kernel(const float* __restrict__ x, const int* __restrict__ lens, int T, int C,
                                   float* __restrict__ out) {
  const int b = blockIdx.x;
  const float* src = x + (static_cast<size_t>(b) * T + lens[b] - 1) * C;
  for (int c = threadIdx.x; c < C; c += blockDim.x) out[static_cast<size_t>(b) * C + c] = src[c];
}
__global__ void add_one_kernel(int* lens, int B) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) lens[b] += 1;
}

__global__ void advance_kernel(int* pos, int* step) {
  griddep_wait();
  *pos += 1;
  *step += 1;
}

// LayerNorm launch with the register bound matched to C (pairs per lane = C / 64).
template <typename TO>
cudaError_t launch_ln(int rows, int C, long long in_stride, const float* x, const float* gamma, const float* beta,
                      TO* y, TO* y_lo, int ldy, cudaStream_t st, bool pdl) {
  const dim3 grid(cdiv(rows, 8)), block(256);
  if (C <= 12 * 64)
    return pdl ? launch_k(layernorm_kernel<TO, 12, true>, grid, block, 0, st, pdl, x, rows, C, in_stride, gamma, beta,
                          y, y_lo, ldy)
               : launch_k(layernorm_kernel<TO, 12, false>, grid, block, 0, st, pdl, x, rows, C, in_stride, gamma,
                          beta, y, y_lo, ldy);
  if (C <= 16 * 64)
    return pdl ? launch_k(layernorm_kernel<TO, 16, true>, grid, block, 0, st, pdl, x, rows, C, in_stride, gamma, beta,
                          y, y_lo, ldy)
               : launch_k(layernorm_kernel<TO, 16, false>, grid, block, 0, st, pdl, x, rows, C, in_stride, gamma,
                          beta, y, y_lo, ldy);
  return launch_k(layernorm_kernel<TO, LN_MAX_PAIRS>, grid, block, 0, st, pdl, x, rows, C, in_stride, gamma, beta, y,
                  y_lo, ldy);
}

int map_error_word(int w) {
  if (w & ERR_TOKEN) return GPT_ETOKEN;
  if (w & ERR_TIMEOUT) return GPT_ETIMEOUT;
  if (w & ERR_POSITION) return GPT_EPOSITION;
  return GPT_OK;
}

// Candidate slots the sampler gets after the V scaled logits: up to 4096, within the 227 KiB
// of dynamic shared memory a CTA may have (minus the kernel's static shared memory).
int sampler_cand_cap(int V) {
  const long long room = 232448LL - 4096 - static_cast<long long>(V) * 4;
  return static_cast<int>(std::max(0LL, std::min(4096LL, room / 4)));
}
size_t sampler_smem(int V) { return static_cast<size_t>(V + sampler_cand_cap(V)) * 4; }

cudaError_t set_sampler_smem(int dev, int V) {
  static int done_bytes[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  const int bytes = static_cast<int>(sampler_smem(V));
  if (done_bytes[dev] >= bytes) return cudaSuccess;
  cudaError_t r = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (r == cudaSuccess) done_bytes[dev] = bytes;
  return r;
}

constexpr int MAX_VOCAB = 57344;

// ------------------------------------------------------------------ stand-alone op scratch

struct OpCtx {
  int* err = nullptr;
  float* ws = nullptr;
  size_t ws_bytes = 0;
  unsigned int* tickets = nullptr;
  size_t n_tickets = 0;
};
OpCtx g_op[64];
std::mutex g_op_mu;

int op_ctx(OpCtx** out, size_t ws_need, size_t tickets_need) {
  int dev = 0;
  CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return GPT_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_op_mu);
  OpCtx& c = g_op[dev];
  if (!c.err) {
    CK(cudaMalloc(&c.err, sizeof(int)));
    CK(cudaMemset(c.err, 0, sizeof(int)));
  }
  if (c.ws_bytes < ws_need) {
    CK(cudaDeviceSynchronize());
    if (c.ws) CK(cudaFree(c.ws));
    c.ws = nullptr;
    c.ws_bytes = 0;
    CK(cudaMalloc(&c.ws, ws_need));
    c.ws_bytes = ws_need;
  }
  if (c.n_tickets < tickets_need) {
    CK(cudaDeviceSynchronize());
    if (c.tickets) CK(cudaFree(c.tickets));
    c.tickets = nullptr;
    c.n_tickets = 0;
    CK(cudaMalloc(&c.tickets, tickets_need * sizeof(unsigned int)));
    CK(cudaMemset(c.tickets, 0, tickets_need * sizeof(unsigned int)));
    c.n_tickets = tickets_need;
  }
  *out = &c;
  return GPT_OK;
}

}  // namespace

// ====================================================================== model

struct LayerDev {
  float *ln1_w = nullptr, *ln1_b = nullptr, *ln2_w = nullptr, *ln2_b = nullptr;
  void *attn_w = nullptr, *proj_w = nullptr, *fc_w = nullptr, *mproj_w = nullptr;
  float *attn_b = nullptr, *proj_b = nullptr, *fc_b = nullptr, *mproj_b = nullptr;
};

struct GraphKey {
  int B = -1, T = -1, N = -1, top_k = 0;
  float temperature = -1.0f;
  unsigned long long seed = 0;
  int* out = nullptr;
  bool operator==(const GraphKey& o) const {
    return B == o.B && T == o.T && N == o.N && top_k == o.top_k && temperature == o.temperature && seed == o.seed &&
           out == o.out;
  }
};

constexpr int DECODE_MAX_CHAINS = 4;
// Chains a decode step of DECODE_CHAINS_MIN .. DL_MAX_ROWS sequences runs as (measured at
// B = 64 on GPT-2 124M: 2 chains 86.4k tok/s, 3 chains 81.3k, 4 chains 85.0k).
constexpr int DECODE_CHAINS = 2;
static_assert(DECODE_CHAINS >= 2 && DECODE_CHAINS <= DECODE_MAX_CHAINS, "decode chains");

struct gpt_model {
  gpt_config_t cfg{};
  cudaStream_t stream = nullptr;
  cudaStream_t cap_stream = nullptr;  // private stream used only to record the decode graph
  // second streams of a decode step that runs as two chains (eager, and while recording)
  // extra streams of a decode step that runs as several chains (eager, and while recording),
  // the events that stagger their starts and join them
  cudaStream_t stream_x[DECODE_MAX_CHAINS] = {}, cap_stream_x[DECODE_MAX_CHAINS] = {};
  cudaEvent_t ev_mark[DECODE_MAX_CHAINS] = {}, ev_join[DECODE_MAX_CHAINS] = {};
  int dev = 0, num_sms = 148;
  bool bf16 = true;
  size_t esz = 2;
  int C = 0, nh = 0, hs = 64, L = 0, V = 0, block = 0, Bmax = 0;
  std::vector<void*> allocs;
  void* wte = nullptr;
  void* wpe = nullptr;
  float* ln_f_w = nullptr;
  float* ln_f_b = nullptr;
  std::vector<LayerDev> layers;
  void* kv = nullptr;
  float* x = nullptr;
  void* xn = nullptr;
  void* q = nullptr;
  void* y = nullptr;
  void* h = nullptr;
  void* xf = nullptr;
  float* logits = nullptr;
  float* ws = nullptr;
  size_t ws_bytes = 0;
  unsigned int* tickets = nullptr;
  size_t n_tickets = 0;
  int* d_err = nullptr;
  int* d_pos = nullptr;
  int* d_step = nullptr;
  int* d_tokens = nullptr;
  // ragged batches (gpt_prefill_ragged): every sequence at its own cache length
  bool ragged = false;
  std::vector<int> h_lens;  // host mirror of d_lens
  int* d_lens = nullptr;
  float* xlast = nullptr;  // each sequence's last prompt position, gathered for ln_f / lm_head
  int cache_len = 0, batch = 0;
  bool hilo_decode = true;  // hi/lo bf16 operands for decode-step GEMMs (memory-bound, so free)
  cudaGraphExec_t gexec = nullptr;
  GraphKey gkey;
  long long launches = 0;       // kernels enqueued so far (graph replays count every kernel node)
  long long graph_kernels = 0;  // kernel nodes in the captured decode-step graph
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  bool timing_valid = false;
  // GEMM timing of prefills (gpt_profile_gemms): events around every prefill GEMM launch
  bool prof_enabled = false, prof_active = false;
  std::vector<cudaEvent_t> prof_ev;
  size_t prof_n = 0;      // events recorded by the last profiled prefill
  double prof_flops = 0;  // 2 M N K summed over its GEMMs
  std::map<std::tuple<uintptr_t, long long, long long, int>, CUtensorMap> wmaps;

  template <typename T>
  T* alloc(size_t count, int* rc) {
    void* p = nullptr;
    cudaError_t e = fail_this_allocation() ? cudaErrorMemoryAllocation : cudaMalloc(&p, count * sizeof(T));
    if (e != cudaSuccess) {
      *rc = cuda_fail(e, "cudaMalloc");
      return nullptr;
    }
    allocs.push_back(p);
    return static_cast<T*>(p);
  }
  void* alloc_bytes(size_t n, int* rc) { return alloc<uint8_t>(n, rc); }

  void* kcache(int l) const { return static_cast<uint8_t*>(kv) + (static_cast<size_t>(l) * 2) * cache_layer_bytes(); }
  void* vcache(int l) const {
    return static_cast<uint8_t*>(kv) + (static_cast<size_t>(l) * 2 + 1) * cache_layer_bytes();
  }
  size_t cache_layer_bytes() const {
    return paged ? static_cast<size_t>(n_pages) * nh * page_size * hs * esz
                 : static_cast<size_t>(Bmax) * nh * block * hs * esz;
  }
  // paged KV cache (gpt_create_paged): n_pages pages of page_size positions for every layer's
  // K and V; sequence b's position pos lives in page h_table[b * pages_per_seq + pos / page_size]
  bool paged = false;
  int page_size = 0, page_shift = 0, n_pages = 0, pages_per_seq = 0;
  int* d_table = nullptr;
  std::vector<int> h_table;  // -1: no page yet
  std::vector<int> free_pages;
  KvLayout kv_layout() const {
    KvLayout k;
    k.nh = nh;
    k.block = block;
    if (paged) {
      k.table = d_table;
      k.pages_per_seq = pages_per_seq;
      k.page_shift = page_shift;
    }
    return k;
  }

  int weight_map(const void* w, long long rows, long long cols, int box_rows, CUtensorMap* out) {
    auto key = std::make_tuple(reinterpret_cast<uintptr_t>(w), rows, cols, box_rows);
    auto it = wmaps.find(key);
    if (it != wmaps.end()) {
      *out = it->second;
      return GPT_OK;
    }
    int rc = make_tmap(out, w, rows, cols, box_rows);
    if (rc == GPT_OK) wmaps[key] = *out;
    return rc;
  }
};

namespace {

void free_model(gpt_model* m) {
  if (!m) return;
  cudaStreamSynchronize(m->stream);
  if (m->gexec) cudaGraphExecDestroy(m->gexec);
  for (auto& e : m->ev)
    if (e) cudaEventDestroy(e);
  for (auto& e : m->prof_ev)
    if (e) cudaEventDestroy(e);
  for (void* p : m->allocs) cudaFree(p);
  if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
  for (int i = 0; i < DECODE_MAX_CHAINS; ++i) {
    if (m->stream_x[i]) cudaStreamDestroy(m->stream_x[i]);
    if (m->cap_stream_x[i]) cudaStreamDestroy(m->cap_stream_x[i]);
    if (m->ev_mark[i]) cudaEventDestroy(m->ev_mark[i]);
    if (m->ev_join[i]) cudaEventDestroy(m->ev_join[i]);
  }
  delete m;
}

// ---- paged KV cache: block tables filled on demand, emptied by every prefill

void release_all_pages(gpt_model* m) {
  if (!m->paged) return;
  std::fill(m->h_table.begin(), m->h_table.end(), -1);
  m->free_pages.clear();
  for (int pg = m->n_pages - 1; pg >= 0; --pg) m->free_pages.push_back(pg);
}

// Give sequences 0..B-1 pages for positions < len(b) (len(b) = lens ? lens[b] : len_all), then
// upload the table (before the kernels that use it are enqueued).  GPT_ENOMEM, before anything
// is enqueued, when the pool has too few free pages.
int ensure_pages(gpt_model* m, int B, const int* lens, int len_all) {
  if (!m->paged) return GPT_OK;
  size_t need = 0;
  for (int b = 0; b < B; ++b) {
    const int n = (std::min(lens ? lens[b] : len_all, m->block) + m->page_size - 1) / m->page_size;
    for (int i = 0; i < n; ++i) need += m->h_table[static_cast<size_t>(b) * m->pages_per_seq + i] < 0;
  }
  if (need > m->free_pages.size()) {
    g_detail = "paged KV cache: " + std::to_string(need) + " more pages needed, " +
               std::to_string(m->free_pages.size()) + " free";
    return GPT_ENOMEM;
  }
  for (int b = 0; b < B; ++b) {
    const int n = (std::min(lens ? lens[b] : len_all, m->block) + m->page_size - 1) / m->page_size;
    for (int i = 0; i < n; ++i) {
      int& slot = m->h_table[static_cast<size_t>(b) * m->pages_per_seq + i];
      if (slot < 0) {
        slot = m->free_pages.back();
        m->free_pages.pop_back();
      }
    }
  }
  CK(cudaMemcpyAsync(m->d_table, m->h_table.data(), m->h_table.size() * sizeof(int), cudaMemcpyHostToDevice,
                     m->stream));
  return GPT_OK;
}

// y = A W^T with the given epilogue, bf16 operands.  A has M rows (2M with hilo).
int gemm_bf16_launch(gpt_model* m, const bf16* A, const void* W, int M, int N, int K, bool hilo, int epi, Epi<bf16> e,
                     bool allow_split);

int gemm_bf16(gpt_model* m, const bf16* A, const void* W, int M, int N, int K, bool hilo, int epi, Epi<bf16> e,
              bool allow_split) {
  const bool prof = m->prof_active && m->prof_n + 2 <= m->prof_ev.size();
  if (prof) CK(cudaEventRecord(m->prof_ev[m->prof_n], m->stream));
  const int rc = gemm_bf16_launch(m, A, W, M, N, K, hilo, epi, e, allow_split);
  if (rc) return rc;
  if (prof) {
    CK(cudaEventRecord(m->prof_ev[m->prof_n + 1], m->stream));
    m->prof_n += 2;
    m->prof_flops += 2.0 * M * N * K;
  }
  return GPT_OK;
}

int gemm_bf16_launch(gpt_model* m, const bf16* A, const void* W, int M, int N, int K, bool hilo, int epi, Epi<bf16> e,
                     bool allow_split) {
  // Enough 128 x BN tiles for every SM: the persistent kernel (one CTA per SM).
  const int bnp = hilo ? 0 : persist_bn(M, N, m->num_sms);
  if (bnp) {
    CUtensorMap ta, tb;
    int rc = make_tmap(&ta, A, M, K, TC_BM);
    if (rc) return rc;
    rc = m->weight_map(W, N, K, bnp, &tb);
    if (rc) return rc;
    e.M = M;
    e.N = N;
    e.splits = 1;
    e.err = m->d_err;
    CK(launch_persist(bnp, epi, ta, tb, K, m->num_sms, e, m->stream));
    ++m->launches;
    return GPT_OK;
  }
  GemmPlan p = plan_gemm(M, N, K, m->num_sms, hilo, m->ws_bytes);
  if (!allow_split) p.splits = 1;
  if (p.splits > 1 && static_cast<size_t>(cdiv(M, TC_BM)) * cdiv(N, p.bn) > m->n_tickets) p.splits = 1;
  CUtensorMap ta, tb;
  int rc = make_tmap(&ta, A, hilo ? 2LL * M : M, K, TC_BM);
  if (rc) return rc;
  rc = m->weight_map(W, N, K, p.bn, &tb);
  if (rc) return rc;
  e.M = M;
  e.N = N;
  e.splits = p.splits;
  e.ws = m->ws;
  e.tickets = m->tickets;
  e.err = m->d_err;
  CK(dispatch_tc(p.bn, hilo, epi, m->dev, ta, tb, M, N, K, p.splits, e, m->stream));
  ++m->launches;
  return GPT_OK;
}

// Decode-shape Linear (M <= 128 token rows given as a hi/lo pair): swap-AB tcgen05 kernel with
// cluster split-K, launched as a programmatic dependent of the previous kernel.
int dec_linear(gpt_model* m, const bf16* A, const void* W, int M, int N, int K, int epi, Epi<bf16> e) {
  const int kb = K / TC_BK, n_tiles = cdiv(N, 128);
  const int splits = plan_dl_splits(n_tiles, kb, M, m->num_sms, m->dev);
  CUtensorMap tx, tw;
  int rc = make_tmap(&tx, A, 2LL * M, K, dl_bp(M));
  if (rc) return rc;
  rc = m->weight_map(W, N, K, 128, &tw);
  if (rc) return rc;
  e.M = M;
  e.N = N;
  e.T = 1;
  e.err = m->d_err;
  CK(launch_dl(epi, tw, tx, kb, splits, dl_stages(kb, splits), n_tiles, e, true,
               m->stream));
  ++m->launches;
  return GPT_OK;
}

template <int EPI>
int gemm_f32(gpt_model* m, const float* A, const void* W, int M, int N, int K, Epi<float> e) {
  e.M = M;
  e.N = N;
  e.err = m->d_err;
  dim3 grid(cdiv(N, F32_BN), cdiv(M, F32_BM));
  gemm_f32_kernel<EPI><<<grid, 256, 0, m->stream>>>(A, static_cast<const float*>(W), K, e);
  CK(cudaGetLastError());
  ++m->launches;
  return GPT_OK;
}

int decode_attn_splits(const gpt_model* m, int B, size_t ws_bytes, size_t n_tickets) {
  const int pairs = B * m->nh;
  int s = cdiv(2 * m->num_sms, pairs);
  s = std::max(1, std::min(s, std::min(32, cdiv(m->block, 16))));
  // a few pairs (B = 1): at most DB_MAX_SPLITS splits, so that the streamed kernel takes them
  if (m->bf16 && m->hs == 64 && pairs <= DB_FEW_PAIRS) s = std::min(s, DB_MAX_SPLITS);
  while (s > 1 && static_cast<size_t>(pairs) * s * (m->hs + 2) * sizeof(float) > ws_bytes) --s;
  if (static_cast<size_t>(pairs) > n_tickets) s = 1;
  return s;
}

// The sequences [row0, row0 + B) of the batch that one forward pass runs, with the scratch it
// may use.  A decode step of a large batch runs as two such chains on two streams (see
// enqueue_decode); everything else runs one chain over the whole batch.
struct Chain {
  int row0 = 0;
  float* x = nullptr;
  void *xn = nullptr, *q = nullptr, *y = nullptr, *h = nullptr, *xf = nullptr;
  float* ws = nullptr;
  size_t ws_bytes = 0;
  unsigned int* tickets = nullptr;
  size_t n_tickets = 0;
  cudaEvent_t mark = nullptr;  // recorded once layer 0's c_attn is enqueued, when set
};

Chain whole_batch(gpt_model* m) {
  Chain c;
  c.x = m->x;
  c.xn = m->xn;
  c.q = m->q;
  c.y = m->y;
  c.h = m->h;
  c.xf = m->xf;
  c.ws = m->ws;
  c.ws_bytes = m->ws_bytes;
  c.tickets = m->tickets;
  c.n_tickets = m->n_tickets;
  return c;
}

// Enqueue the forward pass over B x T new tokens.  decode: T == 1 and the position comes
// from m->d_pos; otherwise the tokens start at position off (0 for a prefill, the cache
// length for a chunk appended by gpt_extend, which m->d_pos then holds).  Logits of each
// sequence's last token go to logits (row stride V).
template <typename TE>
int enqueue_forward(gpt_model* m, const int* tokens, int B, int T, bool decode, float* logits, int off, int tok_ld,
                    const int* lens, const Chain& ch) {
  constexpr bool kBf16 = std::is_same<TE, bf16>::value;
  const int C = m->C, nh = m->nh, V = m->V, rows = B * T;
  const bool hilo = kBf16 && decode && m->hilo_decode;
  // decode-shape Linear layers (swap-AB, cluster split-K) and programmatic dependent launches
  const bool dl = hilo && rows <= DL_MAX_ROWS;
  // up to 8 rows the decode-shape kernels take LayerNorm(x) as their operand directly
  const bool ln_in = dl && rows <= DL_LN_MAX_ROWS;
  const bool pdl = decode;
  const int* pos0 = (decode || off > 0) ? m->d_pos : nullptr;
  // decode steps of a ragged batch: each sequence at its own length; a ragged prefill: rows
  // past lens[b] are padding
  const int* pos_rows = decode && m->ragged ? m->d_lens + ch.row0 : nullptr;
  cudaStream_t st = m->stream;
  float* x = ch.x;
  TE* xn = static_cast<TE*>(ch.xn);
  TE* q = static_cast<TE*>(ch.q);
  TE* y = static_cast<TE*>(ch.y);
  TE* hbuf = static_cast<TE*>(ch.h);
  TE* xf = static_cast<TE*>(ch.xf);
  // this chain's sequences in the KV cache: an offset into the contiguous cache, or into the
  // block table
  KvLayout kvl = m->kv_layout();
  size_t kv_off = 0;
  if (m->paged)
    kvl.table += static_cast<size_t>(ch.row0) * m->pages_per_seq;
  else
    kv_off = static_cast<size_t>(ch.row0) * nh * m->block * m->hs;
  const int rows_per_cta = 8;  // 256 threads, warp per row

  embed_kernel<TE><<<cdiv(rows, rows_per_cta), 256, 0, st>>>(tokens, tok_ld, pos_rows, lens, rows, T, pos0, static_cast<const TE*>(m->wte),
                                                               static_cast<const TE*>(m->wpe), V, m->block, C, x,
                                                               m->d_err);
  CK(cudaGetLastError());
  ++m->launches;
  for (int l = 0; l < m->L; ++l) {
    const LayerDev& w = m->layers[l];
    TE* kc = static_cast<TE*>(m->kcache(l)) + kv_off;
    TE* vc = static_cast<TE*>(m->vcache(l)) + kv_off;
    // ln_1 (in the c_attn kernel when ln_in)
    if (!ln_in) {
      CK(launch_ln<TE>(rows, C, C, x, w.ln1_w, w.ln1_b, xn,
                       hilo ? xn + static_cast<size_t>(rows) * C : static_cast<TE*>(nullptr), C, st, pdl));
      ++m->launches;
    }
    // c_attn + KV append
    {
      Epi<TE> e;
      e.bias = w.attn_b;
      e.q = q;
      e.kc = kc;
      e.vc = vc;
      e.C = C;
      e.nh = nh;
      e.hs = m->hs;
      e.T = T;
      e.block = m->block;
      e.pos0 = pos0;
      e.pos_rows = pos_rows;
      e.kv = kvl;
      if (ln_in) {
        e.ln_x = x;
        e.ln_ldx = C;
        e.ln_g = w.ln1_w;
        e.ln_b = w.ln1_b;
      }
      int rc;
      if constexpr (kBf16)
        rc = dl ? dec_linear(m, xn, w.attn_w, rows, 3 * C, C, EPI_QKV, e)
                : gemm_bf16(m, xn, w.attn_w, rows, 3 * C, C, hilo, EPI_QKV, e, decode);
      else
        rc = gemm_f32<EPI_QKV>(m, xn, w.attn_w, rows, 3 * C, C, e);
      if (rc) return rc;
      if (l == 0 && ch.mark) CK(cudaEventRecord(ch.mark, st));
    }
    // attention
    if (decode) {
      const int splits = decode_attn_splits(m, B, ch.ws_bytes, ch.n_tickets);
      TE* y_lo = hilo ? y + static_cast<size_t>(B) * C : nullptr;
      const TE* qc = q;
      // Launched as an ordinary (not programmatic) dependent: its many small CTAs would otherwise
      // sit on the SMs the c_attn GEMM is still using (measured: 7 % slower decode steps at B=64).
      const int* dpos = static_cast<const int*>(m->d_pos);
      if (m->hs == 64 && m->paged)
        CK((launch_dec_attn<TE, 64, true>(B * nh, splits, st, qc, kc, vc, kvl, nh, m->block, dpos, pos_rows, ch.ws,
                                          ch.tickets, y, y_lo, C, m->d_err, true)));
      else if (m->paged)
        CK((launch_dec_attn<TE, 32, true>(B * nh, splits, st, qc, kc, vc, kvl, nh, m->block, dpos, pos_rows, ch.ws,
                                          ch.tickets, y, y_lo, C, m->d_err, true)));
      else if (m->hs == 64)
        CK((launch_dec_attn<TE, 64, false>(B * nh, splits, st, qc, kc, vc, kvl, nh, m->block, dpos, pos_rows, ch.ws,
                                           ch.tickets, y, y_lo, C, m->d_err, true)));
      else
        CK((launch_dec_attn<TE, 32, false>(B * nh, splits, st, qc, kc, vc, kvl, nh, m->block, dpos, pos_rows, ch.ws,
                                           ch.tickets, y, y_lo, C, m->d_err, true)));
    } else if constexpr (kBf16) {
      // q [B][nh][T][64] and this layer's cache rows as 2-D tensors for TMA
      const long long cache_rows = static_cast<long long>(m->cache_layer_bytes() / (m->hs * m->esz));
      CUtensorMap tq, tk, tv;
      int rc = m->weight_map(q, static_cast<long long>(B) * nh * T, m->hs, PT_BQ, &tq);
      if (!rc) rc = m->weight_map(m->kcache(l), cache_rows, m->hs, PT_BK, &tk);
      if (!rc) rc = m->weight_map(m->vcache(l), cache_rows, m->hs, PT_BK, &tv);
      if (rc) return rc;
      const int items = cdiv(T, PT_BQ) * B * nh;
      attn_prefill_tc<<<std::min(items, PT_CTAS_PER_SM * m->num_sms), PT_THREADS, PT_SMEM, st>>>(
          tq, tk, tv, kvl, nh, B * nh, T, off, y, C, m->d_err);
    } else {
      if (m->hs == 64)
        attn_prefill_f32<64><<<dim3(T, B * nh), 32, (off + T) * sizeof(float), st>>>(q, kc, vc, kvl, nh, T,
                                                                                      m->block, off,
                                                                                      y, C);
      else
        attn_prefill_f32<32><<<dim3(T, B * nh), 32, (off + T) * sizeof(float), st>>>(q, kc, vc, kvl, nh, T,
                                                                                      m->block, off,
                                                                                      y, C);
    }
    CK(cudaGetLastError());
    ++m->launches;
    // attn c_proj + residual
    {
      Epi<TE> e;
      e.bias = w.proj_b;
      e.x = x;
      e.ldx = C;
      int rc;
      if constexpr (kBf16)
        rc = dl ? dec_linear(m, y, w.proj_w, rows, C, C, EPI_RESID, e)
                : gemm_bf16(m, y, w.proj_w, rows, C, C, hilo, EPI_RESID, e, decode);
      else
        rc = gemm_f32<EPI_RESID>(m, y, w.proj_w, rows, C, C, e);
      if (rc) return rc;
    }
    // ln_2 (in the c_fc kernel when ln_in)
    if (!ln_in) {
      CK(launch_ln<TE>(rows, C, C, x, w.ln2_w, w.ln2_b, xn,
                       hilo ? xn + static_cast<size_t>(rows) * C : static_cast<TE*>(nullptr), C, st, pdl));
      ++m->launches;
    }
    // mlp c_fc + GELU
    {
      Epi<TE> e;
      e.bias = w.fc_b;
      if (ln_in) {
        e.ln_x = x;
        e.ln_ldx = C;
        e.ln_g = w.ln2_w;
        e.ln_b = w.ln2_b;
      }
      e.out = hbuf;
      e.out_lo = hilo ? hbuf + static_cast<size_t>(rows) * 4 * C : nullptr;
      e.ldo = 4 * C;
      int rc;
      if constexpr (kBf16)
        rc = dl ? dec_linear(m, xn, w.fc_w, rows, 4 * C, C, EPI_GELU, e)
                : gemm_bf16(m, xn, w.fc_w, rows, 4 * C, C, hilo, EPI_GELU, e, decode);
      else
        rc = gemm_f32<EPI_GELU>(m, xn, w.fc_w, rows, 4 * C, C, e);
      if (rc) return rc;
    }
    // mlp c_proj + residual
    {
      Epi<TE> e;
      e.bias = w.mproj_b;
      e.x = x;
      e.ldx = C;
      int rc;
      if constexpr (kBf16)
        rc = dl ? dec_linear(m, hbuf, w.mproj_w, rows, C, 4 * C, EPI_RESID, e)
                : gemm_bf16(m, hbuf, w.mproj_w, rows, C, 4 * C, hilo, EPI_RESID, e, decode);
      else
        rc = gemm_f32<EPI_RESID>(m, hbuf, w.mproj_w, rows, C, 4 * C, e);
      if (rc) return rc;
    }
  }
  // ln_f on the last position of each sequence (in the lm_head kernel up to 8 sequences),
  // then the tied lm_head.  A ragged prefill first gathers each sequence's last prompt row.
  const float* xlast = x + static_cast<size_t>(T - 1) * C;
  long long xlast_ld = static_cast<long long>(T) * C;
  if (lens) {
    gather_last_kernel<<<B, 256, 0, st>>>(x, lens, T, C, m->xlast);
    CK(cudaGetLastError());
    ++m->launches;
    xlast = m->xlast;
    xlast_ld = C;
  }
  const bool ln_f_in = kBf16 && B <= DL_LN_MAX_ROWS;
  if (!ln_f_in) {
    CK(launch_ln<TE>(B, C, xlast_ld, xlast, m->ln_f_w, m->ln_f_b, xf,
                     kBf16 ? xf + static_cast<size_t>(B) * C : static_cast<TE*>(nullptr), C, st, pdl && !lens));
    ++m->launches;
  }
  {
    Epi<TE> e;
    e.x = logits;
    e.ldx = V;
    if (ln_f_in) {
      e.ln_x = xlast;
      e.ln_ldx = xlast_ld;
      e.ln_g = m->ln_f_w;
      e.ln_b = m->ln_f_b;
    }
    int rc;
    if constexpr (kBf16)
      rc = B <= DL_MAX_ROWS ? dec_linear(m, xf, m->wte, B, V, C, EPI_F32, e)
                            : gemm_bf16(m, xf, m->wte, B, V, C, true, EPI_F32, e, false);
    else
      rc = gemm_f32<EPI_F32>(m, xf, m->wte, B, V, C, e);
    if (rc) return rc;
  }
  return GPT_OK;
}

int forward(gpt_model* m, const int* tokens, int B, int T, bool decode, float* logits, int off = 0, int tok_ld = -1,
            const int* lens = nullptr) {
  if (tok_ld < 0) tok_ld = T;
  m->prof_active = m->prof_enabled && !decode;
  if (m->prof_active) {
    m->prof_n = 0;
    m->prof_flops = 0;
  }
  const Chain ch = whole_batch(m);
  const int rc = m->bf16 ? enqueue_forward<bf16>(m, tokens, B, T, decode, logits, off, tok_ld, lens, ch)
                         : enqueue_forward<float>(m, tokens, B, T, decode, logits, off, tok_ld, lens, ch);
  m->prof_active = false;
  return rc;
}

// A decode step over B sequences (tokens: B ids).  From DECODE_CHAINS_MIN sequences up (bf16,
// decode-shape kernels) it runs as DECODE_CHAINS chains of about B/DECODE_CHAINS sequences on
// their own streams, each starting once the previous one has enqueued layer 0's c_attn.  The
// kernels of one chain are latency-bound (the decode Linear layers and LayerNorms of a few dozen
// rows) while another chain's attention streams its share of the KV cache, so the chains
// overlap; each chain has its own rows of every scratch buffer and its own share of the split-KV
// scratch.  All chains are joined on the model's stream before this returns.
constexpr int DECODE_CHAINS_MIN = 32;

bool decode_multi_chain(const gpt_model* m, int B) {
  return m->bf16 && m->hilo_decode && B >= DECODE_CHAINS_MIN && B <= DL_MAX_ROWS;
}

int decode_forward(gpt_model* m, const int* tokens, int B, float* logits) {
  if (!decode_multi_chain(m, B)) return forward(m, tokens, B, 1, true, logits);
  m->prof_active = false;
  const int n = DECODE_CHAINS;
  const size_t C = m->C, e = m->esz;
  const cudaStream_t s0 = m->stream;
  const bool capturing = s0 == m->cap_stream;
  int rc = GPT_OK;
  for (int i = 0; i < n; ++i) {
    const int r0 = B * i / n, r1 = B * (i + 1) / n;
    Chain c = whole_batch(m);
    c.row0 = r0;
    c.mark = i + 1 < n ? m->ev_mark[i] : nullptr;
    c.ws_bytes = (m->ws_bytes / n) & ~static_cast<size_t>(255);
    c.n_tickets = m->n_tickets / n;
    c.x = m->x + r0 * C;
    c.xn = static_cast<uint8_t*>(m->xn) + 2 * r0 * C * e;  // hi and lo rows of earlier chains come first
    c.q = static_cast<uint8_t*>(m->q) + r0 * C * e;
    c.y = static_cast<uint8_t*>(m->y) + 2 * r0 * C * e;
    c.h = static_cast<uint8_t*>(m->h) + 2 * r0 * 4 * C * e;
    c.xf = static_cast<uint8_t*>(m->xf) + 2 * r0 * C * e;
    c.ws = m->ws + i * (c.ws_bytes / sizeof(float));
    c.tickets = m->tickets + i * c.n_tickets;
    if (i > 0) {
      m->stream = capturing ? m->cap_stream_x[i] : m->stream_x[i];
      CK(cudaStreamWaitEvent(m->stream, m->ev_mark[i - 1], 0));
    }
    rc = enqueue_forward<bf16>(m, tokens + r0, r1 - r0, 1, true, logits + static_cast<size_t>(r0) * m->V, 0, 1,
                               nullptr, c);
    if (!rc && i > 0) {
      if (cudaEventRecord(m->ev_join[i], m->stream) != cudaSuccess) rc = GPT_ECUDA;
    }
    m->stream = s0;
    if (rc) return rc;
  }
  for (int i = 1; i < n; ++i) CK(cudaStreamWaitEvent(s0, m->ev_join[i], 0));
  return GPT_OK;
}

int enqueue_sample(gpt_model* m, int B, float temperature, int top_k, unsigned long long seed, const int* step_dev,
                   int step, int* out, int out_stride, int out_col0, cudaStream_t st, bool pdl = true) {
  CK(set_sampler_smem(m->dev, m->V));
  SampleArgs a;
  a.logits = m->logits;
  a.ld = m->V;
  a.V = m->V;
  a.temperature = temperature;
  a.top_k = top_k;
  a.seed = seed;
  a.step_dev = step_dev;
  a.step = step;
  a.out = out;
  a.out_stride = out_stride;
  a.out_col0 = out_col0;
  a.next_tokens = m->d_tokens;
  a.thr_out = nullptr;
  a.w_out = nullptr;
  a.cand_cap = sampler_cand_cap(m->V);
  CK(launch_k(sample_kernel, dim3(B), dim3(SMP_THREADS), sampler_smem(m->V), st, pdl, a));
  ++m->launches;
  return GPT_OK;
}

template <typename TW>
int copy_vec_f32(gpt_model* m, const void* src, size_t n, float** dst) {
  int rc = GPT_OK;
  *dst = m->alloc<float>(n, &rc);
  if (!*dst) return rc;
  widen_kernel<TW><<<std::min<long long>(1024, cdiv(n, 256)), 256, 0, m->stream>>>(static_cast<const TW*>(src), *dst,
                                                                                    static_cast<long long>(n));
  CK(cudaGetLastError());
  return GPT_OK;
}

int copy_mat(gpt_model* m, const void* src, size_t n, void** dst) {
  int rc = GPT_OK;
  *dst = m->alloc_bytes(n * m->esz, &rc);
  if (!*dst) return rc;
  CK(cudaMemcpyAsync(*dst, src, n * m->esz, cudaMemcpyDeviceToDevice, m->stream));
  return GPT_OK;
}

int copy_vec(gpt_model* m, const void* src, size_t n, float** dst) {
  if (!src) {
    *dst = nullptr;
    return GPT_OK;
  }
  return m->bf16 ? copy_vec_f32<bf16>(m, src, n, dst) : copy_vec_f32<float>(m, src, n, dst);
}

int validate_config(const gpt_config_t* c) {
  if (!c) return GPT_EINVAL;
  if (c->n_layer < 0 || c->n_head < 1 || c->n_embd < 64 || c->n_embd % 64 != 0 || c->n_embd > 2048) return GPT_EINVAL;
  const int hs = c->n_embd % c->n_head == 0 ? c->n_embd / c->n_head : 0;
  if (hs != 64 && !(hs == 32 && c->dtype == GPT_DTYPE_F32)) return GPT_EINVAL;
  if (c->dtype == GPT_DTYPE_F32 && c->block_size > 12288) return GPT_EINVAL;  // fp32 prefill keeps scores in smem
  if (c->block_size < 1 || c->vocab_size < 1 || c->vocab_size > MAX_VOCAB) return GPT_EINVAL;
  if ((c->bias != 0 && c->bias != 1) || (c->dtype != GPT_DTYPE_F32 && c->dtype != GPT_DTYPE_BF16)) return GPT_EINVAL;
  if (c->max_batch < 1 || c->max_batch > 4096) return GPT_EINVAL;
  return GPT_OK;
}

int create_impl(const gpt_config_t* cfg, const gpt_weights_t* w, void* stream, gpt_model* m) {
  m->cfg = *cfg;
  m->stream = static_cast<cudaStream_t>(stream);
  CK(cudaGetDevice(&m->dev));
  if (m->dev >= 64) return GPT_EUNSUPPORTED;
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, m->dev));
  if (prop.major != 10 || prop.minor != 3) {
    g_detail = std::string("device is ") + prop.name + " (sm_" + std::to_string(prop.major) +
               std::to_string(prop.minor) + "); this library is built for sm_103a";
    return GPT_EUNSUPPORTED;
  }
  if (!load_encode()) return GPT_EUNSUPPORTED;
  m->num_sms = prop.multiProcessorCount;
  CK(init_kernel_attrs(m->dev));
  CK(set_sampler_smem(m->dev, cfg->vocab_size));
  CK(cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking));
  for (int i = 1; i < DECODE_MAX_CHAINS; ++i) {
    CK(cudaStreamCreateWithFlags(&m->stream_x[i], cudaStreamNonBlocking));
    CK(cudaStreamCreateWithFlags(&m->cap_stream_x[i], cudaStreamNonBlocking));
  }
  for (int i = 0; i < DECODE_MAX_CHAINS; ++i) {
    CK(cudaEventCreateWithFlags(&m->ev_mark[i], cudaEventDisableTiming));
    CK(cudaEventCreateWithFlags(&m->ev_join[i], cudaEventDisableTiming));
  }
  for (auto& e : m->ev) CK(cudaEventCreate(&e));
  m->bf16 = cfg->dtype == GPT_DTYPE_BF16;
  m->esz = m->bf16 ? 2 : 4;
  m->C = cfg->n_embd;
  m->nh = cfg->n_head;
  m->hs = cfg->n_embd / cfg->n_head;
  m->L = cfg->n_layer;
  m->V = cfg->vocab_size;
  m->block = cfg->block_size;
  m->Bmax = cfg->max_batch;
  const size_t C = m->C, V = m->V, blk = m->block, Bm = m->Bmax;
  const bool has_bias = cfg->bias == 1;
  int rc = GPT_OK;

  // weights
  if ((rc = copy_mat(m, w->wte, V * C, &m->wte))) return rc;
  if ((rc = copy_mat(m, w->wpe, blk * C, &m->wpe))) return rc;
  if ((rc = copy_vec(m, w->ln_f_w, C, &m->ln_f_w))) return rc;
  if ((rc = copy_vec(m, has_bias ? w->ln_f_b : nullptr, C, &m->ln_f_b))) return rc;
  m->layers.resize(m->L);
  for (int l = 0; l < m->L; ++l) {
    const gpt_layer_weights_t& s = w->layers[l];
    LayerDev& d = m->layers[l];
    if ((rc = copy_vec(m, s.ln_1_w, C, &d.ln1_w))) return rc;
    if ((rc = copy_vec(m, has_bias ? s.ln_1_b : nullptr, C, &d.ln1_b))) return rc;
    if ((rc = copy_mat(m, s.c_attn_w, 3 * C * C, &d.attn_w))) return rc;
    if ((rc = copy_vec(m, has_bias ? s.c_attn_b : nullptr, 3 * C, &d.attn_b))) return rc;
    if ((rc = copy_mat(m, s.attn_proj_w, C * C, &d.proj_w))) return rc;
    if ((rc = copy_vec(m, has_bias ? s.attn_proj_b : nullptr, C, &d.proj_b))) return rc;
    if ((rc = copy_vec(m, s.ln_2_w, C, &d.ln2_w))) return rc;
    if ((rc = copy_vec(m, has_bias ? s.ln_2_b : nullptr, C, &d.ln2_b))) return rc;
    if ((rc = copy_mat(m, s.c_fc_w, 4 * C * C, &d.fc_w))) return rc;
    if ((rc = copy_vec(m, has_bias ? s.c_fc_b : nullptr, 4 * C, &d.fc_b))) return rc;
    if ((rc = copy_mat(m, s.mlp_proj_w, 4 * C * C, &d.mproj_w))) return rc;
    if ((rc = copy_vec(m, has_bias ? s.mlp_proj_b : nullptr, C, &d.mproj_b))) return rc;
  }

  // KV cache and activations
  const size_t rows = std::max<size_t>(Bm * blk, 2 * Bm);
  if (!(m->kv = m->alloc_bytes(static_cast<size_t>(m->L > 0 ? m->L : 1) * 2 * m->cache_layer_bytes(), &rc))) return rc;
  CK(cudaMemsetAsync(m->kv, 0, static_cast<size_t>(m->L > 0 ? m->L : 1) * 2 * m->cache_layer_bytes(), m->stream));
  if (!(m->x = m->alloc<float>(rows * C, &rc))) return rc;
  if (!(m->xn = m->alloc_bytes(rows * C * m->esz, &rc))) return rc;
  if (!(m->q = m->alloc_bytes(rows * C * m->esz, &rc))) return rc;
  if (!(m->y = m->alloc_bytes(rows * C * m->esz, &rc))) return rc;
  if (!(m->h = m->alloc_bytes(rows * 4 * C * m->esz, &rc))) return rc;
  if (!(m->xf = m->alloc_bytes(2 * Bm * C * m->esz, &rc))) return rc;
  if (!(m->logits = m->alloc<float>(Bm * V, &rc))) return rc;
  // split-K / split-KV scratch: enough for a decode step at max_batch with up to 16 splits
  m->ws_bytes = std::max<size_t>(16 * Bm * 4 * C * sizeof(float), Bm * m->nh * 32 * (m->hs + 2) * sizeof(float));
  if (!(m->ws = m->alloc<float>(m->ws_bytes / sizeof(float), &rc))) return rc;
  m->n_tickets = std::max<size_t>(4096, Bm * m->nh);
  if (!(m->tickets = m->alloc<unsigned int>(m->n_tickets, &rc))) return rc;
  CK(cudaMemsetAsync(m->tickets, 0, m->n_tickets * sizeof(unsigned int), m->stream));
  if (!(m->d_err = m->alloc<int>(4, &rc))) return rc;
  m->d_pos = m->d_err + 1;
  m->d_step = m->d_err + 2;
  CK(cudaMemsetAsync(m->d_err, 0, 4 * sizeof(int), m->stream));
  if (!(m->d_tokens = m->alloc<int>(Bm, &rc))) return rc;
  if (!(m->d_lens = m->alloc<int>(Bm, &rc))) return rc;
  if (m->paged) {
    m->pages_per_seq = (m->block + m->page_size - 1) / m->page_size;
    m->h_table.assign(static_cast<size_t>(Bm) * m->pages_per_seq, -1);
    if (!(m->d_table = m->alloc<int>(m->h_table.size(), &rc))) return rc;
    CK(cudaMemcpyAsync(m->d_table, m->h_table.data(), m->h_table.size() * sizeof(int), cudaMemcpyHostToDevice,
                       m->stream));
    m->free_pages.clear();
    for (int pg = m->n_pages - 1; pg >= 0; --pg) m->free_pages.push_back(pg);
  }
  if (!(m->xlast = m->alloc<float>(Bm * C, &rc))) return rc;
  CK(cudaStreamSynchronize(m->stream));
  return GPT_OK;
}

}  // namespace

// ====================================================================== C ABI

namespace {
// One CTA waits on an mbarrier, with the bounded wait every pipeline in the library uses, for
// at most limit_ns; arrive = 0 leaves the barrier without an arrival, so the wait runs out.
__global__ void wait_probe_kernel(unsigned long long limit_ns, int arrive, int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (arrive) mbar_arrive(&bar);
    mbar_wait_limit(&bar, 0, err, limit_ns);
  }
}

// The stand-alone decode attention (gpt_attention_decode and its no-allocation variant) on a
// contiguous cache [B][n_head][block][head_size], with the caller's scratch.
int launch_attn_decode_any(const void* q, const void* k_cache, const void* v_cache, int dtype, int B, int n_head,
                           int head_size, int block, const int* pos0_dev, int splits, void* y, void* y_lo, float* ws,
                           unsigned int* tickets, int* err, cudaStream_t st) {
  const int C = head_size * n_head, rows = B * n_head;
  const KvLayout kv{n_head, block};
  cudaError_t e;
  if (dtype == GPT_DTYPE_BF16) {
    const bf16 *qq = static_cast<const bf16*>(q), *kk = static_cast<const bf16*>(k_cache),
               *vv = static_cast<const bf16*>(v_cache);
    bf16 *yy = static_cast<bf16*>(y), *yl = static_cast<bf16*>(y_lo);
    e = head_size == 64 ? launch_dec_attn<bf16, 64, false>(rows, splits, st, qq, kk, vv, kv, n_head, block, pos0_dev,
                                                           nullptr, ws, tickets, yy, yl, C, err)
                        : launch_dec_attn<bf16, 32, false>(rows, splits, st, qq, kk, vv, kv, n_head, block, pos0_dev,
                                                           nullptr, ws, tickets, yy, yl, C, err);
  } else {
    const float *qq = static_cast<const float*>(q), *kk = static_cast<const float*>(k_cache),
                *vv = static_cast<const float*>(v_cache);
    float* yy = static_cast<float*>(y);
    e = head_size == 64 ? launch_dec_attn<float, 64, false>(rows, splits, st, qq, kk, vv, kv, n_head, block, pos0_dev,
                                                            nullptr, ws, tickets, yy, nullptr, C, err)
                        : launch_dec_attn<float, 32, false>(rows, splits, st, qq, kk, vv, kv, n_head, block, pos0_dev,
                                                            nullptr, ws, tickets, yy, nullptr, C, err);
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
  return GPT_OK;
}

// Pointer alignment the stand-alone entry points check before any launch (their kernels use
// vector loads and stores of that width).
bool aligned(const void* p, uintptr_t bytes) { return reinterpret_cast<uintptr_t>(p) % bytes == 0; }
}  // namespace

extern "C" {

const char* gpt_strerror(int code) {
  switch (code) {
    case GPT_OK: return "ok";
    case GPT_EINVAL: return "invalid argument";
    case GPT_ECONTEXT: return "context overflow: cache length + new tokens > block_size";
    case GPT_ECUDA: return "CUDA error";
    case GPT_ENOMEM: return "out of device memory";
    case GPT_ETOKEN: return "token id out of range";
    case GPT_ETIMEOUT: return "a kernel pipeline wait timed out";
    case GPT_EPOSITION: return "position beyond block_size";
    case GPT_EUNSUPPORTED: return "unsupported device or driver";
    case GPT_ESTATE: return "call out of order";
    case GPT_ETOOBIG: return "request exceeds the fixed scratch of the no-allocation entry point";
    default: return "unknown error";
  }
}

const char* gpt_last_error_detail(void) { return g_detail.c_str(); }

int gpt_create(const gpt_config_t* cfg, const gpt_weights_t* weights, void* stream, gpt_model_t** out) {
  if (!out) return GPT_EINVAL;
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc) return rc;
  if (!weights || !weights->wte || !weights->wpe || !weights->ln_f_w || (cfg->n_layer > 0 && !weights->layers))
    return GPT_EINVAL;
  if ((cfg->bias == 1) != (weights->ln_f_b != nullptr)) return GPT_EINVAL;
  for (int l = 0; l < cfg->n_layer; ++l) {
    const gpt_layer_weights_t& s = weights->layers[l];
    if (!s.ln_1_w || !s.c_attn_w || !s.attn_proj_w || !s.ln_2_w || !s.c_fc_w || !s.mlp_proj_w) return GPT_EINVAL;
    const bool all = s.ln_1_b && s.c_attn_b && s.attn_proj_b && s.ln_2_b && s.c_fc_b && s.mlp_proj_b;
    const bool none = !s.ln_1_b && !s.c_attn_b && !s.attn_proj_b && !s.ln_2_b && !s.c_fc_b && !s.mlp_proj_b;
    if (cfg->bias == 1 ? !all : !none) return GPT_EINVAL;
  }
  gpt_model* m = new gpt_model();
  if (g_paged_request.paged) {
    m->paged = true;
    m->page_size = g_paged_request.page_size;
    m->n_pages = g_paged_request.n_pages;
    m->page_shift = 0;
    while ((1 << m->page_shift) < m->page_size) ++m->page_shift;
  }
  rc = create_impl(cfg, weights, stream, m);
  if (rc) {
    free_model(m);
    return rc;
  }
  *out = m;
  return GPT_OK;
}

int gpt_create_paged(const gpt_config_t* cfg, const gpt_weights_t* weights, void* stream, int32_t page_size,
                     int32_t n_pages, gpt_model_t** out) {
  if (!out) return GPT_EINVAL;
  *out = nullptr;
  if (page_size < 64 || page_size > 4096 || (page_size & (page_size - 1)) != 0 || n_pages < 1) return GPT_EINVAL;
  int rc = validate_config(cfg);
  if (rc) return rc;
  gpt_model_t* m = nullptr;
  // gpt_create validates the weights; the pool replaces the contiguous cache before it is allocated
  g_paged_request = {true, page_size, n_pages};
  rc = gpt_create(cfg, weights, stream, &m);
  g_paged_request = {};
  if (rc) return rc;
  *out = m;
  return GPT_OK;
}

void gpt_destroy(gpt_model_t* model) { free_model(model); }

int32_t gpt_cache_length(const gpt_model_t* model) { return model ? model->cache_len : -1; }

int64_t gpt_kernel_launches(const gpt_model_t* model) { return model ? model->launches : -1; }

int gpt_prefill(gpt_model_t* m, const int32_t* tokens, int32_t B, int32_t T, float* logits) {
  if (!m || !tokens || !logits || B < 1 || B > m->Bmax || T < 1) return GPT_EINVAL;
  if (T > m->block) return GPT_ECONTEXT;
  release_all_pages(m);
  m->batch = 0;  // until the prefill is enqueued
  int rc = ensure_pages(m, B, nullptr, T);
  if (rc) return rc;
  rc = forward(m, tokens, B, T, false, logits);
  if (rc) return rc;
  set_ints_kernel<<<1, 1, 0, m->stream>>>(m->d_pos, T, nullptr, 0);
  CK(cudaGetLastError());
  ++m->launches;
  m->cache_len = T;
  m->batch = B;
  m->ragged = false;
  return GPT_OK;
}

int gpt_prefill_ragged(gpt_model_t* m, const int32_t* tokens, const int32_t* lengths, int32_t B, int32_t T,
                       float* logits) {
  if (!m || !tokens || !lengths || !logits || B < 1 || B > m->Bmax || T < 1) return GPT_EINVAL;
  if (T > m->block) return GPT_ECONTEXT;
  int longest = 0;
  for (int b = 0; b < B; ++b) {
    if (lengths[b] < 1 || lengths[b] > T) return GPT_EINVAL;
    longest = std::max(longest, static_cast<int>(lengths[b]));
  }
  m->h_lens.assign(lengths, lengths + B);
  release_all_pages(m);
  m->batch = 0;  // until the prefill is enqueued
  int rc = ensure_pages(m, B, nullptr, T);  // the padding positions are written too
  if (rc) return rc;
  CK(cudaMemcpyAsync(m->d_lens, m->h_lens.data(), B * sizeof(int), cudaMemcpyHostToDevice, m->stream));
  rc = forward(m, tokens, B, T, false, logits, 0, T, m->d_lens);
  if (rc) return rc;
  CK(cudaStreamSynchronize(m->stream));  // h_lens is the source of the copy above until it lands
  m->cache_len = longest;
  m->batch = B;
  m->ragged = true;
  return GPT_OK;
}

int gpt_extend(gpt_model_t* m, const int32_t* tokens, int32_t T, float* logits) {
  if (!m || !tokens || !logits || T < 1) return GPT_EINVAL;
  if (m->batch < 1 || m->ragged) return GPT_ESTATE;
  if (static_cast<long long>(m->cache_len) + T > m->block) return GPT_ECONTEXT;
  const int off = m->cache_len;
  int rc = ensure_pages(m, m->batch, nullptr, off + T);
  if (rc) return rc;
  rc = forward(m, tokens, m->batch, T, false, logits, off);  // d_pos holds the cache length
  if (rc) return rc;
  set_ints_kernel<<<1, 1, 0, m->stream>>>(m->d_pos, off + T, nullptr, 0);
  CK(cudaGetLastError());
  ++m->launches;
  m->cache_len = off + T;
  return GPT_OK;
}

int gpt_decode_step(gpt_model_t* m, const int32_t* tokens, float* logits) {
  if (!m || !tokens || !logits) return GPT_EINVAL;
  if (m->batch < 1) return GPT_ESTATE;
  if (m->cache_len + 1 > m->block) return GPT_ECONTEXT;
  const int B = m->batch;
  int rc;
  if (m->ragged) {
    std::vector<int> next(m->h_lens);
    for (int& v : next) ++v;
    rc = ensure_pages(m, B, next.data(), 0);
  } else {
    rc = ensure_pages(m, B, nullptr, m->cache_len + 1);
  }
  if (rc) return rc;
  CK(cudaMemcpyAsync(m->d_tokens, tokens, B * sizeof(int), cudaMemcpyDeviceToDevice, m->stream));
  rc = decode_forward(m, m->d_tokens, B, logits);
  if (rc) return rc;
  if (m->ragged) {
    add_one_kernel<<<1, 128, 0, m->stream>>>(m->d_lens, B);
    for (int b = 0; b < B; ++b) ++m->h_lens[b];
  } else {
    set_ints_kernel<<<1, 1, 0, m->stream>>>(m->d_pos, m->cache_len + 1, nullptr, 0);
  }
  CK(cudaGetLastError());
  ++m->launches;
  m->cache_len += 1;
  return GPT_OK;
}

int gpt_generate(gpt_model_t* m, const int32_t* idx, int32_t B, int32_t T, int32_t max_new_tokens, float temperature,
                 int32_t top_k, uint64_t seed, int32_t* out) {
  if (!m || !idx || !out || B < 1 || B > m->Bmax || T < 1 || max_new_tokens < 1) return GPT_EINVAL;
  if (!(temperature >= 0.0f) || !std::isfinite(temperature)) return GPT_EINVAL;
  if (static_cast<long long>(T) + max_new_tokens > (1LL << 30)) return GPT_EINVAL;
  const int N = max_new_tokens, W = T + N;
  // Draw j sees the last min(T + j, block) tokens.  While they fit (T0 + j <= block, T0 the
  // cropped prompt) the KV cache serves it; after that every draw needs a forward pass over the
  // window of the last block tokens, whose positions restart at 0, so those run as prefills.
  const int T0 = std::min(T, m->block);
  const int n_cached = std::min(N, m->block - T0 + 1);
  m->timing_valid = false;
  release_all_pages(m);
  m->batch = 0;
  // every position any forward of this call writes: up to T0 + n_cached - 2, or the whole window
  int rc = ensure_pages(m, B, nullptr, n_cached < N ? m->block : T0 + n_cached - 1);
  if (rc) return rc;
  CK(cudaMemcpy2DAsync(out, W * sizeof(int), idx, T * sizeof(int), T * sizeof(int), B, cudaMemcpyDeviceToDevice,
                       m->stream));
  CK(cudaEventRecord(m->ev[0], m->stream));
  rc = forward(m, idx + (T - T0), B, T0, false, m->logits, 0, T);
  if (rc) return rc;
  set_ints_kernel<<<1, 1, 0, m->stream>>>(m->d_pos, T0, m->d_step, 1);
  CK(cudaGetLastError());
  ++m->launches;
  if ((rc = enqueue_sample(m, B, temperature, top_k, seed, nullptr, 0, out, W, T, m->stream))) return rc;
  CK(cudaEventRecord(m->ev[1], m->stream));
  m->cache_len = T0;
  m->batch = B;
  m->ragged = false;
  if (n_cached > 1) {
    GraphKey key;
    key.B = B;
    key.T = T;
    key.N = N;
    key.top_k = top_k;
    key.temperature = temperature;
    key.seed = seed;
    key.out = out;
    if (!m->gexec || !(m->gkey == key)) {
      if (m->gexec) {
        CK(cudaGraphExecDestroy(m->gexec));
        m->gexec = nullptr;
      }
      cudaStream_t saved = m->stream;
      const long long launches0 = m->launches;
      m->stream = m->cap_stream;
      CK(cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal));
      rc = decode_forward(m, m->d_tokens, B, m->logits);
      // after a join of two chains the sampler is an ordinary dependent
      if (!rc)
        rc = enqueue_sample(m, B, temperature, top_k, seed, m->d_step, 0, out, W, T, m->cap_stream,
                            !decode_multi_chain(m, B));
      if (!rc) {
        if (launch_k(advance_kernel, dim3(1), dim3(1), 0, m->cap_stream, true, m->d_pos, m->d_step) != cudaSuccess)
          rc = GPT_ECUDA;
        ++m->launches;
      }
      m->graph_kernels = m->launches - launches0;
      m->launches = launches0;
      cudaGraph_t graph = nullptr;
      cudaError_t ce = cudaStreamEndCapture(m->cap_stream, &graph);
      m->stream = saved;
      if (rc) {
        if (graph) cudaGraphDestroy(graph);
        return rc;
      }
      if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamEndCapture");
      ce = cudaGraphInstantiate(&m->gexec, graph, 0);
      cudaGraphDestroy(graph);
      if (ce != cudaSuccess) return cuda_fail(ce, "cudaGraphInstantiate");
      m->gkey = key;
    }
    for (int j = 1; j < n_cached; ++j) {
      CK(cudaGraphLaunch(m->gexec, m->stream));
      m->launches += m->graph_kernels;
    }
    m->cache_len = T0 + n_cached - 1;
  }
  // Past the cache: each draw j is a prefill of the window out[:, T + j - block, T + j).
  for (int j = n_cached; j < N; ++j) {
    rc = forward(m, out + (T + j - m->block), B, m->block, false, m->logits, 0, W);
    if (rc) return rc;
    if ((rc = enqueue_sample(m, B, temperature, top_k, seed, nullptr, j, out, W, T, m->stream))) return rc;
    m->cache_len = m->block;
  }
  if (n_cached < N) {
    set_ints_kernel<<<1, 1, 0, m->stream>>>(m->d_pos, m->block, nullptr, 0);
    CK(cudaGetLastError());
    ++m->launches;
  }
  CK(cudaEventRecord(m->ev[2], m->stream));
  m->timing_valid = true;
  return GPT_OK;
}

int gpt_last_timing(gpt_model_t* m, float* prefill_ms, float* decode_ms) {
  if (!m) return GPT_EINVAL;
  if (!m->timing_valid) return GPT_ESTATE;
  CK(cudaEventSynchronize(m->ev[2]));
  float a = 0.0f, b = 0.0f;
  CK(cudaEventElapsedTime(&a, m->ev[0], m->ev[1]));
  CK(cudaEventElapsedTime(&b, m->ev[1], m->ev[2]));
  if (prefill_ms) *prefill_ms = a;
  if (decode_ms) *decode_ms = b;
  return GPT_OK;
}

int gpt_profile_gemms(gpt_model_t* m, int32_t enable) {
  if (!m) return GPT_EINVAL;
  if (enable && m->prof_ev.empty()) {
    m->prof_ev.assign(8 * static_cast<size_t>(std::max(1, m->L)) + 8, nullptr);
    for (auto& e : m->prof_ev) CK(cudaEventCreate(&e));
  }
  m->prof_enabled = enable != 0;
  m->prof_n = 0;
  m->prof_flops = 0;
  return GPT_OK;
}

int gpt_gemm_timing(gpt_model_t* m, float* ms, double* flops) {
  if (!m) return GPT_EINVAL;
  if (m->prof_n == 0) return GPT_ESTATE;
  CK(cudaEventSynchronize(m->prof_ev[m->prof_n - 1]));
  float total = 0.0f;
  for (size_t i = 0; i + 1 < m->prof_n; i += 2) {
    float t = 0.0f;
    CK(cudaEventElapsedTime(&t, m->prof_ev[i], m->prof_ev[i + 1]));
    total += t;
  }
  if (ms) *ms = total;
  if (flops) *flops = m->prof_flops;
  return GPT_OK;
}

int gpt_sync_status(gpt_model_t* m) {
  if (!m) return GPT_EINVAL;
  CK(cudaStreamSynchronize(m->stream));
  int w = 0;
  CK(cudaMemcpy(&w, m->d_err, sizeof(int), cudaMemcpyDeviceToHost));
  const int zero = 0;
  CK(cudaMemcpy(m->d_err, &zero, sizeof(int), cudaMemcpyHostToDevice));
  return map_error_word(w);
}

// ------------------------------------------------------------------ stand-alone operations

int gpt_linear_bf16(const void* A, const void* W, const float* bias, float* out, int32_t M, int32_t N, int32_t K,
                    int32_t hilo, int32_t block_n, int32_t splits, void* stream) {
  if (!A || !W || !out || M < 1 || N < 1 || K < 64 || K % 64 != 0 || splits < 1) return GPT_EINVAL;
  if (!aligned(out, 16)) return GPT_EINVAL;  // 16-byte stores of output rows
  if (block_n != 0 && block_n != 64 && block_n != 128 && block_n != 256) return GPT_EINVAL;
  if (hilo && block_n == 256) return GPT_EINVAL;
  if (splits > 1 && N % 16 != 0) return GPT_EINVAL;
  int dev = 0;
  CK(cudaGetDevice(&dev));
  int num_sms = 148;
  CK(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev));
  if (block_n == 0 && splits == 1 && !hilo) {
    const int bnp = persist_bn(M, N, num_sms);
    if (bnp) {
      OpCtx* c = nullptr;
      int rc = op_ctx(&c, 0, 0);
      if (rc) return rc;
      CK(init_persist_attrs_once());
      CUtensorMap ta, tb;
      if ((rc = make_tmap(&ta, A, M, K, TC_BM))) return rc;
      if ((rc = make_tmap(&tb, W, N, K, bnp))) return rc;
      Epi<bf16> e;
      e.M = M;
      e.N = N;
      e.bias = bias;
      e.x = out;
      e.ldx = N;
      e.err = c->err;
      CK(launch_persist(bnp, EPI_F32, ta, tb, K, num_sms, e, static_cast<cudaStream_t>(stream)));
      return GPT_OK;
    }
  }
  GemmPlan p = plan_gemm(M, N, K, num_sms, hilo != 0, ~size_t(0));
  if (block_n) p.bn = block_n;
  p.splits = std::min(splits, K / TC_BK);
  p.splits = cdiv(K / TC_BK, cdiv(K / TC_BK, p.splits));
  OpCtx* c = nullptr;
  const size_t tiles = static_cast<size_t>(cdiv(M, TC_BM)) * cdiv(N, p.bn);
  int rc = op_ctx(&c, p.splits > 1 ? static_cast<size_t>(p.splits) * M * N * sizeof(float) : 256, tiles);
  if (rc) return rc;
  CUtensorMap ta, tb;
  if ((rc = make_tmap(&ta, A, hilo ? 2LL * M : M, K, TC_BM))) return rc;
  if ((rc = make_tmap(&tb, W, N, K, p.bn))) return rc;
  Epi<bf16> e;
  e.M = M;
  e.N = N;
  e.bias = bias;
  e.x = out;
  e.ldx = N;
  e.splits = p.splits;
  e.ws = c->ws;
  e.tickets = c->tickets;
  e.err = c->err;
  CK(dispatch_tc(p.bn, hilo != 0, EPI_F32, dev, ta, tb, M, N, K, p.splits, e, static_cast<cudaStream_t>(stream)));
  return GPT_OK;
}

int gpt_linear_decode_bf16(const void* A, const void* W, const float* bias, float* out, int32_t M, int32_t N,
                           int32_t K, int32_t splits, void* stream) {
  if (!A || !W || !out || M < 1 || M > DL_MAX_ROWS || N < 1 || K < 64 || K % 64 != 0 || splits < 0) return GPT_EINVAL;
  if (!aligned(out, 16)) return GPT_EINVAL;  // 16-byte stores of output rows
  const int kb = K / TC_BK;
  if (splits > 0 && ((splits & (splits - 1)) != 0 || splits > DL_MAX_SPLITS || splits > kb)) return GPT_EINVAL;
  int dev = 0;
  CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return GPT_EUNSUPPORTED;
  CK(init_dl_attrs(dev));
  int num_sms = 148;
  CK(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev));
  const int n_tiles = cdiv(N, 128);
  if (splits == 0) splits = plan_dl_splits(n_tiles, kb, M, num_sms, dev);
  if (splits > 1 && dl_max_clusters(dev, splits, dl_bp(M), dl_stages(kb, splits)) < 1) {
    g_detail = std::to_string(splits) + "-CTA clusters of this size cannot be scheduled on this device";
    return GPT_EUNSUPPORTED;
  }
  OpCtx* c = nullptr;
  int rc = op_ctx(&c, 0, 0);
  if (rc) return rc;
  CUtensorMap tx, tw;
  if ((rc = make_tmap(&tx, A, 2LL * M, K, dl_bp(M)))) return rc;
  if ((rc = make_tmap(&tw, W, N, K, 128))) return rc;
  Epi<bf16> e;
  e.M = M;
  e.N = N;
  e.bias = bias;
  e.x = out;
  e.ldx = N;
  e.err = c->err;
  CK(launch_dl(EPI_F32, tw, tx, kb, splits, dl_stages(kb, splits), n_tiles, e, false,
               static_cast<cudaStream_t>(stream)));
  return GPT_OK;
}

int gpt_layernorm_linear_decode_bf16(const float* x, int64_t x_stride, const float* gamma, const float* beta,
                                     const void* W, const float* bias, float* out, int32_t M, int32_t N, int32_t K,
                                     int32_t splits, void* stream) {
  if (!x || !gamma || !W || !out || M < 1 || M > DL_LN_MAX_ROWS || N < 1 || K < 64 || K % 64 != 0 ||
      K > 64 * LN_MAX_PAIRS || splits < 0 || x_stride < K || x_stride % 4 != 0)
    return GPT_EINVAL;
  // 16-byte loads of x, gamma and beta build the operand; 16-byte stores of output rows
  if (!aligned(x, 16) || !aligned(gamma, 16) || (beta && !aligned(beta, 16)) || !aligned(out, 16)) return GPT_EINVAL;
  const int kb = K / TC_BK;
  if (splits > 0 && ((splits & (splits - 1)) != 0 || splits > DL_MAX_SPLITS || splits > kb)) return GPT_EINVAL;
  int dev = 0;
  CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return GPT_EUNSUPPORTED;
  CK(init_dl_attrs(dev));
  int num_sms = 148;
  CK(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev));
  const int n_tiles = cdiv(N, 128);
  if (splits == 0) splits = plan_dl_splits(n_tiles, kb, M, num_sms, dev);
  if (splits > 1 && dl_max_clusters(dev, splits, dl_bp(M), dl_stages(kb, splits)) < 1) {
    g_detail = std::to_string(splits) + "-CTA clusters of this size cannot be scheduled on this device";
    return GPT_EUNSUPPORTED;
  }
  OpCtx* c = nullptr;
  int rc = op_ctx(&c, 0, 0);
  if (rc) return rc;
  CUtensorMap tw;
  if ((rc = make_tmap(&tw, W, N, K, 128))) return rc;
  Epi<bf16> e;
  e.M = M;
  e.N = N;
  e.bias = bias;
  e.x = out;
  e.ldx = N;
  e.err = c->err;
  e.ln_x = x;
  e.ln_ldx = x_stride;
  e.ln_g = gamma;
  e.ln_b = beta;
  // the operand is built in shared memory: the activation map is never loaded (W's map stands in)
  CK(launch_dl(EPI_F32, tw, tw, kb, splits, dl_stages(kb, splits), n_tiles, e, false,
               static_cast<cudaStream_t>(stream)));
  return GPT_OK;
}

int gpt_layernorm(const float* x, int64_t x_stride, const float* gamma, const float* beta, int32_t rows, int32_t C,
                  int32_t dtype, void* y, void* y_lo, void* stream) {
  if (!x || !gamma || !y || rows < 1 || C < 64 || C % 64 != 0 || C > 64 * LN_MAX_PAIRS || x_stride < C) return GPT_EINVAL;
  if (dtype != GPT_DTYPE_BF16 && dtype != GPT_DTYPE_F32) return GPT_EINVAL;
  if (y_lo && dtype != GPT_DTYPE_BF16) return GPT_EINVAL;
  // the kernel moves column pairs: 8-byte loads of x, gamma and beta, pair stores of y
  if (x_stride % 2 != 0 || !aligned(x, 8) || !aligned(gamma, 8) || (beta && !aligned(beta, 8)) ||
      !aligned(y, dtype == GPT_DTYPE_BF16 ? 4 : 8) || (y_lo && !aligned(y_lo, 4)))
    return GPT_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == GPT_DTYPE_BF16)
    CK(launch_ln<bf16>(rows, C, x_stride, x, gamma, beta, static_cast<bf16*>(y), static_cast<bf16*>(y_lo), C, st,
                       false));
  else
    CK(launch_ln<float>(rows, C, x_stride, x, gamma, beta, static_cast<float*>(y), static_cast<float*>(nullptr), C, st,
                        false));
  return GPT_OK;
}

int gpt_attention_prefill(const void* q, const void* k_cache, const void* v_cache, int32_t dtype, int32_t B,
                          int32_t n_head, int32_t head_size, int32_t T, int32_t block, int32_t pos0, void* y,
                          void* stream) {
  if (!q || !k_cache || !v_cache || !y || B < 1 || n_head < 1 || T < 1 || pos0 < 0 || pos0 + T > block)
    return GPT_EINVAL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16)) return GPT_EINVAL;  // 16-byte row loads
  if (head_size != 64 && !(head_size == 32 && dtype == GPT_DTYPE_F32)) return GPT_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int C = head_size * n_head;
  KvLayout kvl;
  kvl.nh = n_head;
  kvl.block = block;
  if (dtype == GPT_DTYPE_BF16) {
    if (!load_encode()) return GPT_EUNSUPPORTED;
    CK(init_attn_tc_once());
    OpCtx* ctx = nullptr;
    int rc = op_ctx(&ctx, 0, 0);
    if (rc) return rc;
    CUtensorMap tq, tk, tv;
    const long long rows = static_cast<long long>(B) * n_head * block;
    if ((rc = make_tmap(&tq, q, static_cast<long long>(B) * n_head * T, head_size, PT_BQ))) return rc;
    if ((rc = make_tmap(&tk, k_cache, rows, head_size, PT_BK))) return rc;
    if ((rc = make_tmap(&tv, v_cache, rows, head_size, PT_BK))) return rc;
    int dev = 0, sms = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int items = cdiv(T, PT_BQ) * B * n_head;
    attn_prefill_tc<<<std::min(items, PT_CTAS_PER_SM * sms), PT_THREADS, PT_SMEM, st>>>(
        tq, tk, tv, kvl, n_head, B * n_head, T, pos0, static_cast<bf16*>(y), C, ctx->err);
  } else if (dtype == GPT_DTYPE_F32) {
    if ((pos0 + T) * sizeof(float) > 48 * 1024) return GPT_EINVAL;
    auto kern = head_size == 64 ? attn_prefill_f32<64> : attn_prefill_f32<32>;
    kern<<<dim3(T, B * n_head), 32, (pos0 + T) * sizeof(float), st>>>(
        static_cast<const float*>(q), static_cast<const float*>(k_cache), static_cast<const float*>(v_cache), kvl,
        n_head, T, block, pos0, static_cast<float*>(y), C);
  } else {
    return GPT_EINVAL;
  }
  CK(cudaGetLastError());
  return GPT_OK;
}

int gpt_attention_decode(const void* q, const void* k_cache, const void* v_cache, int32_t dtype, int32_t B,
                         int32_t n_head, int32_t head_size, int32_t block, const int32_t* pos0_dev, int32_t splits,
                         void* y, void* y_lo, void* stream) {
  if (!q || !k_cache || !v_cache || !y || !pos0_dev || B < 1 || n_head < 1 || block < 1 || splits < 1 ||
      splits > 1024)
    return GPT_EINVAL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16)) return GPT_EINVAL;  // 16-byte row loads
  if (head_size != 64 && head_size != 32) return GPT_EINVAL;
  if (dtype != GPT_DTYPE_BF16 && dtype != GPT_DTYPE_F32) return GPT_EINVAL;
  if (y_lo && dtype != GPT_DTYPE_BF16) return GPT_EINVAL;
  const size_t pairs = static_cast<size_t>(B) * n_head;
  OpCtx* c = nullptr;
  int rc = op_ctx(&c, pairs * splits * (head_size + 2) * sizeof(float), pairs);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = launch_attn_decode_any(q, k_cache, v_cache, dtype, B, n_head, head_size, block, pos0_dev, splits, y, y_lo,
                              c->ws, c->tickets, c->err, st);
  if (rc) return rc;
  CK(cudaGetLastError());
  return GPT_OK;
}

int gpt_sample(const float* logits, int32_t B, int32_t V, float temperature, int32_t top_k, uint64_t seed,
               int32_t step, int32_t* tokens, float* thresholds, uint64_t* weights, void* stream) {
  if (!logits || !tokens || B < 1 || V < 1 || V > MAX_VOCAB || !(temperature >= 0.0f) || !std::isfinite(temperature))
    return GPT_EINVAL;
  int dev = 0;
  CK(cudaGetDevice(&dev));
  CK(set_sampler_smem(dev, V));
  SampleArgs a;
  a.logits = logits;
  a.ld = V;
  a.V = V;
  a.temperature = temperature;
  a.top_k = top_k;
  a.seed = seed;
  a.step_dev = nullptr;
  a.step = step;
  a.out = nullptr;
  a.out_stride = 0;
  a.out_col0 = 0;
  a.next_tokens = tokens;
  a.thr_out = thresholds;
  a.w_out = reinterpret_cast<unsigned long long*>(weights);
  a.cand_cap = sampler_cand_cap(V);
  sample_kernel<<<B, SMP_THREADS, sampler_smem(V), static_cast<cudaStream_t>(stream)>>>(a);
  CK(cudaGetLastError());
  return GPT_OK;
}

int gpt_op_status(void) {
  OpCtx* c = nullptr;
  int rc = op_ctx(&c, 0, 0);
  if (rc) return rc;
  CK(cudaDeviceSynchronize());
  int w = 0;
  CK(cudaMemcpy(&w, c->err, sizeof(int), cudaMemcpyDeviceToHost));
  const int zero = 0;
  CK(cudaMemcpy(c->err, &zero, sizeof(int), cudaMemcpyHostToDevice));
  return map_error_word(w);
}

// ------------------------------------------------------------------ failure-detection hooks

int gpt_debug_bounded_wait(int32_t limit_us, int32_t arrive, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return GPT_EINVAL;
  OpCtx* c = nullptr;
  int rc = op_ctx(&c, 0, 0);
  if (rc) return rc;
  wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned long long>(limit_us) * 1000ull, arrive ? 1 : 0, c->err);
  CK(cudaGetLastError());
  return GPT_OK;
}

int gpt_debug_fail_allocation(int32_t k) {
  if (k < 0) return GPT_EINVAL;
  g_fail_alloc_countdown.store(k);
  return GPT_OK;
}

// ------------------------------------------------------------------ decode attention without allocation
//
// For callers that must not allocate device memory: a host process whose allocator owns
// all of the GPU's memory (a framework's caching pool, a fixed budget in an embedded or
// multi-tenant server), or code that runs where cudaMalloc is not allowed or would stall
// the device.  The split-KV partial results and merge tickets of this variant live in one
// fixed array in device memory that the library holds for as long as it is loaded.

}  // extern "C"

namespace {

// Layout of the fixed scratch: [error word | pad to 256 B][tickets][split partials].
constexpr size_t NOALLOC_SCRATCH_BYTES = 4u << 20;  // 4 MiB on every GPU that loads the library
constexpr size_t NOALLOC_TICKET_OFFSET = 256;
constexpr size_t NOALLOC_MAX_PAIRS = 16384;  // batch x heads
constexpr size_t NOALLOC_PARTIAL_OFFSET = NOALLOC_TICKET_OFFSET + NOALLOC_MAX_PAIRS * sizeof(unsigned int);
constexpr size_t NOALLOC_PARTIAL_BYTES = NOALLOC_SCRATCH_BYTES - NOALLOC_PARTIAL_OFFSET;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch per device, looked up once with that device current.
unsigned char* g_noalloc_addr[64] = {};
std::mutex g_noalloc_mu;

// The cached address is that of the device's primary context when it was looked up: a
// cudaDeviceReset (or any reset of the primary context) leaves it stale.
int noalloc_scratch(unsigned char** out, cudaStream_t st) {
  int dev = 0;
  CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return GPT_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    // The look-up is not a stream operation; inside a stream capture it could invalidate the
    // capture, so a first call on a device while `st` is capturing is refused.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    CK(cudaStreamIsCapturing(st, &cs));
    if (cs != cudaStreamCaptureStatusNone) {
      g_detail = "gpt_attention_decode_noalloc: the first call on a device must come before any stream capture";
      return GPT_EUNSUPPORTED;
    }
    void* p = nullptr;
    CK(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    g_noalloc_addr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_noalloc_addr[dev];
  return GPT_OK;
}

}  // namespace

extern "C" {

int gpt_attention_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, int32_t dtype, int32_t B,
                                 int32_t n_head, int32_t head_size, int32_t block, const int32_t* pos0_dev,
                                 int32_t splits, void* y, void* y_lo, int32_t* err_dev, void* stream) {
  if (!q || !k_cache || !v_cache || !y || !pos0_dev || B < 1 || n_head < 1 || block < 1 || splits < 1 ||
      splits > 1024)
    return GPT_EINVAL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16)) return GPT_EINVAL;  // 16-byte row loads
  if (head_size != 64 && head_size != 32) return GPT_EINVAL;
  if (dtype != GPT_DTYPE_BF16 && dtype != GPT_DTYPE_F32) return GPT_EINVAL;
  if (y_lo && dtype != GPT_DTYPE_BF16) return GPT_EINVAL;
  const size_t pairs = static_cast<size_t>(B) * n_head;
  const size_t partial_bytes = pairs * splits * (head_size + 2) * sizeof(float);
  if (pairs > NOALLOC_MAX_PAIRS || (splits > 1 && partial_bytes > NOALLOC_PARTIAL_BYTES)) {
    g_detail = "gpt_attention_decode_noalloc: batch*heads = " + std::to_string(pairs) + " (max " +
               std::to_string(NOALLOC_MAX_PAIRS) + "), split partials " + std::to_string(partial_bytes) +
               " bytes (max " + std::to_string(NOALLOC_PARTIAL_BYTES) + ")";
    return GPT_ETOOBIG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned char* base = nullptr;
  int rc = noalloc_scratch(&base, st);
  if (rc) return rc;
  unsigned int* tickets = reinterpret_cast<unsigned int*>(base + NOALLOC_TICKET_OFFSET);
  float* ws = reinterpret_cast<float*>(base + NOALLOC_PARTIAL_OFFSET);
  int* err = err_dev ? err_dev : reinterpret_cast<int*>(base);
  // The array keeps whatever the previous call left: the merge tickets must start at zero.
  if (splits > 1) CK(cudaMemsetAsync(tickets, 0, pairs * sizeof(unsigned int), st));
  rc = launch_attn_decode_any(q, k_cache, v_cache, dtype, B, n_head, head_size, block, pos0_dev, splits, y, y_lo,
                              ws, tickets, err, st);
  if (rc) return rc;
  CK(cudaGetLastError());
  return GPT_OK;
}

}  // extern "C"
