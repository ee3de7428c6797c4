/*
 * gpt.h -- C ABI of libgpt_b300.so: KV-cached GPT-2 generation on one B300 (sm_103a).
 *
 * The model is nanoGPT's GPT-2 decoder as the following pages describe it:
 *   "原生 nanoGPT 模型服务首选" (lzwjava.github.io): §1 LayerNorm(ndim, bias) with eps 1e-5 and
 *       an optional bias; §2 generate(idx, max_new_tokens, temperature, top_k); §"一个值得做的改进"
 *       the KV cache (keep past K/V, feed only the new token).
 *   "极速上手nanoGPT：从模型加载到文本生成的全流程SDK开发指南" (deepseek.csdn.net): §"GPTConfig类"
 *       (block_size, vocab_size, n_layer, n_head, n_embd, bias); §"注意力机制" (causal
 *       scaled-dot-product attention over (B, nh, T, hs)); §"关键参数" (temperature, top_k).
 *   "nanoGPT 架构分析" (wangbinyq.github.io), §4.1: pre-LN blocks, 4x GELU MLP, lm_head tied to
 *       wte and evaluated on the last position only.
 *   "第 4 章 模型构建" (aiknowledge.cn), §4.5: wte + wpe, lower-triangular mask, lm_head
 *       Linear(n_embd, vocab, bias=False).
 *
 * Conventions for every entry point:
 *   - Pointers marked (dev) are CUDA device pointers on the device that was current at
 *     gpt_create (or the current device, for the stand-alone operations); (host) are host
 *     pointers.  The caller owns every pointer it passes; the library never frees them.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls enqueue work on
 *     it and return without synchronising, except where a call says it synchronises.
 *   - Return value: GPT_OK (0) or a negative GPT_E* code.  Argument errors are detected on
 *     the host before anything is enqueued.  Errors found by kernels (bad token ids, a
 *     pipeline wait that timed out) are recorded in a device error word and reported by
 *     gpt_sync_status() / gpt_op_status(); kernels never trap.
 *   - Head size n_embd / n_head: 64 (every GPT-2 shape), or 32 for fp32 models.
 *   - The stand-alone operations check pointer alignment on the host (GPT_EINVAL otherwise):
 *     16 bytes for the operands their kernels move in 16-byte vectors (Linear outputs,
 *     attention q / k / v, the fused LayerNorm operand), as stated per entry point.
 *     Allocations from cudaMalloc or torch always qualify.
 */
#ifndef KVGPT_GPT_H
#define KVGPT_GPT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status codes */
#define GPT_OK 0
#define GPT_EINVAL (-1)       /* bad argument or configuration                         */
#define GPT_ECONTEXT (-2)     /* cache length + new tokens would exceed block_size      */
#define GPT_ECUDA (-3)        /* a CUDA runtime/driver call failed (gpt_last_error_detail) */
#define GPT_ENOMEM (-4)       /* device allocation failed                               */
#define GPT_ETOKEN (-5)       /* a kernel saw a token id outside [0, vocab_size)        */
#define GPT_ETIMEOUT (-6)     /* a kernel's bounded pipeline wait gave up               */
#define GPT_EPOSITION (-7)    /* a kernel saw a position >= block_size                  */
#define GPT_EUNSUPPORTED (-8) /* device is not sm_103, or a driver entry point is missing */
#define GPT_ESTATE (-9)       /* call out of order (e.g. decode before prefill)         */
#define GPT_ETOOBIG (-10)     /* request larger than gpt_attention_decode_noalloc's fixed scratch */

/* ------------------------------------------------------------------ types */
#define GPT_DTYPE_F32 0  /* weights, activations and cache in fp32 (exact fp32 kernels) */
#define GPT_DTYPE_BF16 1 /* weights and cache in bf16; fp32 accumulation, residual, logits */

/* Model shape: the GPTConfig fields, plus storage type and the largest batch served. */
typedef struct gpt_config {
  int32_t n_layer;
  int32_t n_head;
  int32_t n_embd;     /* multiple of 64, <= 2048; n_embd / n_head = 64 (or 32 with GPT_DTYPE_F32) */
  int32_t block_size; /* maximum context (positions 0 .. block_size-1) */
  int32_t vocab_size; /* 1 .. 57344 */
  int32_t bias;       /* 1: Linear and LayerNorm biases present; 0: bias=False */
  int32_t dtype;      /* GPT_DTYPE_F32 or GPT_DTYPE_BF16 */
  int32_t max_batch;  /* >= 1; the KV cache is sized for max_batch sequences */
} gpt_config_t;

/* One block's parameters, named as nanoGPT's state_dict.  (dev) pointers of the model's
 * dtype; Linear weights in nn.Linear layout (out_features, in_features), row-major.
 * Bias pointers must be NULL when bias == 0 and non-NULL when bias == 1. */
typedef struct gpt_layer_weights {
  const void* ln_1_w;      /* (C)        */
  const void* ln_1_b;      /* (C)        */
  const void* c_attn_w;    /* (3C, C): rows [0,C) q, [C,2C) k, [2C,3C) v; head h = 64 rows each */
  const void* c_attn_b;    /* (3C)       */
  const void* attn_proj_w; /* (C, C)     */
  const void* attn_proj_b; /* (C)        */
  const void* ln_2_w;      /* (C)        */
  const void* ln_2_b;      /* (C)        */
  const void* c_fc_w;      /* (4C, C)    */
  const void* c_fc_b;      /* (4C)       */
  const void* mlp_proj_w;  /* (C, 4C)    */
  const void* mlp_proj_b;  /* (C)        */
} gpt_layer_weights_t;

typedef struct gpt_weights {
  const void* wte;                   /* (V, C) token embedding; also the lm_head weight (tied) */
  const void* wpe;                   /* (block_size, C) position embedding */
  const void* ln_f_w;                /* (C) */
  const void* ln_f_b;                /* (C) or NULL when bias == 0 */
  const gpt_layer_weights_t* layers; /* (host) array of n_layer entries */
} gpt_weights_t;

typedef struct gpt_model gpt_model_t;

/* ------------------------------------------------------------------ model */

/* GPT(config) of the pages ("极速上手nanoGPT", §GPTConfig类: block_size, vocab_size, n_layer,
 * n_head, n_embd, bias; "nanoGPT 架构分析", §4.1: the modules and the wte / lm_head tying).
 * Validate `cfg`, copy the weights into library-owned device buffers, and allocate the KV
 * cache (n_layer x 2 x max_batch x n_head x block_size x 64 elements) and all scratch.
 * Keeps no caller pointer after it returns.  Synchronises `stream` once (weight copy).
 * Errors: GPT_EINVAL (bad cfg / weights), GPT_EUNSUPPORTED (not sm_103), GPT_ENOMEM,
 * GPT_ECUDA.  On error *out is NULL and nothing stays allocated. */
int gpt_create(const gpt_config_t* cfg, const gpt_weights_t* weights, void* stream, gpt_model_t** out);

/* gpt_create with a paged KV cache.  Instead of max_batch contiguous caches of block_size
 * positions, every layer's K and V live in n_pages pages of page_size positions (a power of
 * two, 64 .. 4096): [layer][k|v][page][head][page_size][head size].  Sequence b's positions
 * pos map to page table[b][pos / page_size]; the library fills a sequence's table as its cache
 * grows (gpt_prefill*, gpt_extend, gpt_decode_step, gpt_generate) and every prefill or generate
 * returns all pages to the pool first.  A call that needs more pages than are free returns
 * GPT_ENOMEM before anything is enqueued.  Results are identical to the contiguous cache.
 * Errors: as gpt_create, and GPT_EINVAL for a page_size or n_pages out of range. */
int gpt_create_paged(const gpt_config_t* cfg, const gpt_weights_t* weights, void* stream, int32_t page_size,
                     int32_t n_pages, gpt_model_t** out);

/* Release everything gpt_create allocated -- the weights, the KV cache the sketch of
 * "原生 nanoGPT 模型服务首选", §"一个值得做的改进" keeps between steps, and all scratch
 * (synchronises the model's stream first).  NULL is a no-op. */
void gpt_destroy(gpt_model_t* model);

/* Prefill from an empty cache: run the prompt tokens (dev, int32, B x T row-major) through
 * the model, write their K/V into cache positions 0..T-1, and write the last position's
 * logits (dev, fp32, B x vocab_size) -- the "forward on the last position only" of the
 * pages.  Afterwards the cache length is T for all B sequences.
 * Errors: GPT_EINVAL (B < 1, B > max_batch, T < 1, NULL pointers), GPT_ECONTEXT
 * (T > block_size), GPT_ECUDA. */
int gpt_prefill(gpt_model_t* model, const int32_t* tokens, int32_t B, int32_t T, float* logits);

/* Ragged prefill: sequence b has lengths[b] prompt tokens, the first lengths[b] entries of row b
 * of tokens (dev, int32, B x T row-major; entries past lengths[b] are ignored), lengths (host,
 * int32, B) with 1 <= lengths[b] <= T.  Writes each sequence's logits at its own last prompt
 * position (dev, fp32, B x vocab_size).  Afterwards sequence b's cache length is lengths[b], and
 * gpt_decode_step appends each sequence's token at its own length (its query sees keys
 * 0 .. its length); gpt_cache_length reports the longest.  gpt_extend is not available on a
 * ragged batch (GPT_ESTATE); the next gpt_prefill or gpt_generate ends ragged mode.
 * Synchronises the model's stream once (the lengths are copied to the device).
 * Errors: GPT_EINVAL (B, T or a length out of range, NULL pointers), GPT_ECONTEXT
 * (T > block_size), GPT_ECUDA. */
int gpt_prefill_ragged(gpt_model_t* model, const int32_t* tokens, const int32_t* lengths, int32_t B, int32_t T,
                       float* logits);

/* Chunked prefill into the existing cache: append T >= 1 tokens per sequence (tokens: dev,
 * int32, B x T row-major, B = the batch of the last prefill) at positions cache_len ..
 * cache_len + T - 1.  Query t attends to keys 0 .. cache_len + t: the causal mask offset by the
 * cache length (the sketch's `is_causal=(past_kv is None)` is exact only for one new token).
 * Writes the last new position's logits (dev, fp32, B x vocab_size); the cache length grows by T.
 * Runs the prefill kernels (tensor-core GEMMs over B x T rows, tiled attention with the offset).
 * Errors: GPT_ESTATE (no prefill yet), GPT_ECONTEXT (cache length + T > block_size), GPT_EINVAL. */
int gpt_extend(gpt_model_t* model, const int32_t* tokens, int32_t T, float* logits);

/* One KV-cached step, the forward(x, past_kv) of "原生 nanoGPT 模型服务首选",
 * §"一个值得做的改进": only the new token is fed, its K/V are appended to the cache and its
 * query attends to every cached key (no mask is needed for a single new token).
 * Append token tokens[b] (dev, int32, B = the prefill's batch) at position = current cache
 * length, and write that position's logits (dev, fp32, B x vocab_size).  The cache length
 * grows by one.
 * From 32 sequences up (bf16) the step runs as two chains of half the batch, the second on a
 * library-owned stream that waits on the model's stream and is joined back into it before
 * the call returns: the work is still ordered on the model's stream as for any other call.
 * Errors: GPT_ESTATE (no prefill yet), GPT_ECONTEXT (cache full), GPT_EINVAL, GPT_ECUDA. */
int gpt_decode_step(gpt_model_t* model, const int32_t* tokens, float* logits);

/* generate() with a KV cache: prefill `idx` (dev, int32, B x T), then draw max_new_tokens
 * tokens, feeding each one back through gpt_decode_step's computation.  `out` (dev, int32,
 * B x (T + max_new_tokens)) receives idx followed by the new tokens.
 * Sampling: temperature > 0 divides the logits, top_k > 0 keeps the min(top_k, V) largest
 * (ties with the k-th survive), then one draw per row from the softmax by the exact
 * integer inverse CDF with Philox4x64-10 (key = (seed, row), counter = (draw index, 0, 0,
 * 0)); temperature == 0 is greedy argmax (lowest index on ties).
 * Context: draw j conditions on the last min(T + j, block_size) tokens, as the pages'
 * generate() crops idx to its last block_size tokens.  While they fit in the cache the draws
 * run as one captured CUDA graph of a decode step, replayed; past that each draw is a prefill
 * of the window (positions restart at 0, so nothing can be reused), and a prompt longer than
 * block_size is cropped the same way.  Afterwards the cache holds the last forward's keys.
 * Errors: GPT_EINVAL (temperature < 0 or not finite, max_new_tokens < 1, B/T as for
 * prefill), GPT_ECUDA. */
int gpt_generate(gpt_model_t* model, const int32_t* idx, int32_t B, int32_t T, int32_t max_new_tokens,
                 float temperature, int32_t top_k, uint64_t seed, int32_t* out);

/* Device time of the last gpt_generate, split at the end of the prefill's draw
 * (CUDA events on the model's stream).  Synchronises on the events.  Either pointer may
 * be NULL.  GPT_ESTATE if no gpt_generate ran yet. */
int gpt_last_timing(gpt_model_t* model, float* prefill_ms, float* decode_ms);

/* GEMM timing of prefills, for profiling.  enable = 1: every later prefill (gpt_prefill, or the
 * prefill part of gpt_generate) records CUDA events on the model's stream around each of its
 * Linear-layer launches (the lm_head excluded); 0 stops it.  Decode steps are never timed. */
int gpt_profile_gemms(gpt_model_t* model, int32_t enable);

/* Summed device time (ms, from the events) and FLOPs (2 M N K each) of the Linear layers of the
 * last timed prefill.  Synchronises on its last event.  Either pointer may be NULL.
 * GPT_ESTATE if no prefill was timed. */
int gpt_gemm_timing(gpt_model_t* model, float* ms, double* flops);

/* Current cache length (host-side mirror; the longest sequence's after a ragged prefill), or -1
 * for NULL. */
int32_t gpt_cache_length(const gpt_model_t* model);

/* Number of kernels this model has enqueued since gpt_create (each replay of the decode
 * graph counts every kernel node in it), or -1 for NULL. */
int64_t gpt_kernel_launches(const gpt_model_t* model);

/* Synchronise the model's stream, then read and clear its device error word.
 * Returns GPT_OK, GPT_ETOKEN, GPT_ETIMEOUT, GPT_EPOSITION or GPT_ECUDA. */
int gpt_sync_status(gpt_model_t* model);

/* Static description of a code, never NULL. */
const char* gpt_strerror(int code);

/* The message of the last failing CUDA call in this thread ("" if none). */
const char* gpt_last_error_detail(void);

/* ------------------------------------------------------------------ stand-alone operations
 * The kernels the model runs, callable on caller buffers (tests and custom pipelines).
 * They use the current device; errors found by kernels go to a per-device word read by
 * gpt_op_status(). */

/* out (dev, fp32, M x N, row stride N) = A W^T (+ bias), on the tcgen05 tensor-core GEMM.
 * A (dev, bf16): M x K row-major, or with hilo=1 2M x K (rows [0,M) = hi, [M,2M) = lo parts
 * of one operand, both multiplied into the same fp32 accumulator).  W (dev, bf16): N x K
 * (nn.Linear layout).  bias (dev, fp32, N) or NULL.  K % 64 == 0, 1 <= M, N.
 * block_n: output tile width 64, 128 or 256 (256 not with hilo), or 0 = chosen by the library:
 * without hilo or split-K, and with at least one 128-row x 256 (N % 256 == 0) or x 128
 * (N % 128 == 0) tile per SM, the persistent kernel (one CTA per SM walking the tiles, two TMEM
 * accumulators so the epilogue of one tile overlaps the next tile's MMAs).
 * splits: split-K count >= 1 (needs N % 16 == 0 when > 1); partial sums go to library-owned
 * scratch and are added in split order, so results do not depend on CTA timing.
 * out 16-byte aligned. */
int gpt_linear_bf16(const void* A, const void* W, const float* bias, float* out, int32_t M, int32_t N,
                    int32_t K, int32_t hilo, int32_t block_n, int32_t splits, void* stream);

/* The decode-step Linear kernel: out (dev, fp32, M x N, row stride N) = A W^T (+ bias) for
 * 1 <= M <= 128 token rows given as a hi/lo pair.  A (dev, bf16): 2M x K, rows [0,M) = hi,
 * [M,2M) = lo parts of one operand, both multiplied into the same fp32 accumulator.  W (dev,
 * bf16): N x K (nn.Linear layout).  bias (dev, fp32, N) or NULL.  K % 64 == 0, N >= 1.
 * The weight rows are the tensor core's 128-row side; each 128-row tile's K range is split
 * over the CTAs of one thread-block cluster and reduced in split order through distributed
 * shared memory (deterministic, no scratch memory).  splits: 0 = chosen by the library, else
 * a power of two <= 16 and <= K/64 (16 needs 16-CTA clusters: GPT_EUNSUPPORTED where the
 * device cannot schedule them).  out 16-byte aligned. */
int gpt_linear_decode_bf16(const void* A, const void* W, const float* bias, float* out, int32_t M, int32_t N,
                           int32_t K, int32_t splits, void* stream);

/* The decode-step Linear kernel with the LayerNorm before it fused into its operand:
 * out (dev, fp32, M x N, row stride N) = LayerNorm(x) W^T (+ bias), eps 1e-5, biased variance,
 * the normalised rows carried as a bf16 hi/lo pair as in gpt_linear_decode_bf16.  This is how a
 * decode step of up to 8 sequences runs ln_1 + c_attn, ln_2 + c_fc and ln_f + lm_head
 * ("nanoGPT 架构分析", §4.1: pre-LN blocks).  Every CTA takes the whole rows' statistics and
 * normalises its own K-slice.  x (dev, fp32): M rows of K, row r at x + r * x_stride
 * (x_stride % 4 == 0, 16-byte aligned); 1 <= M <= 8; K <= 2048; gamma (dev, fp32, K) and beta
 * (dev, fp32, K, or NULL) 16-byte aligned; W, bias, splits as in gpt_linear_decode_bf16. */
int gpt_layernorm_linear_decode_bf16(const float* x, int64_t x_stride, const float* gamma, const float* beta,
                                     const void* W, const float* bias, float* out, int32_t M, int32_t N, int32_t K,
                                     int32_t splits, void* stream);

/* y (dev, dtype, rows x C) = LayerNorm(x) with eps 1e-5 and biased variance.
 * x (dev, fp32) row r at x + r * x_stride; gamma (dev, fp32, C); beta (dev, fp32, C) or NULL.
 * y_lo (dev, bf16) or NULL: receives y - bf16(y) (only with dtype == GPT_DTYPE_BF16).
 * C % 64 == 0 and C <= 2048.  The kernel moves column pairs: x_stride even, x, gamma and
 * beta 8-byte aligned, y 4-byte (bf16) or 8-byte (fp32) aligned, y_lo 4-byte aligned;
 * anything else is GPT_EINVAL. */
int gpt_layernorm(const float* x, int64_t x_stride, const float* gamma, const float* beta, int32_t rows, int32_t C,
                  int32_t dtype, void* y, void* y_lo, void* stream);

/* Causal attention of T new queries against a cache.  hs = head_size: 64, or 32 for fp32.
 * q (dev, dtype): B x n_head x T x hs.  k_cache, v_cache (dev, dtype): B x n_head x block x
 * hs, holding keys for positions 0 .. pos0+T-1.  Query t sits at position pos0 + t and sees
 * keys 0 .. pos0+t.  y (dev, dtype): (B*T) x (hs*n_head), row b*T + t, column h*hs + d.
 * bf16 runs on the tcgen05 tensor cores (S and O in TMEM, Q/K/V tiles by TMA), fp32 exactly
 * in fp32 (pos0 + T <= 12288).
 * q, k_cache and v_cache 16-byte aligned. */
int gpt_attention_prefill(const void* q, const void* k_cache, const void* v_cache, int32_t dtype, int32_t B,
                          int32_t n_head, int32_t head_size, int32_t T, int32_t block, int32_t pos0, void* y,
                          void* stream);

/* One new query per (b, h) against keys 0 .. *pos0_dev (the new token's key included).
 * head_size 32 or 64.  q (dev, dtype): B x n_head x hs; caches as above; pos0_dev (dev,
 * int32): cache length before the new token.  splits >= 1: the keys are split across that
 * many CTAs per (b, h) and merged by log-sum-exp in split order (library-owned scratch).
 * y (dev, dtype): B x (hs*n_head); y_lo (dev, bf16) or NULL receives y - bf16(y).
 * bf16 with head_size 64 and either splits = 1 and B * n_head <= 512, or splits <= 8 and
 * B * n_head <= 32, streams each (b, h)'s cache rows through shared memory with bulk copies,
 * whole stages of 64 keys per split (the decode step's kernel); other shapes use 16-byte
 * register loads.  q, k_cache and v_cache 16-byte aligned. */
int gpt_attention_decode(const void* q, const void* k_cache, const void* v_cache, int32_t dtype, int32_t B,
                         int32_t n_head, int32_t head_size, int32_t block, const int32_t* pos0_dev, int32_t splits,
                         void* y, void* y_lo, void* stream);

/* Temperature / top-k / softmax / draw on fp32 logits (dev, B x V, row stride V), exactly as
 * gpt_generate does, for draw index `step`.  tokens (dev, int32, B) receive the draws.
 * thresholds (dev, fp32, B) or NULL: the min(top_k, V)-th largest scaled logit (-inf when
 * top_k <= 0, i.e. no top-k).
 * weights (dev, uint64, B x V) or NULL: the integer weights floor(2^40 exp(s - max s)) of
 * the survivors (0 elsewhere).  V <= 57344. */
int gpt_sample(const float* logits, int32_t B, int32_t V, float temperature, int32_t top_k, uint64_t seed,
               int32_t step, int32_t* tokens, float* thresholds, uint64_t* weights, void* stream);

/* Synchronise the current device, then read and clear the stand-alone operations' error
 * word (codes as gpt_sync_status). */
int gpt_op_status(void);

/* ------------------------------------------------------------------ failure-detection hooks
 * Test hooks for the library's own error paths ("nanoGPT 架构分析", §9 总结与评价, 可改进之处:
 * the reference code has no error handling; these let a test reach each path without a GPU
 * fault). */

/* Launch one CTA that waits on a shared-memory mbarrier with the library's bounded wait, for at
 * most limit_us microseconds (1 .. 1,000,000).  arrive = 1: the CTA arrives first and the wait
 * succeeds at once; arrive = 0: nothing arrives, the wait runs out, the kernel records the
 * timeout in the stand-alone operations' error word and returns (gpt_op_status() then gives
 * GPT_ETIMEOUT).  The context stays usable.  Errors: GPT_EINVAL for limit_us out of range. */
int gpt_debug_bounded_wait(int32_t limit_us, int32_t arrive, void* stream);

/* Make the k-th next device allocation a model makes (gpt_create / gpt_create_paged, counted
 * across threads, process-wide) fail as if the device were out of memory; k = 0 turns the
 * injection off.  The create call then returns GPT_ENOMEM, leaves *out NULL and frees what it
 * had allocated.  Errors: GPT_EINVAL for k < 0. */
int gpt_debug_fail_allocation(int32_t k);

/* gpt_attention_decode for callers that cannot allocate device memory.  The pages have no
 * counterpart: this is a deployment variant, not a step of the method.
 *
 * Who needs it: a process whose device memory is owned by another allocator (a framework's
 * caching pool, a fixed per-tenant budget) and code that must not call cudaMalloc, which can
 * block on the device or be forbidden where the caller runs.  This call never allocates:
 * no cudaMalloc, cudaFree or allocating library routine.  Its split partials and merge
 * tickets live in one fixed 4 MiB array in device memory that the library keeps on every GPU
 * that loads it, until the process exits.
 *
 * Arguments and results are those of gpt_attention_decode, plus err_dev (dev, int32) or NULL:
 * error bits the kernel finds (a position at or beyond block) are OR-ed into *err_dev, in the
 * bit layout gpt_sync_status decodes (4 = position); with NULL they are dropped.
 * Limits: B * n_head <= 16384, and when splits > 1, B * n_head * splits * (head_size + 2) * 4
 * bytes must not exceed 4,128,512 (the 4 MiB array minus a 256-byte error-word header and
 * 16384 four-byte merge tickets); larger requests return GPT_ETOOBIG before anything is
 * enqueued (gpt_last_error_detail() gives the sizes).
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current and keeps it for the life of the process; make that first call before
 * any stream capture (a first call on a capturing stream returns GPT_EUNSUPPORTED), and make
 * no call after a cudaDeviceReset, which invalidates the kept address.  Every call shares the
 * array, which keeps the previous call's contents: the call clears the tickets it uses (an
 * asynchronous memset on `stream`), and calls whose kernels overlap on the same GPU (for
 * example on two streams) race on the array: the caller must serialise them. */
int gpt_attention_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, int32_t dtype, int32_t B,
                                 int32_t n_head, int32_t head_size, int32_t block, const int32_t* pos0_dev,
                                 int32_t splits, void* y, void* y_lo, int32_t* err_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVGPT_GPT_H */
