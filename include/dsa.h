/*
 * dsa.h -- C ABI of libdsa, the GB300 (sm_103a) DSA sparse-attention hot path:
 * lightning-indexer scores -> per-query Top-K -> sparse MLA attention over the
 * selected latent-cache rows.
 *
 * Sources of each operation (page title, section):
 *  - "Day0 Inference Adaptation and Performance Optimization for Kimi K3.1 Pro",
 *    section 3: the indexer computes relevance scores between queries and
 *    historical positions, applies head-weight weighting and selects the Top-K
 *    positions, reading a paged cache; sparse flash attention then reads the KV
 *    rows of the selected positions.
 *  - "Large Language Model Inference Acceleration in Practice", section 1.2
 *    (DSA = MLA + LI + SFA; complexity O(N*K)) and section 3.1 (fused LI + SFA:
 *    indices feed SFA without a global round trip; rows read from the paged KV
 *    cache).
 *  - The score formula I[t,s] = sum_h w[t,h] * ReLU(q_I[t,h] . k_I[s]) with FP8
 *    keys and per-token scales, ties to the lower index, and the MQA form of the
 *    latent attention (576-d keys = 512 latent + 64 rope, 512-d values) follow
 *    the method's statement of the DSA path.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates or frees device memory; calls that need scratch take a
 *    caller-provided workspace (256-byte aligned) and report its size through
 *    the matching *_workspace_size() query.
 *  - Every call validates its arguments on the host, then enqueues its kernels
 *    on `stream` (a cudaStream_t; NULL = legacy default stream) and returns
 *    without synchronising.  Nothing is launched when validation fails.
 *  - Errors found on the device (out-of-range page ids or indices, q_pos beyond
 *    max_ctx, a wrong q_per_seq hint, a pipeline wait that timed out) never trap:
 *    the offending element is skipped and a sticky device status word is set;
 *    dsa_check_status() reads and clears it.
 *  - Calls are thread-safe; dsa_last_error()/dsa_last_plan() are per thread.
 *  - Base pointers must be 16-byte aligned.  Row-major, densely packed layouts
 *    unless a stride is given.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 1

typedef enum dsa_status {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad shape or stride      */
  DSA_ERR_UNSUPPORTED = 2,   /* no kernel for this dtype/dimension/K combination  */
  DSA_ERR_WORKSPACE = 3,     /* workspace missing or too small                    */
  DSA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed              */
  DSA_ERR_TIMEOUT = 5,       /* dsa_check_status: a device-side wait gave up      */
  DSA_ERR_DEVICE_CHECK = 6   /* dsa_check_status: a device-side bounds check hit, */
                             /* or a kernel could not run its launch layout      */
} dsa_status_t;

typedef enum dsa_dtype {
  DSA_F32 = 0,
  DSA_BF16 = 1,
  DSA_E4M3 = 2,              /* OCP FP8 E4M3 codes (bias 7, max 448, no inf)      */
  DSA_MXFP8_E4M3 = 3,        /* OCP MXFP8: E4M3 codes, one E8M0 scale byte         */
                             /* 2**(e - 127) per 32 consecutive elements (indexer  */
                             /* only)                                              */
  DSA_E4M3_T128 = 4          /* MLA cache only: 656-byte FP8 rows with one fp32    */
                             /* scale per 128 latent dims (layout below)           */
} dsa_dtype_t;

typedef void* dsa_stream_t;  /* cudaStream_t */

/* Queries, sequences and the paged cache they read.
 * Query t belongs to sequence q_seq[t] and sits at position q_pos[t]; its causal
 * history is the positions s in [0, q_pos[t]] (its own key already cached).
 * Logical position s of sequence b lives in cache row
 *     block_table[b * bt_stride + s / page_size] * page_size + s % page_size.
 * The indexer-key pool and the latent pool share this page table. */
typedef struct dsa_seq_desc {
  int32_t B;                 /* sequences                                          */
  int32_t T;                 /* query tokens (T >= 0)                              */
  int32_t max_ctx;           /* host bound: q_pos[t] + 1 <= max_ctx for every t;   */
                             /* sizes grids and score rows                          */
  int32_t q_per_seq;         /* > 0: sequence b owns queries [b*q_per_seq,          */
                             /* (b+1)*q_per_seq) (T == B*q_per_seq); 0: no layout   */
                             /* promise (each query handled on its own)             */
  const int32_t* q_seq;      /* device int32 [T]                                   */
  const int32_t* q_pos;      /* device int32 [T]                                   */
  const int32_t* block_table;/* device int32 [B, bt_stride] physical page ids      */
  int32_t bt_stride;         /* >= ceil(max_ctx / page_size)                       */
  int32_t page_size;         /* tokens per page (64 on the tensor-core paths)      */
  int64_t cache_rows;        /* rows in each pool; page ids must be < cache_rows / */
                             /* page_size                                          */
} dsa_seq_desc_t;

/* Lightning indexer inputs (dequantised value = code * scale).
 * "Day0 Inference Adaptation and Performance Optimization for Kimi K3.1 Pro",
 * section 4, and "Large Language Model Inference Acceleration in Practice",
 * section 4: FP8 index keys and queries, with MXFP8 (blocks of 32 sharing a
 * power-of-two scale) as the pages' own granularity.
 *   DSA_E4M3:       q_scale fp32 [T, H_I] (per query head), k_scale fp32
 *                   [cache_rows] (per key); either may be NULL for all-ones.
 *   DSA_MXFP8_E4M3: q_scale uint8 [T, H_I, D_I/32], k_scale uint8
 *                   [cache_rows, D_I/32]: E8M0 exponents, element i of a vector
 *                   is code * 2**(scale[i / 32] - 127); both required; D_I a
 *                   multiple of 32.
 *   DSA_F32:        q and k_cache hold fp32 values; scales as for DSA_E4M3. */
typedef struct dsa_indexer_desc {
  int32_t H_I;               /* indexer heads                                      */
  int32_t D_I;               /* indexer head dim                                   */
  dsa_dtype_t dtype;         /* DSA_E4M3, DSA_MXFP8_E4M3 or DSA_F32 (q and k_cache) */
  const void* q;             /* device [T, H_I, D_I]                               */
  const void* q_scale;       /* device query scales (layout by dtype, above)       */
  const float* w;            /* device fp32 [T, H_I] head weights                  */
  const void* k_cache;       /* device [cache_rows, D_I]                           */
  const void* k_scale;       /* device key scales (layout by dtype, above)         */
} dsa_indexer_desc_t;

/* MLA latent attention inputs (MQA form: one latent row per position, shared by
 * all H heads; keys are the first d_latent + d_rope values of a row, values the
 * first d_latent). */
typedef struct dsa_mla_desc {
  int32_t H;                 /* attention heads                                    */
  int32_t d_latent;          /* value dim (512 on the tensor-core path)            */
  int32_t d_rope;            /* extra key dims (64 on the tensor-core path)        */
  dsa_dtype_t dtype;         /* cache format:                                      */
                             /*  DSA_BF16: row = d_latent+d_rope bf16 values       */
                             /*  DSA_E4M3: 656-byte row (d_latent 512, d_rope 64): */
                             /*   [0,512) e4m3 latent codes, [512,516) fp32 scale, */
                             /*   [516,528) reserved, [528,656) 64 bf16 rope       */
                             /*  DSA_E4M3_T128: the same 656-byte row with four    */
                             /*   fp32 scales at [512,528), scale i for latent     */
                             /*   dims [128 i, 128 i + 128) ("per-token-tile-128", */
                             /*   "Large Language Model Inference Acceleration in  */
                             /*   Practice" section 4).  The tensor-core path      */
                             /*   widens code * scale to bf16: exact when every    */
                             /*   scale is a power of two (as the cache writer     */
                             /*   produces them), rounded to bf16 otherwise.       */
                             /*  DSA_F32 : row = d_latent+d_rope fp32 values       */
  const void* q;             /* device [T, H, d_latent+d_rope]: bf16, or fp32 when */
                             /* dtype == DSA_F32                                   */
  const void* kv_cache;      /* device [cache_rows, row_bytes]                     */
  int64_t row_bytes;         /* bytes per cache row (multiple of 16)               */
  float softmax_scale;       /* logit = softmax_scale * q . key                    */
} dsa_mla_desc_t;

int dsa_abi_version(void);
const char* dsa_status_string(dsa_status_t status);
/* Detail of the last failure on the calling thread ("" if none). */
const char* dsa_last_error(void);
/* Kernels chosen by the last successful compute call on the calling thread. */
const char* dsa_last_plan(void);

/* Step 1 -- lightning-indexer scores.
 * scores[t * ld + s] = sum_h w[t,h] * ReLU(q_I[t,h] . k_I[s]) for s <= q_pos[t],
 * accumulated in fp32 from the dequantised FP8 (or fp32) values.  Entries with
 * s > q_pos[t] are not written.  scores: device fp32 [T, ld], ld >= max_ctx,
 * ld % 4 == 0. */
dsa_status_t dsa_indexer_scores(const dsa_seq_desc_t* seq, const dsa_indexer_desc_t* idx,
                                 float* scores, int64_t ld, dsa_stream_t stream);

/* Step 2 -- per-query Top-K.
 * idx[t * K + j]: the min(K, q_pos[t]+1) positions s <= q_pos[t] with the largest
 * scores[t * ld + s] (compared as fp32 values, -0 == +0), ties to the lower s,
 * written in ascending position order, then -1 padding up to K.
 * K >= 1; scores: device fp32 [T, ld], ld >= max_ctx, ld % 4 == 0;
 * idx: device int32 [T, K]. */
dsa_status_t dsa_topk(const dsa_seq_desc_t* seq, const float* scores, int64_t ld, int32_t K,
                      int32_t* idx, dsa_stream_t stream);

/* Step 3 -- sparse MLA attention over the selected rows.
 * For query t and head h, over S = { idx[t*K + j] : idx >= 0 }:
 *   logit_s = softmax_scale * q[t,h,:] . row_s[0 : d_latent+d_rope]
 *   out[t,h,:] = sum_s softmax(logit)_s * row_s[0 : d_latent]
 *   lse[t,h]   = log sum_s exp(logit_s)      (natural log; -inf if S is empty)
 * Entries -1 are skipped wherever they appear; an entry > q_pos[t] is skipped and
 * flagged.  1 <= K <= 16384.  out: device [T, H, d_latent], bf16 (fp32 when dtype == DSA_F32);
 * lse: device fp32 [T, H] or NULL.  workspace may be NULL when
 * dsa_sparse_mla_attn_workspace_size() returns 0; a larger workspace lets the
 * call split each query's rows across more CTAs. */
size_t dsa_sparse_mla_attn_workspace_size(const dsa_seq_desc_t* seq, const dsa_mla_desc_t* mla,
                                          int32_t K);
dsa_status_t dsa_sparse_mla_attn(const dsa_seq_desc_t* seq, const dsa_mla_desc_t* mla,
                                 const int32_t* idx, int32_t K, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, dsa_stream_t stream);

/* Steps 1-3 chained for one decode (or prefill) step: scores stay in the
 * workspace (L2-resident at decode sizes) and feed Top-K, whose indices feed
 * the attention directly.  idx_out (device int32 [T, K]) receives the selected
 * positions when non-NULL.  workspace: >= dsa_decode_workspace_size() bytes. */
size_t dsa_decode_workspace_size(const dsa_seq_desc_t* seq, const dsa_indexer_desc_t* idx,
                                 const dsa_mla_desc_t* mla, int32_t K);
dsa_status_t dsa_decode_step(const dsa_seq_desc_t* seq, const dsa_indexer_desc_t* idx,
                             const dsa_mla_desc_t* mla, int32_t K, void* out, float* lse,
                             int32_t* idx_out, void* workspace, size_t workspace_bytes,
                             dsa_stream_t stream);

/* The decode step with its scratch memory in a device array the library owns,
 * for callers that cannot allocate device memory (for example a plugin inside
 * an engine that owns all device memory and offers plugins no allocator, or a
 * caller whose memory pool is fixed at start-up).  The method itself has no
 * counterpart to this call: it is the same computation as dsa_decode_step, with
 * `workspace` replaced by the library's array.
 *  - Inputs and outputs are the caller's, exactly as for dsa_decode_step.
 *  - DSA_STATIC_WORKSPACE_BYTES of device memory stay reserved on every GPU that
 *    loads the library until the process exits.
 *  - The first call on a device looks up that device's address of the array;
 *    make it before starting any stream capture on that device.
 *  - A step needing more scratch than DSA_STATIC_WORKSPACE_BYTES (see
 *    dsa_decode_workspace_size) fails with DSA_ERR_WORKSPACE.  The call never
 *    allocates device memory.
 *  - All calls share the array and it keeps the last call's contents (the step
 *    needs none of it zeroed).  Calls that overlap on the GPU -- on two streams or
 *    from two host threads -- race on the array: serialise them. */
#define DSA_STATIC_WORKSPACE_BYTES (32ull << 20)
dsa_status_t dsa_decode_step_static_ws(const dsa_seq_desc_t* seq, const dsa_indexer_desc_t* idx,
                                       const dsa_mla_desc_t* mla, int32_t K, void* out, float* lse,
                                       int32_t* idx_out, dsa_stream_t stream);

/* Cache writers -- the prolog side of a step: new tokens into the paged caches.
 * "Large Language Model Inference Acceleration in Practice", section 3.2 (the
 * indexer prolog normalises K and updates the key cache) and section 4 (FP8
 * index keys and KV cache); "Day0 Inference Adaptation and Performance
 * Optimization for Kimi K3.1 Pro", section 4.  New token t goes to the cache
 * row of position q_pos[t] in sequence q_seq[t] (page table as above); the
 * positions of one call must be distinct.  A position or page out of range is
 * skipped and flagged (dsa_check_status).
 *
 * Index keys: k_new device [T, D_I] fp32 or bf16 (src_dtype); per token
 *   scale = amax_i |k_new[t,i]| / 448 in fp32 (1 when the row is all zero),
 *   code_i = the E4M3 value nearest to k_new[t,i] / scale (fp32 quotient), ties
 *   to the even code, magnitudes beyond 448 saturated;
 *   writes k_cache[row, 0:D_I] (uint8, row stride D_I) and k_scale[row] (fp32),
 *   the formats dsa_indexer_scores reads.  4 <= D_I <= 1024, D_I % 4 == 0. */
dsa_status_t dsa_index_cache_append(const dsa_seq_desc_t* seq, int32_t D_I, dsa_dtype_t src_dtype,
                                    const void* k_new, uint8_t* k_cache, float* k_scale, dsa_stream_t stream);
/* MXFP8 index keys (the DSA_MXFP8_E4M3 format dsa_indexer_scores reads): as
 *   above, but every block of 32 consecutive values b gets its own E8M0 byte
 *   k_exp[row, b] = x_b + 127, x_b = floor(log2 max_i |k_new[t, 32 b + i]|) - 8
 *   (8 is the exponent of E4M3's largest normal, 448 = 1.75 * 2**8; -127 for an
 *   all-zero block; clamped to [-127, 127]), and code_i = the E4M3 value nearest
 *   to k_new[t, i] * 2**-x_b (an exact quotient), ties to even, saturated to
 *   +-448.  k_exp: device uint8 [cache_rows, D_I / 32].  32 <= D_I <= 1024,
 *   D_I % 32 == 0; k_new, k_cache and k_exp 16-byte aligned. */
dsa_status_t dsa_index_cache_append_mx(const dsa_seq_desc_t* seq, int32_t D_I, dsa_dtype_t src_dtype,
                                       const void* k_new, uint8_t* k_cache, uint8_t* k_exp, dsa_stream_t stream);
/* Latent rows: kv_new device [T, d_latent + d_rope], bf16 (fp32 when
 *   mla->dtype == DSA_F32); mla gives d_latent, d_rope, the cache dtype and
 *   row_bytes (its q and kv_cache fields are not used); the rows are written to
 *   kv_cache:
 *    DSA_BF16 / DSA_F32: the row copied (its byte size and row_bytes multiples of 16);
 *    DSA_E4M3 (656-byte rows, 512 + 64): the 512 latent values quantised as one
 *      vector by the rule above into [0,512), the fp32 scale at [512,516), zero
 *      bytes at [516,528), the 64 bf16 rope values copied to [528,656);
 *    DSA_E4M3_T128 (656-byte rows, 512 + 64): each 128-value tile i of the latent
 *      part quantised with the exponent rule of dsa_index_cache_append_mx on
 *      128-value blocks, its scale 2**x_i stored as fp32 at [512 + 4 i, 516 + 4 i)
 *      (a power of two, so the attention kernel widens code * scale to bf16
 *      exactly), the rope copied to [528,656). */
dsa_status_t dsa_latent_cache_append(const dsa_seq_desc_t* seq, const dsa_mla_desc_t* mla, const void* kv_new,
                                     void* kv_cache, dsa_stream_t stream);

/* Testing aid for the failure-detection path; the pages have no counterpart.
 * Every pipeline wait in the kernels is bounded: a wait that gives up sets a
 * sticky device flag, every warp of the CTA leaves its loop, in-flight copies
 * and tensor-core work are drained, TMEM is freed and the kernel returns (no
 * trap, the context stays usable).  With enable != 0, launches of the
 * tensor-core attention kernel made after this call have one producer warp
 * withhold its arrival for the first tile of every CTA, so the tile never
 * counts as landed: the issuing warp's wait runs out after wait_limit_ns
 * (1 us .. 1 s) and dsa_check_status() then reports DSA_ERR_TIMEOUT.  Outputs
 * of those launches are undefined.  enable = 0 restores normal launches and the
 * 1 s bound.  Process-wide setting; returns DSA_ERR_INVALID_ARG for a bound
 * outside the range. */
dsa_status_t dsa_debug_withhold_arrival(int32_t enable, uint64_t wait_limit_ns);

/* The indexer prolog -- step 1's inputs made from the new tokens.
 * "Large Language Model Inference Acceleration in Practice", section 3.2
 * "Indexer Prolog": before the indexer runs, a query projection, a key
 * normalisation with the key-cache update, a query quantisation and a
 * head-weight projection (run there on three streams; here the projection tiles
 * of all three weights are one grid).  The pages give the steps, not formulas;
 * this library computes, per new token t (bf16 inputs and weights, fp32 sums):
 *   q[t] = W_q x_q[t]  as H_I heads of D_I = 128 values, each head quantised to
 *          E4M3 with scale amax / 448 (1 for an all-zero head), round to nearest
 *          even, saturated: q_codes [T, H_I, 128] (uint8) and q_scale [T, H_I]
 *          (fp32) -- dsa_indexer_desc_t's q and q_scale for DSA_E4M3;
 *   w[t] = W_w x[t]  -> w [T, H_I] fp32, the head weights;
 *   k[t] = (v - mean(v)) / sqrt(var(v) + 1e-6) * gamma + beta,  v = W_k x[t]
 *          (population variance over the 128 values), quantised like a query
 *          head and written to the index-key cache row of position q_pos[t] of
 *          sequence q_seq[t] (k_cache [cache_rows, 128], k_scale [cache_rows]),
 *          as dsa_index_cache_append does.  Bad positions / pages are skipped and
 *          flagged (dsa_check_status).
 * Layouts: x bf16 [T, d_model], x_q bf16 [T, d_q], W_q bf16 [H_I * 128, d_q],
 * W_k bf16 [128, d_model], W_w bf16 [H_I, d_model] (row = output feature,
 * input dims contiguous), gamma / beta fp32 [128].  D_I must be 128, 1 <= H_I
 * <= 128, d_model and d_q multiples of 64 (else DSA_ERR_UNSUPPORTED).  The call
 * uses a caller-provided workspace of dsa_indexer_prolog_workspace_size() bytes
 * (the fp32 projections). */
typedef struct dsa_prolog_desc {
  int32_t d_model;           /* hidden size (multiple of 64)                       */
  int32_t d_q;               /* query latent size (multiple of 64)                 */
  int32_t H_I;               /* indexer heads (1 .. 128)                           */
  int32_t D_I;               /* indexer head dim (128)                             */
  const void* x;             /* device bf16 [T, d_model]                           */
  const void* x_q;           /* device bf16 [T, d_q]                               */
  const void* w_q;           /* device bf16 [H_I * D_I, d_q]                       */
  const void* w_k;           /* device bf16 [D_I, d_model]                         */
  const void* w_w;           /* device bf16 [H_I, d_model]                         */
  const float* gamma;        /* device fp32 [D_I]                                  */
  const float* beta;         /* device fp32 [D_I]                                  */
} dsa_prolog_desc_t;
size_t dsa_indexer_prolog_workspace_size(const dsa_seq_desc_t* seq, const dsa_prolog_desc_t* pd);
dsa_status_t dsa_indexer_prolog(const dsa_seq_desc_t* seq, const dsa_prolog_desc_t* pd, uint8_t* q_codes,
                                float* q_scale, float* w, uint8_t* k_cache, float* k_scale, void* workspace,
                                size_t workspace_bytes, dsa_stream_t stream);

/* Synchronises `stream`, then returns and clears the device status word:
 * DSA_OK, DSA_ERR_TIMEOUT or DSA_ERR_DEVICE_CHECK (dsa_last_error() names the
 * flags), or DSA_ERR_CUDA if the stream itself reports an error. */
dsa_status_t dsa_check_status(dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
