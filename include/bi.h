/*
 * bi.h — C ABI of libbi, the batch-invariant transformer forward for GB300 (sm_103a).
 *
 * "Batch invariant" means: the bits of any output row depend only on that row's
 * own inputs (and, for attention, on that request's KV length and contents),
 * never on how many other rows share the launch, what those rows hold, padding,
 * or how a prompt was chunked between prefill and decode.
 * Sources for the definitions (cited per call below):
 *   [TML-digest]  devpress.csdn digest of "Defeating Nondeterminism in LLM Inference",
 *                 section 2.3 (definition), 3.1 RMSNorm, 3.2 Matmul, 3.3 Attention
 *   [BI-notes]    "Batch-Invariant Kernel" reading notes (tom-jerr.github.io),
 *                 sections RMSNorm, GEMM, Flash Attention
 *   [BlockLock]   zhaixingw.cn post on BlockLock ("BlockLock 只锁住被保护的那条请求",
 *                 BlockLock-Rows; "坑清单": greedy decoding and top-20 logits)
 *
 * Conventions for every call
 *   - Pointers named as device pointers must be device memory of the current CUDA
 *     device, 16-byte aligned, owned by the caller.  The library never allocates
 *     on these paths; scratch memory ("workspace") is passed in by the caller,
 *     sized with the matching *_workspace() query.  A smaller workspace returns
 *     BI_ERR_WORKSPACE.
 *   - Every call is asynchronous on stream `s` (NULL = legacy default stream) and
 *     returns after enqueueing its kernels.  No call synchronises except
 *     bi_device_error().
 *   - Arguments are validated on the host before anything is launched; on an
 *     error nothing is launched and bi_last_error_message() says why.
 *     A failing launch returns BI_ERR_CUDA.
 *   - Kernels never trap.  Waits inside kernels are bounded; a wait that runs out
 *     sets a device error word read back by bi_device_error() (BI_ERR_TIMEOUT).
 *   - Modes: BI_MODE_INVARIANT uses the fixed reduction geometry for every row.
 *     BI_MODE_FAST lets the geometry follow the batch (split-row RMSNorm, split-K
 *     GEMM, occupancy-chosen split-KV count) exactly as the pages describe the
 *     non-invariant kernels; it exists to measure the cost of invariance and as
 *     a negative control.  BI_MODE_PROTECTED gives the rows of one target the
 *     INVARIANT geometry and lets all other rows take the FAST one, in the same
 *     launches (BlockLock-Rows style [BlockLock]).
 *     BI_MODE_INVARIANT_KSPLIT is INVARIANT with one change in the GEMM: the K
 *     range of every output element is cut into a fixed number of parts that
 *     depends on the weight shape (N, K) only, never on M, and the fp32 partials
 *     are added in part order ("Batch-Invariant Kernel" notes, section GEMM: a K
 *     split that depends on K alone keeps the matmul batch invariant).  Its bits
 *     are batch invariant but differ from INVARIANT's; all other ops are as
 *     INVARIANT.
 */
#ifndef BI_H_
#define BI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* bi_stream; /* a cudaStream_t */

typedef enum bi_status {
  BI_OK = 0,
  BI_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative or inconsistent size */
  BI_ERR_UNSUPPORTED = 2, /* a size or dtype outside what the kernels are built for */
  BI_ERR_WORKSPACE = 3,   /* workspace smaller than the *_workspace() query */
  BI_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a launch failed */
  BI_ERR_TIMEOUT = 5      /* a bounded in-kernel wait ran out (see bi_device_error) */
} bi_status;

typedef enum bi_mode {
  BI_MODE_INVARIANT = 0,
  BI_MODE_FAST = 1,
  BI_MODE_PROTECTED = 2,
  BI_MODE_INVARIANT_KSPLIT = 3
} bi_mode;

typedef enum bi_dtype { BI_F32 = 0, BI_BF16 = 1 } bi_dtype;

/* Fixed geometry constants of the invariant schedule. */
#define BI_SPLIT_TOKENS 256 /* split-KV size in absolute positions [TML-digest §3.3] */
#define BI_PAGE_SIZE 16     /* tokens per KV page */
#define BI_MERGE_DEPTH 16   /* merge-tree depth the merge supports: up to 2^16 splits */
#define BI_TOPK_MAX 32      /* largest k of bi_topk */

/* ------------------------------------------------------------------ misc */
const char* bi_status_string(bi_status st);
/* Detail of the last failing call on this host thread ("" if none). */
const char* bi_last_error_message(void);
int32_t bi_version(void);
/* Streaming-multiprocessor count of the current device (0 if none). */
int32_t bi_num_sms(void);
/* Reads and clears the device error words of all kernels (after synchronising
 * `s`).  *code = 0 when nothing was recorded, else the site code of the first
 * event recorded:
 *   1-4   GEMM: a bounded wait ran out (1 copy slot free, 2 accumulator free,
 *         3 copies landed, 4 accumulator ready)          -> BI_ERR_TIMEOUT
 *   11-15 attention: a bounded wait ran out              -> BI_ERR_TIMEOUT
 *   16    decode attention: a kv_len outside [0, max_pages*16]; it was clamped
 *   17    attention: a block-table entry outside [0, num_pages), or a position
 *         past the request's block-table row; page 0 was read instead
 *   18    decode attention: its dynamic shared memory did not start 1024-byte
 *         aligned, so nothing was computed              -> BI_ERR_UNSUPPORTED
 *   21    K/V store: a position past the block-table row or a page outside the
 *         cache; that token's K/V were not stored
 *   22    K/V store: a position outside the RoPE tables; the last row was used
 *                                                        -> BI_ERR_INVALID_ARG
 * (16, 17, 21, 22: the kernels check these device-side inputs so that no access
 * leaves the caller's buffers; the outputs of the affected rows are undefined.) */
bi_status bi_device_error(int32_t* code, bi_stream s);

/* Test hook for the failure path of the bounded in-kernel waits (the pages have
 * no counterpart).  Arms the next GEMM launch made by this host thread (bi_gemm,
 * bi_gemm_f32a, or a GEMM inside a layer or model call) so that CTA 0 issues no
 * copies for its first stage and every wait of that launch gives up after
 * wait_ns nanoseconds instead of 2 s.  The launch still ends on its own: the
 * wait for the missing stage runs out, all roles stop, copies in flight are
 * drained and tensor memory is freed; bi_device_error() then returns
 * BI_ERR_TIMEOUT with a GEMM site code.  That launch's output is undefined; the
 * next launch is unaffected.  wait_ns in [1e6, 2e9], else BI_ERR_INVALID_ARG. */
bi_status bi_debug_arm_gemm_stall(int64_t wait_ns);

/* Tuning of the non-invariant schedules (FAST mode; the pages have no
 * counterpart: it exists so that the cost of invariance can be measured
 * against the best non-invariant schedule these kernels offer).
 * bi_fast_gemm_plan: FAST GEMMs of shape (M, N, K) (bf16 or fp32 activations)
 * take INVARIANT's tile plan, with no split-K, when plan = 1; plan = 0 restores
 * FAST's own rule (split K over CTAs when there are fewer tiles than SMs).
 * bi_fast_attention_plan: plan = 1 makes FAST decode attention cut every request
 * into the 256-token splits of INVARIANT (combined left to right) instead of
 * the occupancy-chosen unit count of plan = 0.  Process-wide host-side settings
 * (bi_fast_gemm_plan keeps one entry per shape); they change no INVARIANT,
 * INVARIANT_KSPLIT or PROTECTED schedule.  Workspace queries made while a
 * setting is in force size for it.  Any other plan is BI_ERR_INVALID_ARG. */
bi_status bi_fast_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t plan);
bi_status bi_fast_attention_plan(int32_t plan);

/* Kernel timing (off by default).  bi_profile_start creates 2*max_launches CUDA
 * events up front; while it is on, every kernel launch of the library is
 * bracketed by two events recorded on the launching stream (launches beyond
 * max_launches are not timed).  bi_profile_stop stops recording.
 * bi_profile_read synchronises the recorded events and returns, for the kernel
 * named `kernel` (see bi_profile_kernel_name), the number of timed launches and
 * their summed duration in milliseconds.  Not for use inside stream capture. */
bi_status bi_profile_start(int32_t max_launches);
bi_status bi_profile_stop(void);
bi_status bi_profile_read(const char* kernel, int32_t* launches, double* total_ms);
/* Name of kernel tag i (0 <= i < bi_profile_kernel_count()), NULL otherwise. */
const char* bi_profile_kernel_name(int32_t i);
int32_t bi_profile_kernel_count(void);

/* ------------------------------------------------------------------ RMSNorm
 * y[r][j] = x[r][j] * (1 / sqrt(mean_j x[r][j]^2 + eps)) * gamma[j]
 *   [BI-notes "RMSNorm" formula; TML-digest §3.1; data-parallel reduction: one CTA
 *    owns a whole row, BI-notes "批次不变转换方案"]
 * x, y: device [rows][d] of `dtype` (row-major, contiguous); gamma: device [d] of
 * `dtype`.  fp32 math; the sum of squares is reduced in one fixed order that
 * depends on d only.  d must be a multiple of 8 (bf16) or 4 (f32), d <= 16384.
 * y may alias x.  rows == 0 is a no-op.
 * FAST: rows < #SMs splits each row over several CTAs (two passes through the
 * workspace).  PROTECTED: rows [target_row, target_row + target_count) take the
 * INVARIANT path, the rest FAST.
 */
size_t bi_rmsnorm_workspace(int64_t rows, int64_t d, bi_mode mode);
bi_status bi_rmsnorm(const void* x, const void* gamma, void* y, int64_t rows, int64_t d, bi_dtype dtype,
                     float eps, bi_mode mode, int32_t target_row, int32_t target_count, void* workspace,
                     size_t ws_bytes, bi_stream s);

/* ------------------------------------------------------------------ GEMM
 * C[i][j] = sum_k A[i][k] * W[j][k]  (+ residual[i][j])
 *   [TML-digest §3.2: pointwise products then a reduction over k; BI-notes "GEMM"]
 * A: device [M][K] bf16 row-major.  W: device [N][K] bf16 (the linear-layer
 * layout, K contiguous).  C: device [M][N] of `out_dtype` (bf16 or f32).
 * residual: NULL or device [M][N] bf16, added to the fp32 accumulator before the
 * single rounding to out_dtype (C may alias residual).
 * INVARIANT: tcgen05 tensor cores (M=128, K=16 instructions, bf16 in, fp32
 * accumulate in tensor memory), k-tiles of 64 consumed in ascending order, the
 * whole K range of an output element reduced by one CTA; nothing in that order
 * depends on M or N.  FAST: split-K chosen from the tile count and
 * the SM count (the non-invariant behaviour BI-notes "GEMM" describes).
 * PROTECTED: the 128-row tiles holding rows [target_row, target_row+target_count)
 * are never split; other tiles are as FAST.
 * INVARIANT_KSPLIT: the k-tiles (64 wide) are cut into S = bi_gemm_ksplit(N, K)
 * contiguous parts, part s holding k-tiles [floor(s*T/S), floor((s+1)*T/S)) of
 * the T = ceil(K/64); each part is accumulated from zero as above and the
 * result is ((0 + P_0) + P_1) + ... + P_{S-1} in fp32 (+ residual), rounded
 * once.  For M <= 128 the parts run on separate CTAs and a second pass adds
 * them (workspace S*M*N*4 bytes); for larger M one CTA computes the parts of a
 * tile in turn and keeps the running sum in tensor memory.  Both give the same
 * bits.  S = 1 gives exactly the INVARIANT result.
 * K must be a multiple of 8 and >= 8; M, N >= 0 (0 is a no-op); N multiple of 8.
 */
size_t bi_gemm_workspace(int64_t M, int64_t N, int64_t K, bi_mode mode);
/* The part count S of INVARIANT_KSPLIT for an N x K weight (1..16); a pure
 * function of (N, K). */
int32_t bi_gemm_ksplit(int64_t N, int64_t K);
bi_status bi_gemm(const void* A, const void* W, void* C, const void* residual, int64_t M, int64_t N, int64_t K,
                  bi_dtype out_dtype, bi_mode mode, int32_t target_row, int32_t target_count, void* workspace,
                  size_t ws_bytes, bi_stream s);

/* fp32 activations times bf16 weights (the mixed-precision mitigation the
 * TML-digest names in §2 and §6: weights stay 16-bit, activations fp32).
 * A: device [M][K] fp32.  W: device [N][K] bf16.  C: device [M][N] fp32.
 * residual: NULL or device [M][N] fp32 added before C is written (C may alias it).
 * Each fp32 A value is split into three bf16 values hi + mid + lo whose sum is
 * the value (exact for |a| >= 2^-110; below that the error is < 2^-133), and the
 * tensor cores reduce, per k16 step, hi*W, mid*W, lo*W in that order with exact
 * products and fp32 accumulation; otherwise the schedule and every mode are as
 * bi_gemm (same k order, same K-split rules).  The workspace holds the three
 * planes (3*M*K bf16) plus what the mode needs; size from
 * bi_gemm_f32a_workspace.  K, N multiples of 8; A, C, residual 16-byte aligned. */
size_t bi_gemm_f32a_workspace(int64_t M, int64_t N, int64_t K, bi_mode mode);
bi_status bi_gemm_f32a(const float* A, const void* W, float* C, const float* residual, int64_t M, int64_t N,
                       int64_t K, bi_mode mode, int32_t target_row, int32_t target_count, void* workspace,
                       size_t ws_bytes, bi_stream s);

/* ------------------------------------------------------------------ attention
 * Paged KV cache: k_cache and v_cache are device [num_pages][num_kv_heads][page_size][head_dim]
 * bf16 (page_size must be 16).  block_table: device int32 [B][max_pages];
 * entry i of row b names the physical page of tokens [16i, 16i+16) of request b.
 * Entries past a request's length are never read.
 * Query head h reads kv head h / (num_q_heads / num_kv_heads).  head_dim 64 or
 * 128; num_q_heads / num_kv_heads in {1, 2, 4}.
 * act_f32 (dims): 0 = q and out bf16; 1 = q and out fp32 (fp32-activation
 * layers; the cache stays bf16 and the arithmetic is the same).
 *
 * INVARIANT [TML-digest §3.3 fixed split size; BI-notes "Flash Attention"]: the
 * keys of a query at absolute position p are cut into fixed splits
 * [256s, 256s+256) ∩ [0, p]; each split is reduced at full width (masked lanes
 * contribute nothing) by one device function shared by decode and prefill;
 * split states (m, l, o) are combined by a pairwise tree over the split index
 * padded to a constant depth, in which an empty split is an exact identity.
 * Hence decode of the token at position p and any chunked prefill containing it
 * produce identical bits when the cached K/V bits are identical.
 * FAST: the split count follows batch size and SM count (split boundaries move
 * with the batch) and splits are merged left to right.  PROTECTED: request
 * `target_request` takes the INVARIANT geometry, the others FAST.
 */
typedef struct bi_attn_dims {
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size; /* must be BI_PAGE_SIZE */
  int32_t max_pages; /* row stride of block_table */
  int32_t num_pages; /* pages in each cache (for validation of the cache extent) */
  float scale;       /* score scale, normally 1/sqrt(head_dim) */
  int32_t act_f32;   /* 0: q and out bf16; 1: q and out fp32 */
} bi_attn_dims;

/* Decode: one query token per request.  q: device [B][num_q_heads][head_dim] bf16
 * (fp32 when dims->act_f32); the query of request b sits at position kv_lens[b]-1
 * and its own K/V must already be in the cache.  kv_lens: device int32 [B],
 * 1 <= kv_len <= max_pages*16 (a length outside [0, max_pages*16] is clamped and
 * reported by bi_device_error as site 16; block-table entries outside
 * [0, num_pages) are reported as site 17 and read as page 0).
 * out: device [B][num_q_heads][head_dim], as q. */
size_t bi_decode_attention_workspace(int32_t B, const bi_attn_dims* dims, bi_mode mode);
bi_status bi_decode_attention(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                              const int32_t* kv_lens, int32_t B, const bi_attn_dims* dims, void* out, bi_mode mode,
                              int32_t target_request, void* workspace, size_t ws_bytes, bi_stream s);

/* Decode attention for callers that cannot allocate device memory at call time
 * (for example a plugin inside a host framework whose caching allocator owns all
 * of the GPU's memory, or a serving loop that must never call cudaMalloc, which
 * can synchronise the device).  Same arguments, computation and bits as
 * bi_decode_attention, but no workspace: the scratch is a fixed 16 MiB array in
 * the library's own device data, which every GPU that loads the library holds
 * until the process exits.  The pages have no counterpart of this call.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device (and again in a new CUDA context of that
 *     device, e.g. after cudaDeviceReset) looks up the scratch array's device
 *     address (cudaGetSymbolAddress, with that device current) and caches it;
 *     make that first call before any stream capture.
 *   - Batches whose scratch need exceeds 16 MiB are rejected with
 *     BI_ERR_UNSUPPORTED and a message naming the need: U * (num_q_heads *
 *     (head_dim+2) + 1) * 4 bytes plus a few int32 per request, for U split units:
 *     INVARIANT U = B * ceil(max_pages*16/256); FAST U = B * f with
 *     f = min(64, ceil(4 * SMs / (B * num_kv_heads))); PROTECTED
 *     U = (B-1) * f + max(f, ceil(max_pages*16/256)).
 *   - All calls share the one array and each call writes every scratch byte it
 *     reads, so nothing needs clearing between calls; calls whose kernels
 *     overlap on the GPU (e.g. on two streams) race on the array and must be
 *     serialised by the caller. */
bi_status bi_decode_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_table, const int32_t* kv_lens, int32_t B,
                                      const bi_attn_dims* dims, void* out, bi_mode mode, int32_t target_request,
                                      bi_stream s);

/* Prefill (any number of query tokens per request, causal by absolute position).
 * q: device [T][num_q_heads][head_dim] bf16 (fp32 when dims->act_f32), tokens of request b at rows
 * q_start[b] .. q_start[b+1]-1 (q_start device int32 [B+1], q_start[0] = 0,
 * q_start[B] = T), at absolute positions q_pos0[b] + i (q_pos0 device int32 [B]).
 * K/V of every query token must already be in the cache.  out: as q. */
size_t bi_prefill_attention_workspace(int32_t B, int32_t T, const bi_attn_dims* dims, bi_mode mode);
bi_status bi_prefill_attention(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                               const int32_t* q_start, const int32_t* q_pos0, int32_t B, int32_t T,
                               const bi_attn_dims* dims, void* out, bi_mode mode, int32_t target_request,
                               void* workspace, size_t ws_bytes, bi_stream s);

/* ------------------------------------------------------------------ pointwise helpers
 * Pointwise ops act per element and are batch invariant as they stand [TML-digest §3]. */

/* out[t][:] = table[ids[t]][:]  (bf16, device).  ids outside [0, vocab) give a zero row. */
bi_status bi_embed(const int32_t* ids, const void* table, void* out, int64_t T, int64_t d, int64_t vocab,
                   bi_stream s);

/* RoPE tables: cos/sin[p][i] = cos/sin(p * theta^(-2i/head_dim)) rounded to fp32,
 * p < max_pos, i < head_dim/2, computed on the device in float64.
 * cos_out, sin_out: device float [max_pos][head_dim/2]. */
bi_status bi_rope_table(double theta, int32_t head_dim, int32_t max_pos, float* cos_out, float* sin_out,
                        bi_stream s);

/* Splits the fused QKV projection, rotates q and k (rotate-half pairs (i, i+hd/2)),
 * writes q_out [T][Hq][hd] and stores k, v of every token in the paged caches at
 * its absolute position.  qkv: device [T][(Hq+2Hkv)*hd] bf16 (q heads, then k
 * heads, then v heads).  token_pos/token_req: device int32 [T] (absolute position
 * and request of each token). */
bi_status bi_qkv_rope_store(const void* qkv, const float* rope_cos, const float* rope_sin, const int32_t* token_pos,
                            const int32_t* token_req, const int32_t* block_table, int32_t T,
                            const bi_attn_dims* dims, void* q_out, void* k_cache, void* v_cache, bi_stream s);

/* out[t][j] = bf16( silu(gu[t][j]) * gu[t][F + j] ), gu device [T][2F] bf16, out [T][F]. */
bi_status bi_swiglu(const void* gu, void* out, int64_t T, int64_t F, bi_stream s);

/* Gate|up projection followed by SwiGLU, as one call:
 *   act[m][j] = bi_swiglu of the bf16 result of bi_gemm(A, W_gate_up) (INVARIANT
 *   etc. as bi_gemm), i.e. bf16(silu(g) * u) with g = C[m][j], u = C[m][F + j]
 *   and C = A W_gate_up^T rounded to bf16.
 * A: device [M][K] bf16.  W_gate_up: device [2F][K] bf16, the F gate rows then
 * the F up rows.  act: device [M][F] bf16.  Same modes, targets and size rules
 * as bi_gemm (K, F multiples of 8; M = 0 or F = 0 is a no-op).
 * Where the plain [M][2F] GEMM's plan is one CTA per tile with the whole K range
 * (M <= 128 and no split), the SwiGLU runs in that GEMM's epilogue: each tile
 * reads gate and up rows of the same outputs and the [M][2F] product never
 * reaches memory.  Otherwise the call runs bi_gemm into the workspace and then
 * bi_swiglu.  Both give the same bits, which are those of the two separate calls.
 * workspace: device, >= bi_gemm_swiglu_workspace(M, F, K, mode) bytes, 16-byte
 * aligned; it may be NULL when the fused plan applies (M <= 128 in INVARIANT). */
size_t bi_gemm_swiglu_workspace(int64_t M, int64_t F, int64_t K, bi_mode mode);
bi_status bi_gemm_swiglu(const void* A, const void* W_gate_up, void* act, int64_t M, int64_t F, int64_t K,
                         bi_mode mode, int32_t target_row, int32_t target_count, void* workspace, size_t ws_bytes,
                         bi_stream s);

/* Per row, the k largest logits ordered by (value descending, index ascending):
 * ties go to the lowest index, so the result is unique [BlockLock "坑清单" 2, 5].
 * logits: device float [rows][V]; top_v: device float [rows][k]; top_i: device
 * int32 [rows][k].  1 <= k <= BI_TOPK_MAX, k <= V.  NaN logits are not supported. */
bi_status bi_topk(const float* logits, int64_t rows, int64_t V, int32_t k, float* top_v, int32_t* top_i,
                  bi_stream s);

/* ------------------------------------------------------------------ decoder layer / model */
typedef struct bi_layer_weights {
  const void* attn_norm; /* [d] bf16 */
  const void* w_qkv;     /* [(Hq+2Hkv)*hd][d] bf16 */
  const void* w_o;       /* [d][Hq*hd] bf16 */
  const void* ffn_norm;  /* [d] bf16 */
  const void* w_gate_up; /* [2F][d] bf16: gate rows 0..F-1, up rows F..2F-1 */
  const void* w_down;    /* [d][F] bf16 */
  /* Optional per-head RMSNorm of q and k before RoPE (Qwen3; NULL = none):
   * [head_dim] bf16 weights; each head row x of head_dim values becomes
   * (x / sqrt(sum(x^2)/head_dim + rms_eps)) * g in fp32, rounded to bf16 unless the
   * activations are fp32, the sum of squares taken in one fixed order that depends
   * on head_dim only.  Both or neither. */
  const void* q_norm;
  const void* k_norm;
} bi_layer_weights;

typedef struct bi_model_dims {
  int32_t d_model;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t ffn_dim;
  int32_t vocab;
  int32_t page_size; /* BI_PAGE_SIZE */
  int32_t max_pos;   /* rows of the RoPE tables */
  float rms_eps;
  /* 0: bf16 activations (hidden state and every tensor between the steps);
   * 1: fp32 activations with bf16 weights and a bf16 KV cache (the mixed-precision
   * mitigation, TML-digest §2/§6): hidden is fp32, nothing is rounded between the
   * steps except the k and v stored in the cache, and every GEMM multiplies the
   * fp32 activations exactly (bi_gemm_f32a).  Same schedules, same invariance. */
  int32_t act_f32;
} bi_model_dims;

/* A batch of requests.  Request b owns tokens q_start[b] .. q_start[b+1]-1 at
 * absolute positions pos0[b] .. pos0[b]+n_b-1; before the layer runs, its cache
 * holds exactly pos0[b] tokens.  Decode is the case n_b = 1 for all b. */
typedef struct bi_batch {
  int32_t num_requests;       /* B >= 1 */
  int32_t num_tokens;         /* T >= B */
  int32_t max_q_len;          /* max_b n_b (host-known); 1 selects the decode kernels */
  const int32_t* q_start;     /* device [B+1] */
  const int32_t* pos0;        /* device [B] */
  const int32_t* block_table; /* device [B][max_pages] */
  int32_t max_pages;
  int32_t num_pages;
  int32_t target_request; /* PROTECTED: the request whose bits are pinned; -1 = none */
  int32_t target_row;     /* its first token row (host-known; ignored if target_request < 0) */
  int32_t target_count;   /* its token count */
} bi_batch;

/* Pre-norm decoder layer, in place on hidden [T][d] (bf16, or fp32 when dims->act_f32):
 *   x = rms(h)*g1; qkv = x Wqkv^T; rope(q,k); store k,v in the cache; a = attn(q, cache);
 *   h = h + a Wo^T; x = rms(h)*g2; gu = x Wgu^T; h = h + (silu(g)*u) Wd^T
 * with bf16 tensors (fp32 when dims->act_f32) between the steps and the residual adds fused into the GEMMs
 * (reading: the pages fix the three reductions but not the layer, so the
 * standard Llama/Qwen-shaped layer is taken).  The K/V of the batch's tokens are
 * written to the cache before attention, so cached and new tokens are reduced
 * as one sequence [TML-digest §3.3, the 80-cached + 48-new example]. */
size_t bi_layer_workspace(const bi_model_dims* dims, const bi_batch* batch, bi_mode mode);
bi_status bi_layer_forward(const bi_model_dims* dims, const bi_layer_weights* w, const float* rope_cos,
                           const float* rope_sin, void* hidden, const bi_batch* batch, void* k_cache, void* v_cache,
                           bi_mode mode, void* workspace, size_t ws_bytes, bi_stream s);

typedef struct bi_model_weights {
  const void* embed;              /* [vocab][d] bf16 */
  const bi_layer_weights* layers; /* host array [num_layers] */
  int32_t num_layers;
  const void* final_norm; /* [d] bf16 */
  const void* lm_head;    /* [vocab][d] bf16 */
} bi_model_weights;

/* Whole forward for one batch: embedding gather, all layers, final RMSNorm, the
 * lm-head on the last token of every request (fp32 logits), and per-request
 * top-k.  ids: device int32 [T].  k_caches, v_caches: host arrays [num_layers]
 * of device cache pointers.  logits: device float [B][vocab].  top_v/top_i:
 * device [B][k] (k = topk, 1..BI_TOPK_MAX); top_i[b][0] is the greedy token,
 * also written contiguously to greedy_ids (device int32 [B], may be NULL) so it
 * can feed the next decode step's ids directly. */
size_t bi_model_workspace(const bi_model_dims* dims, const bi_batch* batch, bi_mode mode);
bi_status bi_model_forward(const bi_model_dims* dims, const bi_model_weights* w, const float* rope_cos,
                           const float* rope_sin, const int32_t* ids, const bi_batch* batch, void* const* k_caches,
                           void* const* v_caches, float* logits, int32_t topk, float* top_v, int32_t* top_i,
                           int32_t* greedy_ids, bi_mode mode, void* workspace, size_t ws_bytes, bi_stream s);

#ifdef __cplusplus
}
#endif
#endif /* BI_H_ */
