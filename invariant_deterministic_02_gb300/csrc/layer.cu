// Decoder layer and whole-model forward: the ordering of the kernels of one
// batch through the pre-norm layer, with every intermediate in caller-owned
// workspace.  Only RMSNorm, matmul and attention reduce across elements, so
// only they need batch-invariant kernels; the rest is pointwise (devpress digest
// of "Defeating Nondeterminism in LLM Inference", section 3).
#include <vector>

#include "common.cuh"

namespace bi {

bi_status rmsnorm_impl(const void*, const void*, void*, int64_t, int64_t, bi_dtype, float, bi_mode, int32_t, int32_t,
                       void*, size_t, cudaStream_t);
bi_status rmsnorm_planes_impl(const void*, const void*, void*, int64_t, int64_t, float, bi_mode, int32_t, int32_t,
                              void*, size_t, cudaStream_t);
size_t rmsnorm_ws(int64_t, int64_t, bi_mode);
// weights_constant: W is not written by the kernels of this forward pass, so the
// GEMM may start fetching it before the previous kernel has finished
bi_status gemm_impl(const void*, const void*, void*, const void*, int64_t, int64_t, int64_t, bi_dtype, bi_mode,
                    int32_t, int32_t, void*, size_t, cudaStream_t, bool weights_constant);
size_t gemm_ws(int64_t, int64_t, int64_t, bi_mode);
size_t gemm_ws(int64_t, int64_t, int64_t, bi_mode, int planes);
bi_status gemm_planes_impl(const void*, const void*, float*, const float*, int64_t, int64_t, int64_t, bi_mode, int32_t,
                           int32_t, void*, size_t, cudaStream_t, bool weights_constant);
bi_status decode_attention_impl(const void*, const void*, const void*, const int32_t*, const int32_t*, int32_t,
                                const bi_attn_dims*, void*, bi_mode, int32_t, void*, size_t, cudaStream_t);
bi_status prefill_attention_impl(const void*, const void*, const void*, const int32_t*, const int32_t*,
                                 const int32_t*, int32_t, int32_t, const bi_attn_dims*, void*, bi_mode, int32_t,
                                 void*, size_t, cudaStream_t);
size_t decode_attention_ws(int32_t, const bi_attn_dims*);
size_t decode_plan_bytes(int32_t, const bi_attn_dims*);
size_t decode_parts_bytes(int32_t, const bi_attn_dims*);
bi_status decode_attention_layer(const void*, const void*, const void*, const int32_t*, const int32_t*, int32_t,
                                 const bi_attn_dims*, const ActDst&, bi_mode, int32_t, void*, bool, void*, size_t,
                                 cudaStream_t);
bi_status prefill_attention_layer(const void*, const void*, const void*, const int32_t*, const int32_t*,
                                  const int32_t*, int32_t, int32_t, const bi_attn_dims*, const ActDst&, bi_mode,
                                  int32_t, void*, size_t, cudaStream_t);
size_t prefill_attention_ws(int32_t, int32_t, const bi_attn_dims*);
bi_status qkv_rope_store_impl(const void*, const float*, const float*, const int32_t*, const int32_t*,
                              const int32_t*, int32_t, const bi_attn_dims*, void*, void*, void*, cudaStream_t,
                              const void* q_norm, const void* k_norm, float eps, bool act_f32, int max_pos);
bi_status swiglu_impl(const void*, void*, int64_t, int64_t, cudaStream_t);
bi_status gemm_swiglu_impl(const void*, const void*, void*, int64_t, int64_t, int64_t, bi_mode, int32_t, int32_t,
                           cudaStream_t, bool*, bool);
bi_status swiglu_planes_impl(const void*, void*, int64_t, int64_t, cudaStream_t);
bi_status embed_impl(const int32_t*, const void*, void*, int64_t, int64_t, int64_t, cudaStream_t);
bi_status embed_f32_impl(const int32_t*, const void*, void*, int64_t, int64_t, int64_t, cudaStream_t);
bi_status topk_impl(const float*, int64_t, int64_t, int32_t, float*, int32_t*, int32_t*, cudaStream_t);

namespace {

// token -> (request, absolute position); request -> KV length after this batch.
__global__ void batch_index_kernel(const int32_t* __restrict__ q_start, const int32_t* __restrict__ pos0, int B, int T,
                                   int32_t* __restrict__ token_req, int32_t* __restrict__ token_pos,
                                   int32_t* __restrict__ kv_len, int32_t* __restrict__ last_row) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < T) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (q_start[mid] <= i) lo = mid; else hi = mid - 1;
    }
    token_req[i] = lo;
    token_pos[i] = pos0[lo] + (i - q_start[lo]);
  }
  if (i < B) {
    kv_len[i] = pos0[i] + (q_start[i + 1] - q_start[i]);
    last_row[i] = q_start[i + 1] - 1;
  }
}

// out[b] = in[rows[b]] (16-byte chunks)
__global__ void gather_rows_kernel(const uint4* __restrict__ in, const int32_t* __restrict__ rows, uint4* __restrict__ out,
                                   int B, int64_t chunks) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  if (b >= B) return;
  const int64_t r = rows[b];
  for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) out[b * chunks + c] = in[r * chunks + c];
}

// Activations between the steps are bf16, or with fp32 activations: GEMM
// inputs (x, att, act) as three bf16 planes [3][rows][cols], everything else fp32.
struct LayerBufs {
  int32_t* token_req;
  int32_t* token_pos;
  int32_t* kv_len;
  int32_t* last_row;
  void* x;    // [T][d] (planes)
  void* qkv;  // [T][qkv]
  void* q;    // [T][Hq*hd]
  void* att;  // [T][Hq*hd] (planes)
  void* gu;   // [T][2F]
  void* act;  // [T][F] (planes)
  void* dplan;  // decode attention plan (shared by the layers of a step)
  void* sub;  // sub-op workspace
  size_t sub_bytes;
  // model-level extras
  void* hidden;  // [T][d]
  void* xl;      // [B][d]
  size_t bytes;
};

bi_attn_dims attn_dims(const bi_model_dims* dm, const bi_batch* b) {
  bi_attn_dims a;
  a.num_q_heads = dm->num_q_heads;
  a.num_kv_heads = dm->num_kv_heads;
  a.head_dim = dm->head_dim;
  a.page_size = dm->page_size;
  a.max_pages = b->max_pages;
  a.num_pages = b->num_pages;
  a.scale = 1.0f / sqrtf(static_cast<float>(dm->head_dim));
  a.act_f32 = dm->act_f32;
  return a;
}

size_t sub_ws_bytes(const bi_model_dims* dm, const bi_batch* b, bi_mode mode, bool with_head) {
  const int64_t T = b->num_tokens, B = b->num_requests, d = dm->d_model, F = dm->ffn_dim;
  const int64_t hq = static_cast<int64_t>(dm->num_q_heads) * dm->head_dim;
  const int64_t qkvw = static_cast<int64_t>(dm->num_q_heads + 2 * dm->num_kv_heads) * dm->head_dim;
  const int pl = dm->act_f32 ? 3 : 1;
  size_t m = 0;
  m = std::max(m, rmsnorm_ws(T, d, mode));
  m = std::max(m, gemm_ws(T, qkvw, d, mode, pl));
  m = std::max(m, gemm_ws(T, d, hq, mode, pl));
  m = std::max(m, gemm_ws(T, 2 * F, d, mode, pl));
  m = std::max(m, gemm_ws(T, d, F, mode, pl));
  bi_attn_dims ad = attn_dims(dm, b);
  if (b->max_q_len == 1 && T == B)
    m = std::max(m, decode_parts_bytes(static_cast<int32_t>(B), &ad));
  else
    m = std::max(m, prefill_attention_ws(static_cast<int32_t>(B), static_cast<int32_t>(T), &ad));
  if (with_head) {
    m = std::max(m, rmsnorm_ws(B, d, mode));
    m = std::max(m, gemm_ws(B, dm->vocab, d, mode, pl));
  }
  return m;
}

LayerBufs carve(void* ws, size_t cap, const bi_model_dims* dm, const bi_batch* b, bi_mode mode, bool model) {
  WsCarver cv(ws, cap);
  LayerBufs r{};
  const int64_t T = b->num_tokens, B = b->num_requests, d = dm->d_model, F = dm->ffn_dim;
  const int64_t hq = static_cast<int64_t>(dm->num_q_heads) * dm->head_dim;
  const int64_t qkvw = static_cast<int64_t>(dm->num_q_heads + 2 * dm->num_kv_heads) * dm->head_dim;
  r.token_req = cv.take<int32_t>(T);
  r.token_pos = cv.take<int32_t>(T);
  r.kv_len = cv.take<int32_t>(B);
  r.last_row = cv.take<int32_t>(B);
  if (dm->act_f32) {
    r.x = cv.take<__nv_bfloat16>(3 * T * d);
    r.qkv = cv.take<float>(T * qkvw);
    r.q = cv.take<float>(T * hq);
    r.att = cv.take<__nv_bfloat16>(3 * T * hq);
    r.gu = cv.take<float>(T * 2 * F);
    r.act = cv.take<__nv_bfloat16>(3 * T * F);
  } else {
    r.x = cv.take<__nv_bfloat16>(T * d);
    r.qkv = cv.take<__nv_bfloat16>(T * qkvw);
    r.q = cv.take<__nv_bfloat16>(T * hq);
    r.att = cv.take<__nv_bfloat16>(T * hq);
    r.gu = cv.take<__nv_bfloat16>(T * 2 * F);
    r.act = cv.take<__nv_bfloat16>(T * F);
  }
  {
    const bi_attn_dims ad = attn_dims(dm, b);
    r.dplan = cv.take<unsigned char>(decode_plan_bytes(static_cast<int32_t>(B), &ad));
  }
  if (model) {
    const size_t es = dm->act_f32 ? sizeof(float) : sizeof(__nv_bfloat16);
    r.hidden = cv.take<unsigned char>(T * d * es);
    r.xl = cv.take<unsigned char>(B * d * es);
  }
  r.sub_bytes = sub_ws_bytes(dm, b, mode, model);
  r.sub = cv.take<unsigned char>(r.sub_bytes);
  r.bytes = cv.used;
  return r;
}

bi_status check_model_dims(const bi_model_dims* dm) {
  BI_REQUIRE(dm != nullptr, BI_ERR_INVALID_ARG, "null model dims");
  BI_REQUIRE(dm->d_model > 0 && dm->d_model % 8 == 0 && dm->ffn_dim > 0 && dm->ffn_dim % 8 == 0, BI_ERR_UNSUPPORTED,
             "d_model %d / ffn_dim %d must be positive multiples of 8", dm->d_model, dm->ffn_dim);
  BI_REQUIRE(dm->page_size == BI_PAGE_SIZE, BI_ERR_UNSUPPORTED, "page_size %d", dm->page_size);
  BI_REQUIRE(dm->max_pos > 0, BI_ERR_INVALID_ARG, "max_pos %d", dm->max_pos);
  BI_REQUIRE(dm->act_f32 == 0 || dm->act_f32 == 1, BI_ERR_INVALID_ARG, "act_f32 %d (0 or 1)", dm->act_f32);
  return BI_OK;
}

bi_status check_batch(const bi_batch* b) {
  BI_REQUIRE(b != nullptr, BI_ERR_INVALID_ARG, "null batch");
  BI_REQUIRE(b->num_requests >= 1 && b->num_tokens >= b->num_requests && b->max_q_len >= 1, BI_ERR_INVALID_ARG,
             "batch: B=%d T=%d max_q_len=%d", b->num_requests, b->num_tokens, b->max_q_len);
  BI_REQUIRE(b->q_start && b->pos0 && b->block_table, BI_ERR_INVALID_ARG, "batch: null device array");
  BI_REQUIRE(b->max_pages >= 1 && b->num_pages >= 1, BI_ERR_INVALID_ARG, "batch: max_pages/num_pages");
  BI_REQUIRE(b->target_request < b->num_requests, BI_ERR_INVALID_ARG, "batch: target_request %d", b->target_request);
  if (b->target_request >= 0)
    BI_REQUIRE(b->target_row >= 0 && b->target_count >= 1 &&
                   static_cast<int64_t>(b->target_row) + b->target_count <= b->num_tokens,
               BI_ERR_INVALID_ARG, "batch: target rows [%d, +%d)", b->target_row, b->target_count);
  return BI_OK;
}

// The layer body with fp32 activations (bf16 weights and KV cache): the same
// steps and schedules; RMSNorm, attention and SwiGLU write the GEMM inputs as
// three bf16 planes, GEMMs write fp32 and add the fp32 residual.
bi_status layer_body_f32(const bi_model_dims* dm, const bi_layer_weights* w, const float* rc, const float* rs,
                         float* hidden, const bi_batch* b, void* kc, void* vc, bi_mode mode, const LayerBufs& L,
                         bool plan_attention, cudaStream_t s) {
  const int64_t T = b->num_tokens, d = dm->d_model, F = dm->ffn_dim;
  const int64_t hq = static_cast<int64_t>(dm->num_q_heads) * dm->head_dim;
  const int64_t qkvw = static_cast<int64_t>(dm->num_q_heads + 2 * dm->num_kv_heads) * dm->head_dim;
  const bool prot = mode == BI_MODE_PROTECTED && b->target_request >= 0;
  const int32_t trow = prot ? b->target_row : -1;
  const int32_t tcnt = prot ? b->target_count : 0;
  const int32_t treq = prot ? b->target_request : -1;
  bi_attn_dims ad = attn_dims(dm, b);
  float* qkv = static_cast<float*>(L.qkv);
  float* gu = static_cast<float*>(L.gu);
  BI_TRY(rmsnorm_planes_impl(hidden, w->attn_norm, L.x, T, d, dm->rms_eps, mode, trow, tcnt, L.sub, L.sub_bytes, s));
  BI_TRY(gemm_planes_impl(L.x, w->w_qkv, qkv, nullptr, T, qkvw, d, mode, trow, tcnt, L.sub, L.sub_bytes, s, true));
  BI_TRY(qkv_rope_store_impl(qkv, rc, rs, L.token_pos, L.token_req, b->block_table, static_cast<int32_t>(T), &ad,
                             L.q, kc, vc, s, w->q_norm, w->k_norm, dm->rms_eps, true, dm->max_pos));
  const ActDst att{L.att, static_cast<size_t>(T * hq), kActPlanes};
  if (b->max_q_len == 1 && T == b->num_requests) {
    BI_TRY(decode_attention_layer(L.q, kc, vc, b->block_table, L.kv_len, b->num_requests, &ad, att, mode, treq,
                                  L.dplan, plan_attention, L.sub, L.sub_bytes, s));
  } else {
    BI_TRY(prefill_attention_layer(L.q, kc, vc, b->block_table, b->q_start, b->pos0, b->num_requests,
                                   static_cast<int32_t>(T), &ad, att, mode, treq, L.sub, L.sub_bytes, s));
  }
  BI_TRY(gemm_planes_impl(L.att, w->w_o, hidden, hidden, T, d, hq, mode, trow, tcnt, L.sub, L.sub_bytes, s, true));
  BI_TRY(rmsnorm_planes_impl(hidden, w->ffn_norm, L.x, T, d, dm->rms_eps, mode, trow, tcnt, L.sub, L.sub_bytes, s));
  BI_TRY(gemm_planes_impl(L.x, w->w_gate_up, gu, nullptr, T, 2 * F, d, mode, trow, tcnt, L.sub, L.sub_bytes, s, true));
  BI_TRY(swiglu_planes_impl(gu, L.act, T, F, s));
  BI_TRY(gemm_planes_impl(L.act, w->w_down, hidden, hidden, T, d, F, mode, trow, tcnt, L.sub, L.sub_bytes, s, true));
  return BI_OK;
}

// The layer body over precomputed batch indices.
bi_status layer_body(const bi_model_dims* dm, const bi_layer_weights* w, const float* rc, const float* rs,
                     void* hidden, const bi_batch* b, void* kc, void* vc, bi_mode mode, const LayerBufs& L,
                     bool plan_attention, cudaStream_t s) {
  const int64_t T = b->num_tokens, d = dm->d_model, F = dm->ffn_dim;
  const int64_t hq = static_cast<int64_t>(dm->num_q_heads) * dm->head_dim;
  const int64_t qkvw = static_cast<int64_t>(dm->num_q_heads + 2 * dm->num_kv_heads) * dm->head_dim;
  const bool prot = mode == BI_MODE_PROTECTED && b->target_request >= 0;
  const int32_t trow = prot ? b->target_row : -1;
  const int32_t tcnt = prot ? b->target_count : 0;
  const int32_t treq = prot ? b->target_request : -1;
  BI_REQUIRE(w && w->attn_norm && w->w_qkv && w->w_o && w->ffn_norm && w->w_gate_up && w->w_down, BI_ERR_INVALID_ARG,
             "layer: null weight pointer");
  bi_attn_dims ad = attn_dims(dm, b);
  if (dm->act_f32) return layer_body_f32(dm, w, rc, rs, static_cast<float*>(hidden), b, kc, vc, mode, L,
                                         plan_attention, s);
  BI_TRY(rmsnorm_impl(hidden, w->attn_norm, L.x, T, d, BI_BF16, dm->rms_eps, mode, trow, tcnt, L.sub, L.sub_bytes, s));
  BI_TRY(gemm_impl(L.x, w->w_qkv, L.qkv, nullptr, T, qkvw, d, BI_BF16, mode, trow, tcnt, L.sub, L.sub_bytes, s, true));
  BI_TRY(qkv_rope_store_impl(L.qkv, rc, rs, L.token_pos, L.token_req, b->block_table, static_cast<int32_t>(T), &ad,
                             L.q, kc, vc, s, w->q_norm, w->k_norm, dm->rms_eps, false, dm->max_pos));
  if (b->max_q_len == 1 && T == b->num_requests) {
    BI_TRY(decode_attention_layer(L.q, kc, vc, b->block_table, L.kv_len, b->num_requests, &ad,
                                  ActDst{L.att, 0, kActBF16}, mode, treq, L.dplan, plan_attention, L.sub, L.sub_bytes,
                                  s));
  } else {
    BI_TRY(prefill_attention_impl(L.q, kc, vc, b->block_table, b->q_start, b->pos0, b->num_requests,
                                  static_cast<int32_t>(T), &ad, L.att, mode, treq, L.sub, L.sub_bytes, s));
  }
  BI_TRY(gemm_impl(L.att, w->w_o, hidden, hidden, T, d, hq, BI_BF16, mode, trow, tcnt, L.sub, L.sub_bytes, s, true));
  BI_TRY(rmsnorm_impl(hidden, w->ffn_norm, L.x, T, d, BI_BF16, dm->rms_eps, mode, trow, tcnt, L.sub, L.sub_bytes, s));
  bool fused = false;
  BI_TRY(gemm_swiglu_impl(L.x, w->w_gate_up, L.act, T, F, d, mode, trow, tcnt, s, &fused, true));
  if (!fused) {
    BI_TRY(gemm_impl(L.x, w->w_gate_up, L.gu, nullptr, T, 2 * F, d, BI_BF16, mode, trow, tcnt, L.sub, L.sub_bytes, s,
                     true));
    BI_TRY(swiglu_impl(L.gu, L.act, T, F, s));
  }
  BI_TRY(gemm_impl(L.act, w->w_down, hidden, hidden, T, d, F, BI_BF16, mode, trow, tcnt, L.sub, L.sub_bytes, s, true));
  return BI_OK;
}

bi_status batch_index(const bi_batch* b, const LayerBufs& L, cudaStream_t s) {
  const int n = std::max(b->num_tokens, b->num_requests);
  BI_TIMED(::bi::kTagBatchIndex, s, BI_PDL_CHECK(launch_pdl(batch_index_kernel, dim3((n + 255) / 256), dim3(256), 0, s, b->q_start, b->pos0, b->num_requests, b->num_tokens, L.token_req,
                                                     L.token_pos, L.kv_len, L.last_row)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

}  // namespace

size_t layer_ws(const bi_model_dims* dm, const bi_batch* b, bi_mode mode) {
  if (check_model_dims(dm) != BI_OK || check_batch(b) != BI_OK) return 0;
  return carve(nullptr, 0, dm, b, mode, false).bytes;
}

size_t model_ws(const bi_model_dims* dm, const bi_batch* b, bi_mode mode) {
  if (check_model_dims(dm) != BI_OK || check_batch(b) != BI_OK) return 0;
  return carve(nullptr, 0, dm, b, mode, true).bytes;
}

bi_status layer_forward_impl(const bi_model_dims* dm, const bi_layer_weights* w, const float* rc, const float* rs,
                             void* hidden, const bi_batch* b, void* kc, void* vc, bi_mode mode, void* ws,
                             size_t ws_bytes, cudaStream_t s) {
  clear_error();
  BI_TRY(check_model_dims(dm));
  BI_TRY(check_batch(b));
  BI_REQUIRE(mode_valid(mode), BI_ERR_INVALID_ARG, "mode %d",
             static_cast<int>(mode));
  BI_REQUIRE(hidden && kc && vc && rc && rs, BI_ERR_INVALID_ARG, "bi_layer_forward: null pointer");
  LayerBufs L = carve(ws, ws_bytes, dm, b, mode, false);
  BI_REQUIRE(ws != nullptr && L.bytes <= ws_bytes, BI_ERR_WORKSPACE, "bi_layer_forward: workspace %zu < %zu",
             ws_bytes, L.bytes);
  BI_TRY(batch_index(b, L, s));
  return layer_body(dm, w, rc, rs, hidden, b, kc, vc, mode, L, true, s);
}

bi_status model_forward_impl(const bi_model_dims* dm, const bi_model_weights* mw, const float* rc, const float* rs,
                             const int32_t* ids, const bi_batch* b, void* const* kcs, void* const* vcs, float* logits,
                             int32_t topk, float* top_v, int32_t* top_i, int32_t* greedy, bi_mode mode, void* ws,
                             size_t ws_bytes, cudaStream_t s) {
  clear_error();
  BI_TRY(check_model_dims(dm));
  BI_TRY(check_batch(b));
  BI_REQUIRE(mode_valid(mode), BI_ERR_INVALID_ARG, "mode %d",
             static_cast<int>(mode));
  BI_REQUIRE(mw && mw->embed && mw->final_norm && mw->lm_head && mw->num_layers >= 0 &&
                 (mw->num_layers == 0 || (mw->layers && kcs && vcs)),
             BI_ERR_INVALID_ARG, "bi_model_forward: null model pointer");
  BI_REQUIRE(ids && logits && top_v && top_i && rc && rs, BI_ERR_INVALID_ARG, "bi_model_forward: null pointer");
  BI_REQUIRE(dm->vocab >= 1 && dm->vocab % 8 == 0, BI_ERR_UNSUPPORTED, "vocab %d must be a multiple of 8", dm->vocab);
  LayerBufs L = carve(ws, ws_bytes, dm, b, mode, true);
  BI_REQUIRE(ws != nullptr && L.bytes <= ws_bytes, BI_ERR_WORKSPACE, "bi_model_forward: workspace %zu < %zu",
             ws_bytes, L.bytes);
  const int64_t T = b->num_tokens, B = b->num_requests, d = dm->d_model;
  BI_TRY(batch_index(b, L, s));
  if (dm->act_f32) BI_TRY(embed_f32_impl(ids, mw->embed, L.hidden, T, d, dm->vocab, s));
  else BI_TRY(embed_impl(ids, mw->embed, L.hidden, T, d, dm->vocab, s));
  for (int i = 0; i < mw->num_layers; ++i) {
    BI_REQUIRE(kcs[i] && vcs[i], BI_ERR_INVALID_ARG, "bi_model_forward: null cache of layer %d", i);
    BI_TRY(layer_body(dm, &mw->layers[i], rc, rs, L.hidden, b, kcs[i], vcs[i], mode, L, i == 0, s));
  }
  const void* last = L.hidden;
  if (T != B) {
    BI_TIMED(::bi::kTagGather, s, BI_PDL_CHECK(launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>(B)), dim3(128), 0, s, static_cast<const uint4*>(L.hidden), L.last_row,
                                                                static_cast<uint4*>(L.xl), static_cast<int>(B), dm->act_f32 ? d / 4 : d / 8)));
    BI_LAUNCH_CHECK();
    last = L.xl;
  }
  const bool prot = mode == BI_MODE_PROTECTED && b->target_request >= 0;
  const int32_t trow = prot ? b->target_request : -1;
  const int32_t tcnt = prot ? 1 : 0;
  if (dm->act_f32) {
    BI_TRY(rmsnorm_planes_impl(last, mw->final_norm, L.x, B, d, dm->rms_eps, mode, trow, tcnt, L.sub, L.sub_bytes, s));
    BI_TRY(gemm_planes_impl(L.x, mw->lm_head, logits, nullptr, B, dm->vocab, d, mode, trow, tcnt, L.sub, L.sub_bytes,
                            s, true));
  } else {
    BI_TRY(rmsnorm_impl(last, mw->final_norm, L.x, B, d, BI_BF16, dm->rms_eps, mode, trow, tcnt, L.sub, L.sub_bytes,
                        s));
    BI_TRY(gemm_impl(L.x, mw->lm_head, logits, nullptr, B, dm->vocab, d, BI_F32, mode, trow, tcnt, L.sub,
                     L.sub_bytes, s, true));
  }
  BI_TRY(topk_impl(logits, B, dm->vocab, topk, top_v, top_i, greedy, s));
  return BI_OK;
}

}  // namespace bi

extern "C" size_t bi_layer_workspace(const bi_model_dims* dims, const bi_batch* batch, bi_mode mode) {
  return bi::layer_ws(dims, batch, mode);
}

extern "C" bi_status bi_layer_forward(const bi_model_dims* dims, const bi_layer_weights* w, const float* rope_cos,
                                      const float* rope_sin, void* hidden, const bi_batch* batch, void* k_cache,
                                      void* v_cache, bi_mode mode, void* workspace, size_t ws_bytes, bi_stream s) {
  return bi::layer_forward_impl(dims, w, rope_cos, rope_sin, hidden, batch, k_cache, v_cache, mode, workspace,
                                ws_bytes, reinterpret_cast<cudaStream_t>(s));
}

extern "C" size_t bi_model_workspace(const bi_model_dims* dims, const bi_batch* batch, bi_mode mode) {
  return bi::model_ws(dims, batch, mode);
}

extern "C" bi_status bi_model_forward(const bi_model_dims* dims, const bi_model_weights* w, const float* rope_cos,
                                      const float* rope_sin, const int32_t* ids, const bi_batch* batch,
                                      void* const* k_caches, void* const* v_caches, float* logits, int32_t topk,
                                      float* top_v, int32_t* top_i, int32_t* greedy_ids, bi_mode mode, void* workspace,
                                      size_t ws_bytes, bi_stream s) {
  return bi::model_forward_impl(dims, w, rope_cos, rope_sin, ids, batch, k_caches, v_caches, logits, topk, top_v,
                                top_i, greedy_ids, mode, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(s));
}
