// Pointwise steps of the decoder layer: embedding gather, RoPE tables, the QKV
// split with rotary embedding and the paged K/V store, SwiGLU gating.
// Each output element depends on its own inputs only, so these steps are batch
// invariant as they stand (devpress digest of "Defeating Nondeterminism in LLM
// Inference", section 3: pointwise operations need no change).
#include <cmath>
#include <type_traits>

#include "common.cuh"

namespace bi {
namespace {

__global__ void embed_kernel(const int32_t* __restrict__ ids, const uint4* __restrict__ table, uint4* __restrict__ out,
                             int64_t T, int64_t chunks_per_row, int64_t vocab) {
  pdl_wait();
  pdl_trigger();
  const int64_t t = blockIdx.x;
  if (t >= T) return;
  const int64_t id = ids[t];
  const bool ok = id >= 0 && id < vocab;
  for (int64_t c = threadIdx.x; c < chunks_per_row; c += blockDim.x)
    out[t * chunks_per_row + c] = ok ? table[id * chunks_per_row + c] : make_uint4(0, 0, 0, 0);
}

// cos/sin(p * theta^(-2i/hd)) in float64, rounded once to fp32.
__global__ void rope_table_kernel(double theta, int hd, int max_pos, float* __restrict__ cs, float* __restrict__ sn) {
  pdl_wait();
  pdl_trigger();
  const int half = hd / 2;
  const int64_t n = static_cast<int64_t>(max_pos) * half;
  for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < n;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int p = static_cast<int>(k / half);
    const int i = static_cast<int>(k % half);
    const double f = pow(theta, -2.0 * i / hd);
    double sv, cv;
    sincos(static_cast<double>(p) * f, &sv, &cv);
    cs[k] = static_cast<float>(cv);
    sn[k] = static_cast<float>(sv);
  }
}

__device__ __forceinline__ float round_bf16f(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// One warp per (token, head row): task k < hq rotates q head k, then the kv
// heads' k rows are rotated and stored in the paged cache, then their v rows
// are copied there.  Lane j handles the rotation pairs (i, i + hd/2) for
// i = 2j', 2j'+1 (j' = j, j+32, ...), so loads and stores move two elements.
// With qn / kn (Qwen3's per-head norms) a q or k row is first RMS-normalised
// over its hd values: lane sums of squares in the order (i, i+1, i+hd/2,
// i+hd/2+1) per pair, a xor butterfly over the warp (every lane gets the same
// bits), r = 1/sqrt(sum/hd + eps), x -> (x*r)*g (rounded to bf16 with bf16
// activations), then rotated.
// F32 (fp32 activations): qkv and q_out are fp32 and nothing is rounded except
// the k and v rows stored in the bf16 cache.
template <bool F32>
struct QkvIo {
  using T = typename std::conditional<F32, float, __nv_bfloat16>::type;
  // elements (i, i+1) of a row as floats
  static __device__ __forceinline__ float2 ld2(const T* p) {
    if constexpr (F32) {
      return *reinterpret_cast<const float2*>(p);
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
      return make_float2(bf16_lo(v), bf16_hi(v));
    }
  }
};

// Error word of this file: 21 a K/V store whose position lies past the
// block-table row or whose page lies outside the cache (the store is skipped);
// 22 a position outside the RoPE table (the last row is used).
__device__ unsigned int g_pw_err_word = 0;
constexpr unsigned kSiteBadStore = 21;
constexpr unsigned kSiteBadPos = 22;

// Cache page of position `pos` of request `req`, or -1 (reported) when the
// position lies past the block-table row or the entry lies outside the cache.
__device__ __forceinline__ int store_page(const int32_t* __restrict__ block_table, int req, int pos, int max_pages,
                                          int num_pages) {
  const int pi = pos / BI_PAGE_SIZE;
  const int pg = (pos >= 0 && pi < max_pages) ? block_table[static_cast<size_t>(req) * max_pages + pi] : -1;
  if (pg < 0 || pg >= num_pages) {
    atomicCAS(&g_pw_err_word, 0u, kSiteBadStore);
    return -1;
  }
  return pg;
}

template <bool F32>
__global__ void __launch_bounds__(256) qkv_rope_store_kernel(
    const typename QkvIo<F32>::T* __restrict__ qkv, const float* __restrict__ rc, const float* __restrict__ rs,
    const int32_t* __restrict__ token_pos, const int32_t* __restrict__ token_req,
    const int32_t* __restrict__ block_table, int max_pages, int num_pages, int max_pos, int hq, int hkv, int hd,
    typename QkvIo<F32>::T* __restrict__ q_out, __nv_bfloat16* __restrict__ kc, __nv_bfloat16* __restrict__ vc,
    const __nv_bfloat16* __restrict__ qn, const __nv_bfloat16* __restrict__ kn, float eps) {
  using T = typename QkvIo<F32>::T;
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int task = blockIdx.y * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (task >= hq + 2 * hkv) return;
  const int pos = token_pos[t];
  const int width = (hq + 2 * hkv) * hd;
  const T* row = qkv + static_cast<size_t>(t) * width;
  if (task >= hq + hkv) {
    // v row of kv head h: stored in the cache (rounded to bf16 from fp32 activations)
    const int h = task - hq - hkv;
    const int page = store_page(block_table, token_req[t], pos, max_pages, num_pages);
    if (page < 0) return;
    const T* src = row + (hq + hkv + h) * hd;
    uint4* dst = reinterpret_cast<uint4*>(vc + ((static_cast<size_t>(page) * hkv + h) * BI_PAGE_SIZE +
                                                pos % BI_PAGE_SIZE) * hd);
    for (int k = lane; k < hd / 8; k += 32) {
      if constexpr (F32) {
        const float4 a = reinterpret_cast<const float4*>(src)[2 * k];
        const float4 b = reinterpret_cast<const float4*>(src)[2 * k + 1];
        dst[k] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                            pack_bf16x2(b.z, b.w));
      } else {
        dst[k] = reinterpret_cast<const uint4*>(src)[k];
      }
    }
    return;
  }
  const bool is_q = task < hq;
  const int h = is_q ? task : task - hq;
  const int half = hd / 2;
  const T* src = row + (is_q ? 0 : hq * hd) + h * hd;
  T* qdst = nullptr;
  uint16_t* kdst = nullptr;
  if (is_q) {
    qdst = q_out + (static_cast<size_t>(t) * hq + h) * hd;
  } else {
    const int page = store_page(block_table, token_req[t], pos, max_pages, num_pages);
    if (page < 0) return;
    kdst = reinterpret_cast<uint16_t*>(kc) + ((static_cast<size_t>(page) * hkv + h) * BI_PAGE_SIZE +
                                              pos % BI_PAGE_SIZE) * hd;
  }
  int tpos = pos;  // row of the RoPE tables
  if (tpos < 0 || tpos >= max_pos) {
    if (lane == 0) atomicCAS(&g_pw_err_word, 0u, kSiteBadPos);
    tpos = tpos < 0 ? 0 : max_pos - 1;
  }
  const float* c_row = rc + static_cast<size_t>(tpos) * half;
  const float* s_row = rs + static_cast<size_t>(tpos) * half;
  const __nv_bfloat16* g = is_q ? qn : kn;
  float r = 0.f;
  if (g != nullptr) {
    float ss = 0.f;
    for (int j = lane; j < half / 2; j += 32) {
      const int i = 2 * j;
      const float2 av = QkvIo<F32>::ld2(src + i);
      const float2 bv = QkvIo<F32>::ld2(src + i + half);
      const float x[4] = {av.x, av.y, bv.x, bv.y};
#pragma unroll
      for (int e = 0; e < 4; ++e) ss = __fadd_rn(ss, __fmul_rn(x[e], x[e]));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(hd)), eps)));
  }
  for (int j = lane; j < half / 2; j += 32) {
    const int i = 2 * j;
    const float2 av = QkvIo<F32>::ld2(src + i);
    const float2 bv = QkvIo<F32>::ld2(src + i + half);
    const float2 c = *reinterpret_cast<const float2*>(c_row + i);
    const float2 sn = *reinterpret_cast<const float2*>(s_row + i);
    float a0 = av.x, a1 = av.y, b0 = bv.x, b1 = bv.y;
    if (g != nullptr) {
      const uint32_t ga = *reinterpret_cast<const uint32_t*>(g + i);
      const uint32_t gb = *reinterpret_cast<const uint32_t*>(g + i + half);
      a0 = __fmul_rn(__fmul_rn(a0, r), bf16_lo(ga));
      a1 = __fmul_rn(__fmul_rn(a1, r), bf16_hi(ga));
      b0 = __fmul_rn(__fmul_rn(b0, r), bf16_lo(gb));
      b1 = __fmul_rn(__fmul_rn(b1, r), bf16_hi(gb));
      if constexpr (!F32) {
        a0 = round_bf16f(a0);
        a1 = round_bf16f(a1);
        b0 = round_bf16f(b0);
        b1 = round_bf16f(b1);
      }
    }
    const float lo0 = __fsub_rn(__fmul_rn(a0, c.x), __fmul_rn(b0, sn.x));
    const float lo1 = __fsub_rn(__fmul_rn(a1, c.y), __fmul_rn(b1, sn.y));
    const float hi0 = __fadd_rn(__fmul_rn(b0, c.x), __fmul_rn(a0, sn.x));
    const float hi1 = __fadd_rn(__fmul_rn(b1, c.y), __fmul_rn(a1, sn.y));
    if (kdst != nullptr || !F32) {
      uint16_t* d = kdst != nullptr ? kdst : reinterpret_cast<uint16_t*>(qdst);
      *reinterpret_cast<uint32_t*>(d + i) = pack_bf16x2(lo0, lo1);
      *reinterpret_cast<uint32_t*>(d + i + half) = pack_bf16x2(hi0, hi1);
    } else {
      float* d = reinterpret_cast<float*>(qdst);
      *reinterpret_cast<float2*>(d + i) = make_float2(lo0, lo1);
      *reinterpret_cast<float2*>(d + i + half) = make_float2(hi0, hi1);
    }
  }
}

__global__ void swiglu_kernel(const __nv_bfloat16* __restrict__ gu, __nv_bfloat16* __restrict__ out, int64_t T,
                              int64_t F) {
  pdl_wait();
  pdl_trigger();
  const int64_t chunks = F / 8;
  const int64_t n = T * chunks;
  for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < n;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = k / chunks, c = k % chunks;
    const uint4 gv = *reinterpret_cast<const uint4*>(gu + t * 2 * F + c * 8);
    const uint4 uv = *reinterpret_cast<const uint4*>(gu + t * 2 * F + F + c * 8);
    float g[8], u[8], o[8];
    unpack8(gv, g);
    unpack8(uv, u);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = swiglu1(g[e], u[e]);
    *reinterpret_cast<uint4*>(out + t * F + c * 8) = pack8(o);
  }
}

// fp32 activations: gu fp32 [T][2F], out three bf16 planes [3][T][F]; the same
// per-element arithmetic as the bf16 kernel.
__global__ void swiglu_planes_kernel(const float* __restrict__ gu, uint16_t* __restrict__ out, int64_t T, int64_t F) {
  pdl_wait();
  pdl_trigger();
  const int64_t chunks = F / 4;
  const int64_t n = T * chunks;
  const size_t plane = static_cast<size_t>(T) * F;
  for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < n;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = k / chunks, c = k % chunks;
    const float4 gv = *reinterpret_cast<const float4*>(gu + t * 2 * F + c * 4);
    const float4 uv = *reinterpret_cast<const float4*>(gu + t * 2 * F + F + c * 4);
    const float g[4] = {gv.x, gv.y, gv.z, gv.w};
    const float u[4] = {uv.x, uv.y, uv.z, uv.w};
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = swiglu1(g[e], u[e]);
    store_planes4(out + t * F + c * 4, plane, o[0], o[1], o[2], o[3]);
  }
}

// fp32 activations: the bf16 embedding row widened to fp32.
__global__ void embed_f32_kernel(const int32_t* __restrict__ ids, const uint4* __restrict__ table,
                                 float4* __restrict__ out, int64_t T, int64_t chunks_per_row, int64_t vocab) {
  pdl_wait();
  pdl_trigger();
  const int64_t t = blockIdx.x;
  if (t >= T) return;
  const int64_t id = ids[t];
  const bool ok = id >= 0 && id < vocab;
  for (int64_t c = threadIdx.x; c < chunks_per_row; c += blockDim.x) {
    const uint4 u = ok ? table[id * chunks_per_row + c] : make_uint4(0, 0, 0, 0);
    out[(t * chunks_per_row + c) * 2] = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    out[(t * chunks_per_row + c) * 2 + 1] = make_float4(bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w));
  }
}

}  // namespace

bi_status embed_impl(const int32_t* ids, const void* table, void* out, int64_t T, int64_t d, int64_t vocab,
                     cudaStream_t s) {
  BI_REQUIRE(T >= 0 && d > 0 && d % 8 == 0 && vocab > 0, BI_ERR_INVALID_ARG, "bi_embed: T=%lld d=%lld vocab=%lld",
             static_cast<long long>(T), static_cast<long long>(d), static_cast<long long>(vocab));
  if (T == 0) return BI_OK;
  BI_REQUIRE(ids && table && out && aligned16(table) && aligned16(out), BI_ERR_INVALID_ARG,
             "bi_embed: null or misaligned pointer");
  BI_TIMED(::bi::kTagEmbed, s, BI_PDL_CHECK(launch_pdl(embed_kernel, dim3(static_cast<unsigned>(T)), dim3(128), 0, s, ids, static_cast<const uint4*>(table), static_cast<uint4*>(out),
                                                        T, d / 8, vocab)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

bi_status qkv_rope_store_impl(const void* qkv, const float* rc, const float* rs, const int32_t* token_pos,
                              const int32_t* token_req, const int32_t* block_table, int32_t T,
                              const bi_attn_dims* dm, void* q_out, void* kc, void* vc, cudaStream_t s,
                              const void* q_norm, const void* k_norm, float eps, bool act_f32, int max_pos) {
  BI_REQUIRE(dm && T >= 0, BI_ERR_INVALID_ARG, "bi_qkv_rope_store: dims/T");
  BI_REQUIRE(dm->head_dim % 16 == 0 && dm->head_dim >= 16 && dm->num_kv_heads >= 1 && dm->num_q_heads >= 1,
             BI_ERR_UNSUPPORTED, "bi_qkv_rope_store: head_dim %d", dm->head_dim);
  BI_REQUIRE(dm->page_size == BI_PAGE_SIZE, BI_ERR_UNSUPPORTED, "bi_qkv_rope_store: page_size %d", dm->page_size);
  if (T == 0) return BI_OK;
  BI_REQUIRE(qkv && rc && rs && token_pos && token_req && block_table && q_out && kc && vc, BI_ERR_INVALID_ARG,
             "bi_qkv_rope_store: null pointer");
  BI_REQUIRE(aligned16(qkv) && aligned16(q_out) && aligned16(kc) && aligned16(vc), BI_ERR_INVALID_ARG,
             "bi_qkv_rope_store: misaligned pointer");
  BI_REQUIRE((q_norm == nullptr) == (k_norm == nullptr) && (q_norm == nullptr || (aligned16(q_norm) && aligned16(k_norm))),
             BI_ERR_INVALID_ARG, "layer: q_norm and k_norm must be both null or both 16-byte aligned");
  const dim3 grid(T, (dm->num_q_heads + 2 * dm->num_kv_heads + 7) / 8);
  if (act_f32) {
    BI_TIMED(::bi::kTagQkvRope, s, BI_PDL_CHECK(launch_pdl(qkv_rope_store_kernel<true>, grid, dim3(256), 0, s, static_cast<const float*>(qkv), rc, rs, token_pos, token_req,
                                            block_table, dm->max_pages, dm->num_pages, max_pos, dm->num_q_heads,
                                            dm->num_kv_heads, dm->head_dim,
                                            static_cast<float*>(q_out), static_cast<__nv_bfloat16*>(kc),
                                            static_cast<__nv_bfloat16*>(vc), static_cast<const __nv_bfloat16*>(q_norm),
                                            static_cast<const __nv_bfloat16*>(k_norm), eps)));
  } else {
    BI_TIMED(::bi::kTagQkvRope, s, BI_PDL_CHECK(launch_pdl(qkv_rope_store_kernel<false>, grid, dim3(256), 0, s, static_cast<const __nv_bfloat16*>(qkv), rc, rs, token_pos, token_req,
                                            block_table, dm->max_pages, dm->num_pages, max_pos, dm->num_q_heads,
                                            dm->num_kv_heads, dm->head_dim,
                                            static_cast<__nv_bfloat16*>(q_out), static_cast<__nv_bfloat16*>(kc),
                                            static_cast<__nv_bfloat16*>(vc), static_cast<const __nv_bfloat16*>(q_norm),
                                            static_cast<const __nv_bfloat16*>(k_norm), eps)));
  }
  BI_LAUNCH_CHECK();
  return BI_OK;
}

bi_status swiglu_impl(const void* gu, void* out, int64_t T, int64_t F, cudaStream_t s) {
  BI_REQUIRE(T >= 0 && F > 0 && F % 8 == 0, BI_ERR_INVALID_ARG, "bi_swiglu: T=%lld F=%lld", static_cast<long long>(T),
             static_cast<long long>(F));
  if (T == 0) return BI_OK;
  BI_REQUIRE(gu && out && aligned16(gu) && aligned16(out), BI_ERR_INVALID_ARG, "bi_swiglu: null or misaligned");
  const int64_t n = T * (F / 8);
  const int64_t grid = std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(num_sms()) * 16);
  BI_TIMED(::bi::kTagSwiglu, s, BI_PDL_CHECK(launch_pdl(swiglu_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, static_cast<const __nv_bfloat16*>(gu),
                                                            static_cast<__nv_bfloat16*>(out), T, F)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

// fp32 activations: gu fp32 [T][2F] -> three bf16 planes [3][T][F].
bi_status swiglu_planes_impl(const void* gu, void* out, int64_t T, int64_t F, cudaStream_t s) {
  BI_REQUIRE(T >= 0 && F > 0 && F % 8 == 0, BI_ERR_INVALID_ARG, "swiglu: T=%lld F=%lld", static_cast<long long>(T),
             static_cast<long long>(F));
  if (T == 0) return BI_OK;
  BI_REQUIRE(gu && out && aligned16(gu) && aligned16(out), BI_ERR_INVALID_ARG, "swiglu: null or misaligned");
  const int64_t n = T * (F / 4);
  const int64_t grid = std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(num_sms()) * 16);
  BI_TIMED(::bi::kTagSwiglu, s, BI_PDL_CHECK(launch_pdl(swiglu_planes_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, static_cast<const float*>(gu),
                                                            static_cast<uint16_t*>(out), T, F)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

// fp32 activations: embedding rows (bf16 table) widened to fp32 [T][d].
bi_status embed_f32_impl(const int32_t* ids, const void* table, void* out, int64_t T, int64_t d, int64_t vocab,
                         cudaStream_t s) {
  BI_REQUIRE(T >= 0 && d > 0 && d % 8 == 0 && vocab > 0, BI_ERR_INVALID_ARG, "embed: T=%lld d=%lld vocab=%lld",
             static_cast<long long>(T), static_cast<long long>(d), static_cast<long long>(vocab));
  if (T == 0) return BI_OK;
  BI_REQUIRE(ids && table && out && aligned16(table) && aligned16(out), BI_ERR_INVALID_ARG,
             "embed: null or misaligned pointer");
  BI_TIMED(::bi::kTagEmbed, s, BI_PDL_CHECK(launch_pdl(embed_f32_kernel, dim3(static_cast<unsigned>(T)), dim3(128), 0, s, ids, static_cast<const uint4*>(table), static_cast<float4*>(out),
                                                        T, d / 8, vocab)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

bi_status rope_table_impl(double theta, int32_t hd, int32_t max_pos, float* cs, float* sn, cudaStream_t s) {
  BI_REQUIRE(theta > 1.0 && hd > 0 && hd % 2 == 0 && max_pos >= 0, BI_ERR_INVALID_ARG,
             "bi_rope_table: theta=%g head_dim=%d max_pos=%d", theta, hd, max_pos);
  if (max_pos == 0) return BI_OK;
  BI_REQUIRE(cs && sn, BI_ERR_INVALID_ARG, "bi_rope_table: null pointer");
  const int64_t n = static_cast<int64_t>(max_pos) * (hd / 2);
  const int64_t grid = std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(num_sms()) * 8);
  BI_TIMED(::bi::kTagRopeTable, s, BI_PDL_CHECK(launch_pdl(rope_table_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, theta, hd, max_pos, cs, sn)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

}  // namespace bi

extern "C" bi_status bi_embed(const int32_t* ids, const void* table, void* out, int64_t T, int64_t d, int64_t vocab,
                              bi_stream s) {
  bi::clear_error();
  return bi::embed_impl(ids, table, out, T, d, vocab, reinterpret_cast<cudaStream_t>(s));
}

extern "C" bi_status bi_rope_table(double theta, int32_t head_dim, int32_t max_pos, float* cos_out, float* sin_out,
                                   bi_stream s) {
  bi::clear_error();
  return bi::rope_table_impl(theta, head_dim, max_pos, cos_out, sin_out, reinterpret_cast<cudaStream_t>(s));
}

namespace bi {

int take_pointwise_device_error(cudaStream_t s, int32_t* code) {
  unsigned v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_pw_err_word, sizeof(v), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return 1;
  if (cudaStreamSynchronize(s) != cudaSuccess) return 1;
  if (v != 0) {
    unsigned zero = 0;
    if (cudaMemcpyToSymbolAsync(g_pw_err_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return 1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return 1;
  }
  *code = static_cast<int32_t>(v);
  return 0;
}

}  // namespace bi

extern "C" bi_status bi_qkv_rope_store(const void* qkv, const float* rope_cos, const float* rope_sin,
                                       const int32_t* token_pos, const int32_t* token_req, const int32_t* block_table,
                                       int32_t T, const bi_attn_dims* dims, void* q_out, void* k_cache, void* v_cache,
                                       bi_stream s) {
  bi::clear_error();
  return bi::qkv_rope_store_impl(qkv, rope_cos, rope_sin, token_pos, token_req, block_table, T, dims, q_out, k_cache,
                                 v_cache, reinterpret_cast<cudaStream_t>(s), nullptr, nullptr, 0.f, false, INT32_MAX);
}

extern "C" bi_status bi_swiglu(const void* gu, void* out, int64_t T, int64_t F, bi_stream s) {
  bi::clear_error();
  return bi::swiglu_impl(gu, out, T, F, reinterpret_cast<cudaStream_t>(s));
}
