// Batch-invariant RMSNorm.
//
// y[r][j] = x[r][j] * (1 / sqrt(mean_j x[r][j]^2 + eps)) * gamma[j]
// ("Batch-Invariant Kernel" notes, section RMSNorm: the formula and the
// data-parallel reduction in which one CTA owns a whole row; devpress digest of
// "Defeating Nondeterminism in LLM Inference", section 3.1).
//
// INVARIANT: one CTA of 256 threads per row, whatever the number of rows.
// Thread t loads 16-byte vectors t, t+256, t+512, ... of the row, accumulates
// their squares in order with fused multiply-adds, the warp reduces with a
// fixed xor-butterfly, and the eight warp sums are combined in a fixed pairwise
// tree.  The whole order depends on d only.  A grid-stride loop over rows keeps
// the grid a multiple of the SM count without touching any row's arithmetic.
//
// FAST (the non-invariant schedule the pages describe): when there are fewer
// rows than SMs, each row is split over several CTAs whose partial sums are
// combined in a second pass, so a row's reduction order depends on the batch.
//
// fp32-activation layers: x fp32, gamma bf16 (weights stay 16-bit), y written
// as three bf16 planes for the GEMM that consumes it (common.cuh).
#include "common.cuh"

namespace bi {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxChunks = 8;  // register-resident 16-byte vectors per thread
constexpr int kSplitThreads = 128;

template <typename T>
struct VecOf;
template <>
struct VecOf<float> {
  static constexpr int N = 4;
};
template <>
struct VecOf<__nv_bfloat16> {
  static constexpr int N = 8;
};

__device__ __forceinline__ void load_vec(const float* p, float (&f)[4]) {
  float4 v = *reinterpret_cast<const float4*>(p);
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float (&f)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  unpack8(u, f);
}
__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float (&f)[4]) {
  uint2 u = *reinterpret_cast<const uint2*>(p);
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
}
__device__ __forceinline__ void store_vec(float* p, const float (&f)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
}
__device__ __forceinline__ void store_vec(__nv_bfloat16* p, const float (&f)[8]) {
  *reinterpret_cast<uint4*>(p) = pack8(f);
}

// Output of V values at element offset off of row y: the input type, or
// (PL, fp32 input) three bf16 planes `plane` elements apart.
template <typename TX, bool PL, int V>
__device__ __forceinline__ void store_out(void* y, size_t plane, size_t off, const float (&o)[V]) {
  if constexpr (PL) {
    static_assert(V == 4, "planes are written from fp32 rows");
    store_planes4(static_cast<uint16_t*>(y) + off, plane, o[0], o[1], o[2], o[3]);
  } else {
    store_vec(static_cast<TX*>(y) + off, o);
  }
}

// Fixed xor-butterfly: every lane ends with the same bits (fp add commutes).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// Sum of the eight warp partials in a fixed pairwise tree (every thread computes it).
__device__ __forceinline__ float sum8(const float* r) {
  float a = __fadd_rn(__fadd_rn(r[0], r[1]), __fadd_rn(r[2], r[3]));
  float b = __fadd_rn(__fadd_rn(r[4], r[5]), __fadd_rn(r[6], r[7]));
  return __fadd_rn(a, b);
}

__device__ __forceinline__ float inv_rms(float sumsq, int d, float eps) {
  float mean = __fdiv_rn(sumsq, static_cast<float>(d));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
}

// The invariant computation of one row by one CTA of kThreads threads; y and
// plane: the row's output (element offsets within it as for x).
template <typename TX, typename TG, bool PL>
__device__ __forceinline__ void rms_row(const TX* __restrict__ x, const TG* __restrict__ gamma, void* y, size_t plane,
                                        int d, float eps, float* red) {
  constexpr int V = VecOf<TX>::N;
  const int nchunks = d / V;
  const int t = threadIdx.x;
  float xs[kMaxChunks][V];
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxChunks; ++i) {
    const int c = t + i * kThreads;
    if (c < nchunks) {
      load_vec(x + static_cast<size_t>(c) * V, xs[i]);
#pragma unroll
      for (int e = 0; e < V; ++e) acc = __fmaf_rn(xs[i][e], xs[i][e], acc);
    }
  }
  acc = warp_sum(acc);
  if ((t & 31) == 0) red[t >> 5] = acc;
  __syncthreads();
  const float r = inv_rms(sum8(red), d, eps);
  __syncthreads();  // red is reused by the next row
#pragma unroll
  for (int i = 0; i < kMaxChunks; ++i) {
    const int c = t + i * kThreads;
    if (c < nchunks) {
      float g[V], o[V];
      load_vec(gamma + static_cast<size_t>(c) * V, g);
#pragma unroll
      for (int e = 0; e < V; ++e) o[e] = __fmul_rn(__fmul_rn(xs[i][e], r), g[e]);
      store_out<TX, PL, V>(y, plane, static_cast<size_t>(c) * V, o);
    }
  }
}

// Output row r of y (the row's first element; planes share the row offset).
template <typename TX, bool PL>
__device__ __forceinline__ void* out_row(void* y, int64_t r, int d) {
  if constexpr (PL) return static_cast<uint16_t*>(y) + r * d;
  else return static_cast<TX*>(y) + r * d;
}

// Raw 16-byte vectors of a row (NCH per thread, chunk c = t + 256 i) and their
// conversion: the row data stays packed in registers until it is used.
template <typename TX>
struct RawOf;
template <>
struct RawOf<float> {
  using T = float4;
  static __device__ __forceinline__ void unpack(const float4& v, float (&f)[4]) {
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
};
template <>
struct RawOf<__nv_bfloat16> {
  using T = uint4;
  static __device__ __forceinline__ void unpack(const uint4& v, float (&f)[8]) { unpack8(v, f); }
};

template <typename TX, int NCH>
__device__ __forceinline__ void load_row(const TX* __restrict__ x, int nchunks, typename RawOf<TX>::T (&raw)[NCH]) {
  using R = typename RawOf<TX>::T;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int c = threadIdx.x + i * kThreads;
    if (c < nchunks) {
      const uint4 u = ld_stream(reinterpret_cast<const R*>(x) + c);
      raw[i] = *reinterpret_cast<const R*>(&u);
    }
  }
}

// INVARIANT kernel: a grid-stride loop over rows, one row per CTA at a time,
// the next row's vectors loaded before the current row is reduced so that two
// rows per CTA are in flight.  NCH = 16-byte vectors per thread (d / (V * 256),
// rounded up): the row lives in registers, so the register count, and with it
// the number of resident CTAs, follows d.  The arithmetic is rms_row's: the
// same per-thread order, warp butterfly and pairwise tree of warp sums.
template <typename TX, typename TG, bool PL, int NCH>
__global__ void __launch_bounds__(kThreads) rms_invariant_kernel(const TX* __restrict__ x, const TG* __restrict__ gamma,
                                                                 void* y, size_t plane, int64_t row_begin,
                                                                 int64_t row_end, int d, float eps) {
  using R = typename RawOf<TX>::T;
  constexpr int V = VecOf<TX>::N;
  pdl_wait();
  pdl_trigger();
  __shared__ float red[kWarps];
  const int t = threadIdx.x;
  const int nchunks = d / V;
  int64_t r = row_begin + blockIdx.x;
  R cur[NCH], nxt[NCH];
  if (r < row_end) load_row<TX, NCH>(x + r * d, nchunks, cur);
  for (; r < row_end; r += gridDim.x) {
    const int64_t rn = r + gridDim.x;
    if (rn < row_end) load_row<TX, NCH>(x + rn * d, nchunks, nxt);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      if (t + i * kThreads < nchunks) {
        float f[V];
        RawOf<TX>::unpack(cur[i], f);
#pragma unroll
        for (int e = 0; e < V; ++e) acc = __fmaf_rn(f[e], f[e], acc);
      }
    }
    acc = warp_sum(acc);
    if ((t & 31) == 0) red[t >> 5] = acc;
    __syncthreads();
    const float rr = inv_rms(sum8(red), d, eps);
    __syncthreads();  // red is reused by the next row
    void* yr = out_row<TX, PL>(y, r, d);
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int c = t + i * kThreads;
      if (c < nchunks) {
        float f[V], g[V], o[V];
        RawOf<TX>::unpack(cur[i], f);
        load_vec(gamma + static_cast<size_t>(c) * V, g);
#pragma unroll
        for (int e = 0; e < V; ++e) o[e] = __fmul_rn(__fmul_rn(f[e], rr), g[e]);
        store_out<TX, PL, V>(yr, plane, static_cast<size_t>(c) * V, o);
      }
    }
#pragma unroll
    for (int i = 0; i < NCH; ++i) cur[i] = nxt[i];
  }
}

// FAST pass 1: CTA (row, s) sums the squares of chunk range s of its row.
template <typename TX>
__global__ void __launch_bounds__(kSplitThreads) rms_split_partial_kernel(const TX* __restrict__ x, float* partial,
                                                                          int64_t rows, int d, int splits,
                                                                          int64_t skip_begin, int64_t skip_end) {
  pdl_wait();
  pdl_trigger();
  constexpr int V = VecOf<TX>::N;
  const int64_t r = blockIdx.x / splits;
  const int s = blockIdx.x % splits;
  if (r >= rows || (r >= skip_begin && r < skip_end)) return;
  const int nchunks = d / V;
  const int per = (nchunks + splits - 1) / splits;
  const int c0 = s * per, c1 = min(nchunks, c0 + per);
  float acc = 0.f;
  for (int c = c0 + threadIdx.x; c < c1; c += kSplitThreads) {
    float f[V];
    load_vec(x + r * d + static_cast<int64_t>(c) * V, f);
#pragma unroll
    for (int e = 0; e < V; ++e) acc = __fmaf_rn(f[e], f[e], acc);
  }
  acc = warp_sum(acc);
  __shared__ float red[kSplitThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < kSplitThreads / 32; ++w) tot = __fadd_rn(tot, red[w]);
    partial[r * splits + s] = tot;
  }
}

// FAST pass 2: one CTA per row; split rows add their partials left to right,
// rows in [inv_begin, inv_end) run the invariant row function instead.
template <typename TX, typename TG, bool PL>
__global__ void __launch_bounds__(kThreads) rms_split_finish_kernel(const TX* __restrict__ x,
                                                                    const TG* __restrict__ gamma, void* y, size_t plane,
                                                                    const float* partial, int64_t rows, int d,
                                                                    int splits, float eps, int64_t inv_begin,
                                                                    int64_t inv_end) {
  pdl_wait();
  pdl_trigger();
  constexpr int V = VecOf<TX>::N;
  __shared__ float red[kWarps];
  const int64_t r = blockIdx.x;
  if (r >= rows) return;
  void* yr = out_row<TX, PL>(y, r, d);
  if (r >= inv_begin && r < inv_end) {
    rms_row<TX, TG, PL>(x + r * d, gamma, yr, plane, d, eps, red);
    return;
  }
  float tot = 0.f;
  for (int s = 0; s < splits; ++s) tot = __fadd_rn(tot, partial[r * splits + s]);
  const float rr = inv_rms(tot, d, eps);
  const int nchunks = d / V;
  for (int c = threadIdx.x; c < nchunks; c += kThreads) {
    float f[V], g[V], o[V];
    load_vec(x + r * d + static_cast<int64_t>(c) * V, f);
    load_vec(gamma + static_cast<int64_t>(c) * V, g);
#pragma unroll
    for (int e = 0; e < V; ++e) o[e] = __fmul_rn(__fmul_rn(f[e], rr), g[e]);
    store_out<TX, PL, V>(yr, plane, static_cast<size_t>(c) * V, o);
  }
}

int fast_splits(int64_t rows, int d, int vec) {
  const int sms = num_sms();
  if (rows <= 0 || rows >= sms) return 1;
  const int by_sms = static_cast<int>(sms / rows);
  const int by_work = max(1, (d / vec) / kSplitThreads);
  return max(1, min(by_sms, by_work));
}

template <typename TX, typename TG, bool PL>
bi_status launch(const void* xv, const void* gv, void* y, int64_t rows, int d, float eps, bi_mode mode,
                 int64_t tb, int64_t te, void* ws, size_t ws_bytes, cudaStream_t s) {
  const TX* x = static_cast<const TX*>(xv);
  const TG* g = static_cast<const TG*>(gv);
  const size_t plane = static_cast<size_t>(rows) * d;
  constexpr int V = VecOf<TX>::N;
  const int splits = mode_invariant(mode) ? 1 : fast_splits(rows, d, V);
  if (splits == 1) {
    // Unsplit: the data-parallel schedule, identical to INVARIANT for every row.
    const int nch = (d / V + kThreads - 1) / kThreads;
    auto go = [&](auto kern) -> bi_status {
      const void* fn = reinterpret_cast<const void*>(kern);
      // every SM holds as many CTAs as its registers allow, each working through rows
      const int64_t grid =
          std::min<int64_t>(rows, static_cast<int64_t>(num_sms()) * occupancy_per_sm(fn, kThreads, 0));
      BI_TIMED(::bi::kTagRmsnorm, s, BI_PDL_CHECK(launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0,
                                                             s, x, g, y, plane, int64_t(0), rows, d, eps)));
      BI_LAUNCH_CHECK();
      return BI_OK;
    };
    if (nch <= 1) return go(rms_invariant_kernel<TX, TG, PL, 1>);
    if (nch <= 2) return go(rms_invariant_kernel<TX, TG, PL, 2>);
    if (nch <= 4) return go(rms_invariant_kernel<TX, TG, PL, 4>);
    return go(rms_invariant_kernel<TX, TG, PL, kMaxChunks>);
  }
  const size_t need = static_cast<size_t>(rows) * splits * sizeof(float);
  BI_REQUIRE(ws != nullptr && ws_bytes >= need, BI_ERR_WORKSPACE, "bi_rmsnorm: workspace %zu < %zu bytes", ws_bytes,
             need);
  float* partial = static_cast<float*>(ws);
  BI_TIMED(::bi::kTagRmsnormSplit, s, BI_PDL_CHECK(launch_pdl(rms_split_partial_kernel<TX>, dim3(static_cast<unsigned>(rows * splits)), dim3(kSplitThreads), 0, s, x, partial, rows, d,
                                                                                             splits, tb, te)));
  BI_LAUNCH_CHECK();
  BI_TIMED(::bi::kTagRmsnormSplit, s, BI_PDL_CHECK(launch_pdl(rms_split_finish_kernel<TX, TG, PL>, dim3(static_cast<unsigned>(rows)), dim3(kThreads), 0, s, x, g, y, plane, partial, rows, d, splits, eps,
                                                                              tb, te)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

bi_status check_target(bi_mode mode, int64_t rows, int32_t target_row, int32_t target_count, int64_t* tb,
                       int64_t* te) {
  *tb = 0;
  *te = 0;
  if (mode != BI_MODE_PROTECTED || target_row < 0) return BI_OK;
  BI_REQUIRE(target_count >= 1 && target_row + static_cast<int64_t>(target_count) <= rows, BI_ERR_INVALID_ARG,
             "target rows [%d, %d) outside [0, %lld)", target_row, target_row + target_count,
             static_cast<long long>(rows));
  *tb = target_row;
  *te = target_row + static_cast<int64_t>(target_count);
  return BI_OK;
}

}  // namespace

bi_status rmsnorm_impl(const void* x, const void* gamma, void* y, int64_t rows, int64_t d, bi_dtype dtype, float eps,
                       bi_mode mode, int32_t target_row, int32_t target_count, void* ws, size_t ws_bytes,
                       cudaStream_t s) {
  clear_error();
  BI_REQUIRE(rows >= 0 && d > 0, BI_ERR_INVALID_ARG, "bi_rmsnorm: rows=%lld d=%lld", static_cast<long long>(rows),
             static_cast<long long>(d));
  BI_REQUIRE(dtype == BI_F32 || dtype == BI_BF16, BI_ERR_UNSUPPORTED, "bi_rmsnorm: dtype %d", static_cast<int>(dtype));
  BI_REQUIRE(mode_valid(mode), BI_ERR_INVALID_ARG, "bi_rmsnorm: mode %d",
             static_cast<int>(mode));
  const int vec = dtype == BI_F32 ? 4 : 8;
  BI_REQUIRE(d % vec == 0 && d / vec <= kThreads * kMaxChunks, BI_ERR_UNSUPPORTED,
             "bi_rmsnorm: d=%lld must be a multiple of %d and at most %d", static_cast<long long>(d), vec,
             kThreads * kMaxChunks * vec);
  BI_REQUIRE(eps >= 0.f && eps == eps, BI_ERR_INVALID_ARG, "bi_rmsnorm: eps must be >= 0");
  int64_t tb, te;
  BI_TRY(check_target(mode, rows, target_row, target_count, &tb, &te));
  if (rows == 0) return BI_OK;
  BI_REQUIRE(x && gamma && y, BI_ERR_INVALID_ARG, "bi_rmsnorm: null pointer");
  BI_REQUIRE(aligned16(x) && aligned16(gamma) && aligned16(y), BI_ERR_INVALID_ARG,
             "bi_rmsnorm: pointers must be 16-byte aligned");
  if (dtype == BI_F32)
    return launch<float, float, false>(x, gamma, y, rows, static_cast<int>(d), eps, mode, tb, te, ws, ws_bytes, s);
  return launch<__nv_bfloat16, __nv_bfloat16, false>(x, gamma, y, rows, static_cast<int>(d), eps, mode, tb, te, ws,
                                                     ws_bytes, s);
}

// fp32-activation layers: x fp32 [rows][d], gamma bf16 [d], y three bf16 planes
// [3][rows][d] (rows*d elements apart).  Same reduction order as bi_rmsnorm on
// fp32 rows.
bi_status rmsnorm_planes_impl(const void* x, const void* gamma, void* y, int64_t rows, int64_t d, float eps,
                              bi_mode mode, int32_t target_row, int32_t target_count, void* ws, size_t ws_bytes,
                              cudaStream_t s) {
  BI_REQUIRE(rows >= 0 && d > 0 && d % 4 == 0 && d / 4 <= kThreads * kMaxChunks, BI_ERR_UNSUPPORTED,
             "rmsnorm (fp32 activations): rows=%lld d=%lld", static_cast<long long>(rows), static_cast<long long>(d));
  BI_REQUIRE(mode_valid(mode), BI_ERR_INVALID_ARG, "rmsnorm: mode %d", static_cast<int>(mode));
  int64_t tb, te;
  BI_TRY(check_target(mode, rows, target_row, target_count, &tb, &te));
  if (rows == 0) return BI_OK;
  BI_REQUIRE(x && gamma && y && aligned16(x) && aligned16(gamma) && aligned16(y), BI_ERR_INVALID_ARG,
             "rmsnorm (fp32 activations): null or misaligned pointer");
  return launch<float, __nv_bfloat16, true>(x, gamma, y, rows, static_cast<int>(d), eps, mode, tb, te, ws, ws_bytes, s);
}

size_t rmsnorm_ws(int64_t rows, int64_t d, bi_mode mode) {
  if (mode_invariant(mode) || rows <= 0) return 0;
  const int sms = num_sms();
  if (rows >= sms) return 0;
  return static_cast<size_t>(rows) * sms * sizeof(float);
}

}  // namespace bi

extern "C" size_t bi_rmsnorm_workspace(int64_t rows, int64_t d, bi_mode mode) { return bi::rmsnorm_ws(rows, d, mode); }

extern "C" bi_status bi_rmsnorm(const void* x, const void* gamma, void* y, int64_t rows, int64_t d, bi_dtype dtype,
                                float eps, bi_mode mode, int32_t target_row, int32_t target_count, void* workspace,
                                size_t ws_bytes, bi_stream s) {
  return bi::rmsnorm_impl(x, gamma, y, rows, d, dtype, eps, mode, target_row, target_count, workspace, ws_bytes,
                          reinterpret_cast<cudaStream_t>(s));
}
