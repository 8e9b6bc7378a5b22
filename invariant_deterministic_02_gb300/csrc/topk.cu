// Deterministic per-row top-k of fp32 logits.
//
// Greedy decoding only picks the largest of the logits it is given, so equal
// logits are required for equal tokens, and near-ties are where tiny numeric
// differences flip the choice (zhaixingw.cn post on BlockLock, "坑清单" items 2
// and 5; LLM full-stack book section 19.7.4).  The order used here is (value
// descending, index ascending): a total order, so the selected set and its
// order are unique and do not depend on how the scan is parallelised.
//
// One CTA of 32 warps per row.  Each warp scans a contiguous segment of the row
// (four consecutive elements per lane per step, 16-byte loads) and keeps its
// best k in a sorted list spread over its lanes (lane j holds entry j); an
// element enters only if it beats the list's last entry, so after the first few
// steps almost every step is one compare and one ballot.  Warp 0 then folds the
// 32 warp lists into one with the same insertion.
#include <climits>

#include "common.cuh"

namespace bi {
namespace {

constexpr int kTopkWarps = 32;

__device__ __forceinline__ bool better(float av, int ai, float bv, int bi) { return av > bv || (av == bv && ai < bi); }

// Insert (v, i) into the warp's sorted list (lanes < k hold entries, best first);
// the caller has checked that it beats entry k-1.
__device__ __forceinline__ void warp_insert(float& lv, int& li, float v, int i, int lane, int k) {
  const unsigned m = __ballot_sync(0xffffffffu, lane < k && better(lv, li, v, i));
  const int p = __popc(m);  // entries that stay ahead of the new one
  const float uv = __shfl_up_sync(0xffffffffu, lv, 1);
  const int ui = __shfl_up_sync(0xffffffffu, li, 1);
  if (lane < k) {
    if (lane == p) {
      lv = v;
      li = i;
    } else if (lane > p) {
      lv = uv;
      li = ui;
    }
  }
}

// Offer the 32 candidates held one per lane to the list.
__device__ __forceinline__ void warp_offer(float& lv, int& li, float& tv, int& ti, float cv, int ci, int lane,
                                           int k) {
  unsigned mask = __ballot_sync(0xffffffffu, better(cv, ci, tv, ti));
  while (mask) {
    const int src = __ffs(mask) - 1;
    mask &= mask - 1;
    const float v = __shfl_sync(0xffffffffu, cv, src);
    const int i = __shfl_sync(0xffffffffu, ci, src);
    if (better(v, i, tv, ti)) {
      warp_insert(lv, li, v, i, lane, k);
      tv = __shfl_sync(0xffffffffu, lv, k - 1);
      ti = __shfl_sync(0xffffffffu, li, k - 1);
    }
  }
}

__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(const float* __restrict__ logits, int64_t V, int k,
                                                               float* __restrict__ top_v, int32_t* __restrict__ top_i,
                                                               int32_t* __restrict__ greedy) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sv[kTopkWarps][32];
  __shared__ int si[kTopkWarps][32];
  const int64_t row = blockIdx.x;
  const float* x = logits + row * V;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  float lv = -INFINITY, tv = -INFINITY;
  int li = INT_MAX, ti = INT_MAX;
  // segment of this warp: a multiple of 128 elements
  const int64_t per = ((V + kTopkWarps - 1) / kTopkWarps + 127) / 128 * 128;
  const int64_t s0 = warp * per, s1 = min(V, s0 + per);
  const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
  int64_t e = s0;
  if (vec) {
    for (; e + 128 <= s1; e += 128) {
      const float4 f = *reinterpret_cast<const float4*>(x + e + 4 * lane);
      const int base = static_cast<int>(e) + 4 * lane;
      warp_offer(lv, li, tv, ti, f.x, base, lane, k);
      warp_offer(lv, li, tv, ti, f.y, base + 1, lane, k);
      warp_offer(lv, li, tv, ti, f.z, base + 2, lane, k);
      warp_offer(lv, li, tv, ti, f.w, base + 3, lane, k);
    }
  }
  for (; e < s1; e += 32) {
    const int64_t idx = e + lane;
    const float v = idx < s1 ? x[idx] : -INFINITY;
    warp_offer(lv, li, tv, ti, v, idx < s1 ? static_cast<int>(idx) : INT_MAX, lane, k);
  }
  sv[warp][lane] = lv;
  si[warp][lane] = li;
  __syncthreads();
  if (warp == 0) {
    lv = sv[0][lane];
    li = si[0][lane];
    tv = __shfl_sync(0xffffffffu, lv, k - 1);
    ti = __shfl_sync(0xffffffffu, li, k - 1);
    for (int w = 1; w < kTopkWarps; ++w) {
      const float cv = lane < k ? sv[w][lane] : -INFINITY;
      const int ci = lane < k ? si[w][lane] : INT_MAX;
      warp_offer(lv, li, tv, ti, cv, ci, lane, k);
    }
    if (lane < k) {
      top_v[row * k + lane] = lv;
      top_i[row * k + lane] = li;
    }
    if (greedy != nullptr && lane == 0) greedy[row] = li;
  }
}

}  // namespace

bi_status topk_impl(const float* logits, int64_t rows, int64_t V, int32_t k, float* tv, int32_t* ti,
                    int32_t* greedy, cudaStream_t s) {
  BI_REQUIRE(rows >= 0 && V >= 1 && V < INT_MAX, BI_ERR_INVALID_ARG, "bi_topk: rows=%lld V=%lld",
             static_cast<long long>(rows), static_cast<long long>(V));
  BI_REQUIRE(k >= 1 && k <= BI_TOPK_MAX && k <= V, BI_ERR_UNSUPPORTED, "bi_topk: k=%d (1..%d, <= V)", k, BI_TOPK_MAX);
  if (rows == 0) return BI_OK;
  BI_REQUIRE(logits && tv && ti, BI_ERR_INVALID_ARG, "bi_topk: null pointer");
  BI_TIMED(::bi::kTagTopk, s,
           BI_PDL_CHECK(launch_pdl(topk_kernel, dim3(static_cast<unsigned>(rows)), dim3(kTopkWarps * 32), 0, s, logits, V, k, tv, ti, greedy)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

}  // namespace bi

extern "C" bi_status bi_topk(const float* logits, int64_t rows, int64_t V, int32_t k, float* top_v, int32_t* top_i,
                             bi_stream s) {
  bi::clear_error();
  return bi::topk_impl(logits, rows, V, k, top_v, top_i, nullptr, reinterpret_cast<cudaStream_t>(s));
}
