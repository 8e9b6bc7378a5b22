// Deterministic per-row top-k of fp32 logits.
//
// Greedy decoding only picks the largest of the logits it is given, so equal
// logits are required for equal tokens, and near-ties are where tiny numeric
// differences flip the choice (zhaixingw.cn post on BlockLock, "坑清单" items 2
// and 5; LLM full-stack book section 19.7.4).  The order used here is (value
// descending, index ascending): a total order, so the selected set and its
// order are unique and do not depend on how the scan is parallelised.
//
// A cluster of four CTAs of 16 warps per row (the row's 64 warps on up to four
// SMs, whose load capacity they share).  Each warp scans a contiguous segment of the row
// (8 consecutive elements per lane per step as two 16-byte loads, the next
// step's loads issued before the current step is examined) and keeps its best k
// in a sorted list spread over its lanes (lane j holds entry j).  Elements are
// offered to the list only when they beat a filter: a lower bound on the row's
// k-th entry.  Any warp's own k-th entry is such a bound (that warp alone holds k
// entries at least as good), so the warps publish theirs to a shared maximum
// after every step; before its list fills, a warp uses the k-th largest of its
// lanes' maxima over the first step (k distinct elements reach it).  An element
// that fails the filter cannot be among the row's k best, so skipping it changes
// nothing, and almost every step is two loads, eight compares and one vote.
// The 16 warp lists of a CTA are then folded pairwise in four rounds (8, 4, 2,
// 1 warps), each warp merging its partner's list into its own with a bitonic
// merge, and the first CTA of the cluster merges the other three CTAs' lists
// (read from their shared memory) into its own.  The selected set and its order are unique under the
// total order, so how the row is cut up does not change the result.
#include <climits>

#include <cooperative_groups.h>

#include "common.cuh"

namespace bi {
namespace {

constexpr int kTopkWarps = 16;
constexpr int kTopkCtas = 4;  // CTAs (one cluster) per row

__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
  const uint4 u = ld_stream(p);
  return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
}

__device__ __forceinline__ bool better(float av, int ai, float bv, int bi) { return av > bv || (av == bv && ai < bi); }

// 64-bit key ordered like `better` for non-NaN values: the float's bits mapped to
// an unsigned integer of the same order (-0 taken as +0, which compare equal),
// then the index reversed so that the lower index is the larger key.
__device__ __forceinline__ unsigned long long entry_key(float v, int i) {
  unsigned u = __float_as_uint(v == 0.f ? 0.f : v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) | (0xffffffffu - static_cast<unsigned>(i));
}

// Descending bitonic sort of one value per lane across the warp.
__device__ __forceinline__ float warp_sort_desc(float v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool lower = (lane & stride) == 0;     // this lane keeps the larger value if descending here
      const bool desc = (lane & size) == 0 || size == 32;
      v = (lower == desc) ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
}

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

// Merge of two lists of 32 entries, each sorted best first (lane j holds entry
// j; unused entries are (-inf, INT_MAX), worse than any element), keeping the
// 32 best in order: the better of own[j] and other[31 - j] form a bitonic
// sequence holding the 32 best of both, which five half-cleaner stages of a
// bitonic network sort.  `better` is a total order, so the result is unique.
__device__ __forceinline__ void warp_merge32(float& lv, int& li, float rv, int ri, int lane) {
  // rv, ri: the other list's entry 31 - lane
  if (better(rv, ri, lv, li)) {
    lv = rv;
    li = ri;
  }
#pragma unroll
  for (int stride = 16; stride >= 1; stride >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, lv, stride);
    const int oi = __shfl_xor_sync(0xffffffffu, li, stride);
    const bool keep_better = (lane & stride) == 0;  // the lower lane of the pair takes the better entry
    const bool other_better = better(ov, oi, lv, li);
    if (keep_better == other_better) {
      lv = ov;
      li = oi;
    }
  }
}

__global__ void __cluster_dims__(kTopkCtas, 1, 1) __launch_bounds__(kTopkWarps * 32)
    topk_kernel(const float* __restrict__ logits, int64_t V, int k, float* __restrict__ top_v,
                int32_t* __restrict__ top_i, int32_t* __restrict__ greedy) {
  constexpr int kU = 2;               // 16-byte loads per lane per step
  constexpr int kStep = kU * 4 * 32;  // elements per warp step
  static_assert(kU * kTopkWarps == 32, "one first-step group maximum per lane of the sorting warp");
  __shared__ float sv[kTopkWarps][32];
  __shared__ int si[kTopkWarps][32];
  __shared__ unsigned long long s_filter;  // the best k-th entry any warp has published (a key)
  __shared__ float s_gmax[kU * kTopkWarps];  // maxima of the 128-element groups of every warp's first step
  if (threadIdx.x == 0) s_filter = 0ull;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int part = static_cast<int>(cluster.block_rank());
  const int64_t row = blockIdx.x / kTopkCtas;
  const float* x = logits + row * V;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  float lv = -INFINITY, tv = -INFINITY;
  int li = INT_MAX, ti = INT_MAX;
  unsigned long long filter = 0ull, published = 0ull;
  // segment of this warp (warp `part * 16 + warp` of the row's 64): a multiple of kStep elements
  constexpr int kRowWarps = kTopkWarps * kTopkCtas;
  const int64_t per = ((V + kRowWarps - 1) / kRowWarps + kStep - 1) / kStep * kStep;
  const int64_t s0 = min(V, (part * kTopkWarps + warp) * per), s1 = min(V, s0 + per);
  const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
  int64_t e = s0;
  const bool vec_run = vec && e + kStep <= s1;  // warp-uniform
  float4 cur[kU], nxt[kU];
  {
    // First filter, from the first step's elements (NaNs are never kept): the k-th largest of the warp's
    // 32 lane maxima, and the k-th largest of the CTA's 32 group maxima (each warp's first step is two
    // groups of 128 consecutive elements, one per 16-byte load of its lanes).  Each is the k-th largest
    // of maxima of disjoint groups, so at least k elements of the row reach it; the second is the much
    // tighter one, so few elements get past it before the lists fill.
    float m = -INFINITY, gm[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) gm[u] = -INFINITY;
    if (vec_run) {
#pragma unroll
      for (int u = 0; u < kU; ++u) cur[u] = ld_stream_f4(x + e + 128 * u + 4 * lane);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const float mu = fmaxf(fmaxf(cur[u].x, cur[u].y), fmaxf(cur[u].z, cur[u].w));
        gm[u] = mu == mu ? mu : -INFINITY;
        m = fmaxf(m, mu);
      }
    }
    const float tw = __shfl_sync(0xffffffffu, warp_sort_desc(m == m ? m : -INFINITY, lane), k - 1);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      float g = gm[u];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, o));
      if (lane == 0) s_gmax[kU * warp + u] = g;
    }
    __syncthreads();
    const float tc = __shfl_sync(0xffffffffu, warp_sort_desc(s_gmax[lane], lane), k - 1);
    filter = entry_key(fmaxf(tw, tc), INT_MAX);
  }
  if (vec_run) {
    for (;;) {
      const int64_t en = e + kStep;
      const bool more = en + kStep <= s1;
      if (more) {
#pragma unroll
        for (int u = 0; u < kU; ++u) nxt[u] = ld_stream_f4(x + en + 128 * u + 4 * lane);
      }
      bool any = false;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int base = static_cast<int>(e) + 128 * u + 4 * lane;
        any |= (entry_key(cur[u].x, base) > filter) | (entry_key(cur[u].y, base + 1) > filter) |
               (entry_key(cur[u].z, base + 2) > filter) | (entry_key(cur[u].w, base + 3) > filter);
      }
      if (__any_sync(0xffffffffu, any)) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int base = static_cast<int>(e) + 128 * u + 4 * lane;
          const float c[4] = {cur[u].x, cur[u].y, cur[u].z, cur[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const bool pass = entry_key(c[q], base + q) > filter;
            warp_offer(lv, li, tv, ti, pass ? c[q] : -INFINITY, pass ? base + q : INT_MAX, lane, k);
          }
        }
        if (ti != INT_MAX) {
          // the list is full: its k-th entry bounds the row's from below
          const unsigned long long key = entry_key(tv, ti);
          if (key > published) {
            published = key;
            if (lane == 0) atomicMax(&s_filter, key);
          }
        }
      }
      filter = max(filter, max(published, *reinterpret_cast<volatile unsigned long long*>(&s_filter)));
      e = en;
      if (!more) break;
#pragma unroll
      for (int u = 0; u < kU; ++u) cur[u] = nxt[u];
    }
  }
  for (; e < s1; e += 32) {
    const int64_t idx = e + lane;
    const float v = idx < s1 ? x[idx] : -INFINITY;
    const bool pass = idx < s1 && entry_key(v, static_cast<int>(idx)) > filter;
    warp_offer(lv, li, tv, ti, pass ? v : -INFINITY, pass ? static_cast<int>(idx) : INT_MAX, lane, k);
  }
  sv[warp][lane] = lv;
  si[warp][lane] = li;
  __syncthreads();
  // pairwise folds: in the round of h warps, warp w < h merges list w + h into its own
  // (lists hold their k entries in lanes < k and (-inf, INT_MAX) or worse entries after them)
  for (int h = kTopkWarps / 2; h >= 1; h >>= 1) {
    if (warp < h) {
      warp_merge32(lv, li, sv[warp + h][31 - lane], si[warp + h][31 - lane], lane);
      sv[warp][lane] = lv;
      si[warp][lane] = li;
    }
    __syncthreads();
  }
  // every CTA's list is in its shared memory (sv[0], si[0]); the first CTA takes the others' in
  cluster.sync();
  if (part == 0 && warp == 0) {
    for (int r = 1; r < kTopkCtas; ++r) {
      const float* rv = cluster.map_shared_rank(&sv[0][0], r);
      const int* ri = cluster.map_shared_rank(&si[0][0], r);
      warp_merge32(lv, li, rv[31 - lane], ri[31 - lane], lane);
    }
    if (lane < k) {
      top_v[row * k + lane] = lv;
      top_i[row * k + lane] = li;
    }
    if (greedy != nullptr && lane == 0) greedy[row] = li;
  }
  // no CTA leaves (and frees its shared memory) before the first one has read it
  cluster.sync();
}

}  // namespace

bi_status topk_impl(const float* logits, int64_t rows, int64_t V, int32_t k, float* tv, int32_t* ti,
                    int32_t* greedy, cudaStream_t s) {
  BI_REQUIRE(rows >= 0 && rows <= INT_MAX / kTopkCtas && V >= 1 && V < INT_MAX, BI_ERR_INVALID_ARG,
             "bi_topk: rows=%lld V=%lld", static_cast<long long>(rows), static_cast<long long>(V));
  BI_REQUIRE(k >= 1 && k <= BI_TOPK_MAX && k <= V, BI_ERR_UNSUPPORTED, "bi_topk: k=%d (1..%d, <= V)", k, BI_TOPK_MAX);
  if (rows == 0) return BI_OK;
  BI_REQUIRE(logits && tv && ti, BI_ERR_INVALID_ARG, "bi_topk: null pointer");
  BI_TIMED(::bi::kTagTopk, s,
           BI_PDL_CHECK(launch_pdl(topk_kernel, dim3(static_cast<unsigned>(rows * kTopkCtas)), dim3(kTopkWarps * 32), 0, s, logits, V, k, tv, ti, greedy)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

}  // namespace bi

extern "C" bi_status bi_topk(const float* logits, int64_t rows, int64_t V, int32_t k, float* top_v, int32_t* top_i,
                             bi_stream s) {
  bi::clear_error();
  return bi::topk_impl(logits, rows, V, k, top_v, top_i, nullptr, reinterpret_cast<cudaStream_t>(s));
}
