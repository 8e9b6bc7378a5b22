// Deterministic per-row top-k of fp32 logits.
//
// Greedy decoding only picks the largest of the logits it is given, so equal
// logits are required for equal tokens, and near-ties are where tiny numeric
// differences flip the choice (zhaixingw.cn post on BlockLock, "坑清单" items 2
// and 5; LLM full-stack book section 19.7.4).  The order used here is (value
// descending, index ascending): a total order, so the selected set and its
// order are unique and do not depend on how the scan is parallelised.
//
// One CTA of 256 threads per row: thread t scans elements t, t+256, ... keeping
// a sorted register list of the best KCAP, then the 256 lists are merged
// pairwise in shared memory.
#include <climits>

#include "common.cuh"

namespace bi {
namespace {

constexpr int kTopkThreads = 256;

struct Cand {
  float v;
  int i;
};

__device__ __forceinline__ bool better(float av, int ai, float bv, int bi) { return av > bv || (av == bv && ai < bi); }

template <int KCAP>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ logits, int64_t V, int k,
                                                            float* __restrict__ top_v, int32_t* __restrict__ top_i,
                                                            int32_t* __restrict__ greedy) {
  extern __shared__ Cand lists[];  // [kTopkThreads][KCAP]
  const int64_t row = blockIdx.x;
  const float* x = logits + row * V;
  float av[KCAP];
  int ai[KCAP];
#pragma unroll
  for (int j = 0; j < KCAP; ++j) {
    av[j] = -INFINITY;
    ai[j] = INT_MAX;
  }
  for (int64_t e = threadIdx.x; e < V; e += kTopkThreads) {
    const float v = x[e];
    const int idx = static_cast<int>(e);
    if (!better(v, idx, av[KCAP - 1], ai[KCAP - 1])) continue;
#pragma unroll
    for (int j = KCAP - 1; j >= 1; --j) {
      if (better(v, idx, av[j - 1], ai[j - 1])) {
        av[j] = av[j - 1];
        ai[j] = ai[j - 1];
      } else if (better(v, idx, av[j], ai[j])) {
        av[j] = v;
        ai[j] = idx;
      }
    }
    if (better(v, idx, av[0], ai[0])) {
      av[0] = v;
      ai[0] = idx;
    }
  }
  Cand* mine = lists + threadIdx.x * KCAP;
#pragma unroll
  for (int j = 0; j < KCAP; ++j) mine[j] = Cand{av[j], ai[j]};
  __syncthreads();
  // pairwise merges: list t takes the best KCAP of lists t and t + stride
  for (int stride = 1; stride < kTopkThreads; stride <<= 1) {
    if ((threadIdx.x % (2 * stride)) == 0) {
      const Cand* a = lists + threadIdx.x * KCAP;
      const Cand* b = lists + (threadIdx.x + stride) * KCAP;
      Cand out[KCAP];
      int ia = 0, ib = 0;
#pragma unroll
      for (int j = 0; j < KCAP; ++j) {
        const bool take_a = better(a[ia].v, a[ia].i, b[ib].v, b[ib].i);
        out[j] = take_a ? a[ia] : b[ib];
        ia += take_a ? 1 : 0;
        ib += take_a ? 0 : 1;
      }
      Cand* dst = lists + threadIdx.x * KCAP;
#pragma unroll
      for (int j = 0; j < KCAP; ++j) dst[j] = out[j];
    }
    __syncthreads();
  }
  if (threadIdx.x < k) {
    top_v[row * k + threadIdx.x] = lists[threadIdx.x].v;
    top_i[row * k + threadIdx.x] = lists[threadIdx.x].i;
  }
  if (greedy != nullptr && threadIdx.x == 0) greedy[row] = lists[0].i;
}

template <int KCAP>
bi_status launch(const float* logits, int64_t rows, int64_t V, int k, float* tv, int32_t* ti, int32_t* greedy,
                 cudaStream_t s) {
  const size_t smem = sizeof(Cand) * KCAP * kTopkThreads;
  static bool attr = false;
  if (!attr) {
    BI_CUDA_TRY(cudaFuncSetAttribute(topk_kernel<KCAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)));
    attr = true;
  }
  BI_TIMED(::bi::kTagTopk, s, topk_kernel<KCAP><<<static_cast<unsigned>(rows), kTopkThreads, smem, s>>>(logits, V, k, tv, ti, greedy));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

}  // namespace

bi_status topk_impl(const float* logits, int64_t rows, int64_t V, int32_t k, float* tv, int32_t* ti,
                    int32_t* greedy, cudaStream_t s) {
  BI_REQUIRE(rows >= 0 && V >= 1 && V < INT_MAX, BI_ERR_INVALID_ARG, "bi_topk: rows=%lld V=%lld",
             static_cast<long long>(rows), static_cast<long long>(V));
  BI_REQUIRE(k >= 1 && k <= BI_TOPK_MAX && k <= V, BI_ERR_UNSUPPORTED, "bi_topk: k=%d (1..%d, <= V)", k, BI_TOPK_MAX);
  if (rows == 0) return BI_OK;
  BI_REQUIRE(logits && tv && ti, BI_ERR_INVALID_ARG, "bi_topk: null pointer");
  if (k == 1) return launch<1>(logits, rows, V, k, tv, ti, greedy, s);
  if (k <= 8) return launch<8>(logits, rows, V, k, tv, ti, greedy, s);
  return launch<32>(logits, rows, V, k, tv, ti, greedy, s);
}

}  // namespace bi

extern "C" bi_status bi_topk(const float* logits, int64_t rows, int64_t V, int32_t k, float* top_v, int32_t* top_i,
                             bi_stream s) {
  bi::clear_error();
  return bi::topk_impl(logits, rows, V, k, top_v, top_i, nullptr, reinterpret_cast<cudaStream_t>(s));
}
