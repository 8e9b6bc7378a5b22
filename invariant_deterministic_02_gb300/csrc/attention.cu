// Paged split-KV attention: decode and prefill share one split-reduction device function.
//
// Definition (devpress digest of "Defeating Nondeterminism in LLM Inference",
// section 3.3; "Batch-Invariant Kernel" notes, section Flash Attention):
//   out_h = sum_j softmax_j(q_h . k_j * scale) v_j   over keys j <= p (query position p)
// The invariant schedule cuts the keys into fixed splits of 256 absolute
// positions (never a fixed split COUNT), reduces every split at full width with
// masked lanes contributing nothing, and combines the split states with a
// pairwise tree over the split index padded to a constant depth.  Because the
// cached and the new K/V of a request are one sequence in the paged cache, a
// query's reduction order depends on its absolute position only: token-by-token
// decode and any chunked prefill produce the same bits.
//
// Split state of one query head over a split: m = max z (log2 domain), l =
// sum exp2(z - m), o = sum exp2(z - m) v, z = (q.k) * scale * log2(e).
//
// Thread mapping of the split function (one group of 128 threads = 4 warps):
// warp w owns positions [64w, 64w+64) of the split; lane = 8*slot + c; slot is
// the position within a step of 4, c picks dims {8c..8c+7} (and {64+8c..} for
// head_dim 128).  Dot products: per-lane FMA chains in dim order, then a
// xor-butterfly over the 8 lanes (offsets 4, 2, 1).  Sum of exponentials: lane
// L adds positions 8L..8L+7 in order, then a 32-lane butterfly.  Weighted sum
// of values: per-lane FMA chain over the slot's 16 positions in order, xor 8
// then 16 across slots, then the four warp sums added warp 0 + 1 + 2 + 3.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <tuple>
#include <vector>

#include "common.cuh"

namespace bi {
namespace attn {

constexpr int kGroupThreads = 128;
constexpr int kSplit = BI_SPLIT_TOKENS;
constexpr int kPage = BI_PAGE_SIZE;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxFastUnits = 64;
constexpr int kPrefillQBlock = 16;
constexpr int kPrefillGroups = 4;

enum : int { kPlanInvariant = 0, kPlanFast = 1 };

__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "r"(kGroupThreads) : "memory");
}

// Barrier of one group that also returns whether any of its threads passed `p`:
// every thread of the group leaves with the same answer.
__device__ __forceinline__ bool group_any(int group, bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred ip, op;\n\t"
      "setp.ne.u32 ip, %1, 0;\n\t"
      "barrier.red.or.pred op, %2, %3, ip;\n\t"
      "selp.u32 %0, 1, 0, op;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(p)), "r"(group + 1), "r"(kGroupThreads)
      : "memory");
  return r != 0;
}

// Per-group shared scratch of the split function.
// (o is written only after every warp has finished with z and e, so it shares
// their storage: the smaller scratch lets three decode CTAs share an SM.)
template <int HD, int G>
struct SplitSmem {
  union {
    struct {
      float z[G][kSplit];               // scores (log2 domain), -inf where masked
      __align__(16) uint32_t e[kSplit][4]; // weights exp2(z - m) as bf16 (hi, lo) pairs, position-major, heads padded to 4
    };
    __align__(16) float o[4][G][HD];  // per-warp partial weighted sums
  };
  float m[G];
  float l[G];
};

// ------------------------------------------------------------------ mbarrier / bulk-copy helpers
__device__ unsigned int g_attn_err_word = 0;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: after 2 s (or once another thread of the CTA has given up) it
// records `site` in the error word and returns false; callers then carry on
// with whatever shared memory holds, so no thread is ever left waiting on a
// barrier and the kernel always finishes (with wrong values, reported by
// bi_device_error).
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, int site) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u) {
      if (*abort_flag) return false;
      const uint64_t now = global_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitLimitNs) {
        atomicCAS(&g_attn_err_word, 0u, static_cast<unsigned>(site));
        *abort_flag = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, site);
}
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity) && global_ns() - t0 < kWaitLimitNs) {
  }
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Shared-memory layout of K and V (decode ring stages and prefill staging
// alike): a split is four quarters of 64 positions, a quarter four pages of 16
// positions, and a page is stored as HD/64 halves of [16 positions][64 dims]
// (128-byte rows) with the 128-byte swizzle: the 16-byte chunk c of row r sits
// at chunk position c ^ (r & 7).  This is the layout a TMA tensor copy of one
// page writes (box {64 dims, 16 positions, HD/64 halves}), and it lets the
// warp-level MMA fragments (ldmatrix over 8 consecutive positions) read
// shared memory without bank conflicts.
template <int HD>
struct PageLayout {
  static constexpr int kPageBytes = 16 * HD * 2;    // one page of one kv head
  static constexpr int kQuarterBytes = 4 * kPageBytes;
  // byte offset, within a quarter, of the 16-byte chunk `c` (dims 8c .. 8c+7) of position q (0..63)
  static __device__ __forceinline__ int chunk(int q, int c) {
    const int pos = q & 15;
    return (q >> 4) * kPageBytes + (c >> 3) * 2048 + pos * 128 + (((c & 7) ^ (pos & 7)) << 4);
  }
};

// Loaders hand out the K and V pieces of a split; the before_*/after_* hooks
// bracket a warp's reads of its quarter (positions [64w, 64w+64)); they
// synchronise with the copy engine but do no arithmetic.
//
// Decode: quarters of the split stream through a ring of shared-memory stages,
// filled page by page with TMA tensor copies; order K0..K3, V0..V3 per split.
template <int HD>
struct RingKV {
  const unsigned char* ring;  // [stages][quarter bytes], 1024-byte aligned
  uint32_t full0, empty0;     // mbarrier arrays
  int n0;                     // linear stage index of K0 of this split
  int stages;
  volatile int* abort_flag;
  __device__ __forceinline__ int slot(int j) const { return (n0 + j) % stages; }
  __device__ __forceinline__ uint32_t parity(int j) const { return static_cast<uint32_t>(((n0 + j) / stages) & 1); }
  __device__ __forceinline__ const unsigned char* kq(int w) const {
    return ring + static_cast<size_t>(slot(w)) * PageLayout<HD>::kQuarterBytes;
  }
  __device__ __forceinline__ const unsigned char* vq(int w) const {
    return ring + static_cast<size_t>(slot(4 + w)) * PageLayout<HD>::kQuarterBytes;
  }
  __device__ __forceinline__ void before_k(int w) const { wait_bounded(full0 + 8 * slot(w), parity(w), abort_flag, 11); }
  __device__ __forceinline__ void after_k(int w) const {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(empty0 + 8 * slot(w));
  }
  __device__ __forceinline__ void before_v(int w) const {
    wait_bounded(full0 + 8 * slot(4 + w), parity(4 + w), abort_flag, 12);
  }
  __device__ __forceinline__ void after_v(int w) const {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(empty0 + 8 * slot(4 + w));
  }
};

// Prefill: the split's keys and values are staged whole in shared memory, in
// the same layout (quarter w at w * quarter bytes).
template <int HD>
struct SmemKV {
  const unsigned char* ks;
  const unsigned char* vs;
  __device__ __forceinline__ const unsigned char* kq(int w) const { return ks + w * PageLayout<HD>::kQuarterBytes; }
  __device__ __forceinline__ const unsigned char* vq(int w) const { return vs + w * PageLayout<HD>::kQuarterBytes; }
  __device__ __forceinline__ void before_k(int) const {}
  __device__ __forceinline__ void after_k(int) const {}
  __device__ __forceinline__ void before_v(int) const {}
  __device__ __forceinline__ void after_v(int) const {}
};

// ------------------------------------------------------------------ warp-level MMA split reduction
// The two products of a split run on the tensor cores as warp-level MMAs
// (mma.sync m16n8k16, bf16 operands, fp32 accumulation), reading K and V
// straight from the swizzled pages with ldmatrix:
//   scores  S^T[pos][head] = K[pos][:] . q[head][:]          (A = K: 16 positions x 16 dims; B = q^T, heads padded to 8)
//   values  O^T[dim][head] = sum_pos V[pos][dim] P[head][pos] (A = V^T, read by ldmatrix.trans; B = P^T)
// Operands the MMA cannot take exactly in one bf16 value are split into bf16
// terms whose sum is the value, and one MMA is issued per term on the same A
// fragment, in term order (every bf16 x bf16 product is exact in fp32):
//   * fp32 queries (fp32-activation layers): three terms hi, mid, lo (exact,
//     as in the fp32-activation GEMM); bf16 queries: one;
//   * the softmax weights p = exp2(z - m): two terms p_hi = bf16(p),
//     p_lo = bf16(p - p_hi); the weight used is p_hi + p_lo (exact in fp32,
//     within 2^-16 of p) and l sums those, so o / l is a weighted mean of V with
//     exactly the weights the MMAs used.
// Every sum has one fixed order (per k step the terms in order, k steps
// ascending, then the four warps' partial sums 0+1+2+3), whoever calls it:
// decode and prefill give the same bits.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// d = a * b + d (m16n8k16, bf16 in, fp32 accumulate)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Outputs per thread of the split function: thread t of the group holds the
// weighted sums k = t + 128 j (head k / HD, dim k % HD).
__host__ __device__ constexpr int outputs_per_thread(int HD, int G) { return (G * HD + kGroupThreads - 1) / kGroupThreads; }

// B operand of the score MMAs: q^T, 16 dims x 8 columns (query heads g*G.., zero
// past G), per k step of 16 dims, per term.
template <int HD, int PL>
struct QFrags {
  uint32_t b[PL][HD / 16][2];
};

// The G query rows [G][HD] of the item (bf16, in shared or global memory).
template <int HD, int G>
__device__ __forceinline__ void load_qfrags(const __nv_bfloat16* qrow, QFrags<HD, 1>& qf) {
  const int lane = threadIdx.x & 31;
  const int n = lane >> 2;         // column = query head
  const int k0 = (lane & 3) * 2;   // first of the two k values this lane holds
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
    qf.b[0][ks][0] = n < G ? *reinterpret_cast<const uint32_t*>(qrow + n * HD + 16 * ks + k0) : 0u;
    qf.b[0][ks][1] = n < G ? *reinterpret_cast<const uint32_t*>(qrow + n * HD + 16 * ks + 8 + k0) : 0u;
  }
}
// The same from fp32 query rows (global memory), each value split into three bf16 terms.
template <int HD, int G>
__device__ __forceinline__ void load_qfrags(const float* qrow, QFrags<HD, 3>& qf) {
  const int lane = threadIdx.x & 31;
  const int n = lane >> 2;
  const int k0 = (lane & 3) * 2;
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float2 v = make_float2(0.f, 0.f);
      if (n < G) v = *reinterpret_cast<const float2*>(qrow + n * HD + 16 * ks + 8 * half + k0);
      float h0, m0, l0, h1, m1, l1;
      split3(v.x, h0, m0, l0);
      split3(v.y, h1, m1, l1);
      qf.b[0][ks][half] = pack_bf16x2(h0, h1);
      qf.b[1][ks][half] = pack_bf16x2(m0, m1);
      qf.b[2][ks][half] = pack_bf16x2(l0, l1);
    }
}

template <int HD, int G, int PL, class KV>
__device__ __forceinline__ void split_reduce(const QFrags<HD, PL>& qf, const KV& kv, int valid, float scale_log2,
                                             SplitSmem<HD, G>& sm, int group, float (&out)[outputs_per_thread(HD, G)]) {
  const int tid = threadIdx.x % kGroupThreads;
  const int w = tid >> 5;
  const int lane = tid & 31;
  const int g8 = lane >> 2;        // fragment row group
  const int c4 = lane & 3;         // fragment column pair
  const int mi = lane >> 3;        // ldmatrix: the matrix this lane addresses
  const int mr = lane & 7;         //           and its row
  const int base = 64 * w;         // this warp's positions [base, base + 64) = quarter w
  const int nvalid = min(64, valid - base);  // positions of this warp that take part (warp-uniform)

  // ---- scores: one m16 tile of 16 positions per page of the quarter
  kv.before_k(w);
  {
    const uint32_t kq = static_cast<uint32_t>(__cvta_generic_to_shared(kv.kq(w)));
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      if (16 * mt >= nvalid) break;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      // matrices: (pos 0-7, dims 0-7), (pos 8-15, dims 0-7), (pos 0-7, dims 8-15), (pos 8-15, dims 8-15)
      const int qpos = 16 * mt + (mi & 1) * 8 + mr;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kq + PageLayout<HD>::chunk(qpos, 2 * ks + (mi >> 1)), a0, a1, a2, a3);
#pragma unroll
        for (int pl = 0; pl < PL; ++pl) mma_bf16(d, a0, a1, a2, a3, qf.b[pl][ks][0], qf.b[pl][ks][1]);
      }
      // d: (pos g8, head 2c4), (pos g8, head 2c4+1), (pos g8+8, head 2c4), (pos g8+8, head 2c4+1)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hh = 2 * c4 + (e & 1);
        const int pp = base + 16 * mt + g8 + (e >> 1) * 8;
        if (hh < G) sm.z[hh][pp] = (pp < valid) ? __fmul_rn(d[e], scale_log2) : -INFINITY;
      }
    }
    // positions of this warp past the split's valid ones
    for (int pp = base + max(nvalid, 0) + lane; pp < base + 64; pp += 32)
#pragma unroll
      for (int hh = 0; hh < G; ++hh) sm.z[hh][pp] = -INFINITY;
  }
  kv.after_k(w);
  group_sync(group);

  // ---- per-head max (exact, order-free), the weights as two bf16 terms, and their sum (fixed order)
  for (int hh = w; hh < G; hh += 4) {
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) mx = fmaxf(mx, sm.z[hh][lane + 32 * j]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int pp = lane + 32 * j;
      const float e = (pp < valid) ? exp2f(__fsub_rn(sm.z[hh][pp], mx)) : 0.f;
      const float hi = __bfloat162float(__float2bfloat16_rn(e));
      const float lo = __bfloat162float(__float2bfloat16_rn(__fsub_rn(e, hi)));
      sm.e[pp][hh] = pack_bf16x2(hi, lo);
      s = __fadd_rn(s, __fadd_rn(hi, lo));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    if (lane == 0) {
      sm.m[hh] = mx;
      sm.l[hh] = s;
    }
  }
  group_sync(group);

  // ---- weighted sum of values: O^T (HD dims x 8 columns) over this warp's positions
  float acc[HD / 16][4];
#pragma unroll
  for (int mt = 0; mt < HD / 16; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
  kv.before_v(w);
  {
    const uint32_t vq = static_cast<uint32_t>(__cvta_generic_to_shared(kv.vq(w)));
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {  // 16 positions per step: page ks of the quarter
      if (16 * ks >= nvalid) break;
      // B = P^T, hi and lo terms: (pos 2c4, 2c4+1 | +8) x column g8 (a query head, zero past G)
      uint32_t bh0 = 0u, bh1 = 0u, bl0 = 0u, bl1 = 0u;
      if (g8 < G) {
        const int p0 = base + 16 * ks + 2 * c4;
        const uint32_t e0 = sm.e[p0][g8], e1 = sm.e[p0 + 1][g8], e8 = sm.e[p0 + 8][g8], e9 = sm.e[p0 + 9][g8];
        bh0 = (e0 & 0xffffu) | (e1 << 16);
        bl0 = (e0 >> 16) | (e1 & 0xffff0000u);
        bh1 = (e8 & 0xffffu) | (e9 << 16);
        bl1 = (e8 >> 16) | (e9 & 0xffff0000u);
      }
      const bool partial = 16 * ks + 16 > nvalid;
      // the A fragment's positions: 2c4, 2c4+1 (a0, a1) and 8+2c4, 8+2c4+1 (a2, a3)
      const int lim = nvalid - 16 * ks;
#pragma unroll
      for (int mt = 0; mt < HD / 16; ++mt) {
        // A = V^T: matrices (dims 0-7, pos 0-7), (dims 8-15, pos 0-7), (dims 0-7, pos 8-15), (dims 8-15, pos 8-15),
        // each read as 8 rows of positions and transposed
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vq + PageLayout<HD>::chunk(16 * ks + (mi >> 1) * 8 + mr, 2 * mt + (mi & 1)), a0, a1, a2, a3);
        if (partial) {
          // positions past the valid ones hold stale or never-written data: take no part (0 x NaN would)
          const uint32_t m0 = ((2 * c4 < lim) ? 0x0000ffffu : 0u) | ((2 * c4 + 1 < lim) ? 0xffff0000u : 0u);
          const uint32_t m1 = ((8 + 2 * c4 < lim) ? 0x0000ffffu : 0u) | ((8 + 2 * c4 + 1 < lim) ? 0xffff0000u : 0u);
          a0 &= m0;
          a1 &= m0;
          a2 &= m1;
          a3 &= m1;
        }
        mma_bf16(acc[mt], a0, a1, a2, a3, bh0, bh1);
        mma_bf16(acc[mt], a0, a1, a2, a3, bl0, bl1);
      }
    }
  }
  kv.after_v(w);
  group_sync(group);  // every warp is done with e before o overwrites it
  // acc[mt]: (dim 16mt + g8, head 2c4), (.., head 2c4+1), (dim 16mt + g8 + 8, head 2c4), (.., 2c4+1)
#pragma unroll
  for (int mt = 0; mt < HD / 16; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int hh = 2 * c4 + (e & 1);
      if (hh < G) sm.o[w][hh][16 * mt + g8 + (e >> 1) * 8] = acc[mt][e];
    }
  group_sync(group);
#pragma unroll
  for (int j = 0; j < outputs_per_thread(HD, G); ++j) {
    const int k = tid + kGroupThreads * j;
    if (k < G * HD) {
      const int hh = k / HD, d = k % HD;
      out[j] = __fadd_rn(__fadd_rn(__fadd_rn(sm.o[0][hh][d], sm.o[1][hh][d]), sm.o[2][hh][d]), sm.o[3][hh][d]);
    }
  }
}

// Combination of two split states (a covers lower positions than b).  An empty
// state (m = -inf) is an exact identity on either side.
__device__ __forceinline__ void merge_state(float& m, float& l, float& o, float mb, float lb, float ob) {
  if (mb == -INFINITY) return;
  if (m == -INFINITY) {
    m = mb;
    l = lb;
    o = ob;
    return;
  }
  const float mx = fmaxf(m, mb);
  const float ea = exp2f(__fsub_rn(m, mx));
  const float eb = exp2f(__fsub_rn(mb, mx));
  l = __fadd_rn(__fmul_rn(ea, l), __fmul_rn(eb, lb));
  o = __fadd_rn(__fmul_rn(ea, o), __fmul_rn(eb, ob));
  m = mx;
}

// merge_state applied to four outputs that share (m, l): each component gets
// exactly the operations merge_state would give it.
__device__ __forceinline__ void merge_state4(float& m, float& l, float4& o, float mb, float lb, const float4& ob) {
  if (mb == -INFINITY) return;
  if (m == -INFINITY) {
    m = mb;
    l = lb;
    o = ob;
    return;
  }
  const float mx = fmaxf(m, mb);
  const float ea = exp2f(__fsub_rn(m, mx));
  const float eb = exp2f(__fsub_rn(mb, mx));
  l = __fadd_rn(__fmul_rn(ea, l), __fmul_rn(eb, lb));
  o.x = __fadd_rn(__fmul_rn(ea, o.x), __fmul_rn(eb, ob.x));
  o.y = __fadd_rn(__fmul_rn(ea, o.y), __fmul_rn(eb, ob.y));
  o.z = __fadd_rn(__fmul_rn(ea, o.z), __fmul_rn(eb, ob.z));
  o.w = __fadd_rn(__fmul_rn(ea, o.w), __fmul_rn(eb, ob.w));
  m = mx;
}

struct Partials {
  float* m;  // [units][Hq]
  float* l;  // [units][Hq]
  float* o;  // [units][Hq][HD]
};

// Merge of the split states of one row (a decode request or a prefill token)
// for all heads of one kv group: thread (hh, d0) owns dims d0..d0+3.  INVARIANT rows combine the
// states in a pairwise tree over the split index (binary-counter form: the same
// tree as the level-by-level tree over 2^BI_MERGE_DEPTH leaves padded with
// empty states, since an empty state is an exact identity); FAST rows combine
// left to right.  States are fetched 16 at a time (their loads in flight
// together); an INVARIANT chunk of 16 consecutive splits is one complete
// level-4 subtree, reduced level by level in registers, and the chunk results
// go through the binary counter.
// Partial states are read through L2 (__ldcg): in the decode kernel they were
// written by other CTAs of the same launch.
constexpr int kMergeChunk = 16;  // split states fetched together; a chunk is one level-4 subtree

__device__ __forceinline__ void merge_row(const Partials& part, size_t first_unit, int n, bool tree, int hq, int hd,
                                          int h, int d0, float& out_m, float& out_l, float4& out_o) {
  float m = -INFINITY, l = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  // stack of complete subtrees over chunk results (level 4 and up of the padded tree)
  float sm_[BI_MERGE_DEPTH - 3], sl_[BI_MERGE_DEPTH - 3];
  float4 so_[BI_MERGE_DEPTH - 3];
  unsigned occ = 0;
  for (int c0 = 0; c0 < n; c0 += kMergeChunk) {
    // the chunk's states, loaded together (empty past n)
    float cm[kMergeChunk], cl[kMergeChunk];
    float4 co[kMergeChunk];
#pragma unroll
    for (int j = 0; j < kMergeChunk; ++j) {
      if (c0 + j < n) {
        const size_t pi = (first_unit + c0 + j) * hq + h;
        cm[j] = __ldcg(part.m + pi);
        cl[j] = __ldcg(part.l + pi);
        co[j] = __ldcg(reinterpret_cast<const float4*>(part.o + pi * hd + d0));
      } else {
        cm[j] = -INFINITY;
        cl[j] = 0.f;
        co[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (!tree) {
      // FAST: left to right
#pragma unroll
      for (int j = 0; j < kMergeChunk; ++j) merge_state4(m, l, o, cm[j], cl[j], co[j]);
      continue;
    }
    // pairwise tree inside the chunk, level by level: (0,1), (2,3), ... then pairs of those
#pragma unroll
    for (int w = 1; w < kMergeChunk; w *= 2)
#pragma unroll
      for (int i = 0; i < kMergeChunk; i += 2 * w) merge_state4(cm[i], cl[i], co[i], cm[i + w], cl[i + w], co[i + w]);
    // push the chunk's subtree; equal-sized subtrees merge pairwise (binary counter)
    float xm = cm[0], xl = cl[0];
    float4 xo = co[0];
    int lvl = 0;
    while (occ & (1u << lvl)) {
      float am = sm_[lvl], al = sl_[lvl];
      float4 ao = so_[lvl];
      merge_state4(am, al, ao, xm, xl, xo);  // stack entry covers the lower indices
      xm = am; xl = al; xo = ao;
      occ &= ~(1u << lvl);
      ++lvl;
    }
    sm_[lvl] = xm; sl_[lvl] = xl; so_[lvl] = xo;
    occ |= (1u << lvl);
  }
  if (tree) {
    // fold what is left, smallest (rightmost) subtree first: merge(stack[lvl], acc)
    for (int lvl = 0; lvl <= BI_MERGE_DEPTH - 4; ++lvl) {
      if (occ & (1u << lvl)) {
        float am = sm_[lvl], al = sl_[lvl];
        float4 ao = so_[lvl];
        merge_state4(am, al, ao, m, l, o);
        m = am; l = al; o = ao;
      }
    }
  }
  out_m = m;
  out_l = l;
  out_o = o;
}

// out[d0..d0+3] of one (row, head) at element offset off: o / l (0 where
// l == 0), rounded to bf16, kept in fp32, or split into three bf16 planes.
__device__ __forceinline__ void store_out4(const ActDst& out, size_t off, float l, const float4& o) {
  const float r0 = (l > 0.f) ? __fdiv_rn(o.x, l) : 0.f;
  const float r1 = (l > 0.f) ? __fdiv_rn(o.y, l) : 0.f;
  const float r2 = (l > 0.f) ? __fdiv_rn(o.z, l) : 0.f;
  const float r3 = (l > 0.f) ? __fdiv_rn(o.w, l) : 0.f;
  act_store4(out, off, r0, r1, r2, r3);
}

// ------------------------------------------------------------------ decode
// Plan per request b: geometry (invariant or fast), unit length, unit count,
// exclusive prefix of unit counts.  One CTA; B may be large.
struct DecodePlan {
  int* len;      // [B] KV length, clamped to [0, max_pages*16] (an out-of-range length is reported)
  int* mode;     // [B]
  int* ulen;     // [B] positions per unit
  int* nunits;   // [B]
  int* prefix;   // [B+1]
  int* counter;  // [1] next unclaimed work item of the split kernel (0 between launches)
  int* unit_row; // [units] request row of each unit (one load instead of a search over prefix)
};

// Error-word site codes of this file: 11-15 a bounded wait ran out; 16 a KV
// length outside [0, max_pages*16] (clamped); 17 a block-table entry outside
// [0, num_pages) or a position past the block-table row (page 0 read instead).
constexpr unsigned kSiteBadLength = 16;
constexpr unsigned kSiteBadPage = 17;
constexpr unsigned kSiteSmemAlign = 18;  // the decode kernel's shared memory is not 1024-byte aligned (output not written)

// Page of position-block `pi` of a request's block-table row, checked: an entry
// past the row or outside the cache is reported and replaced by page 0, so no
// access leaves the caller's buffers.
__device__ __forceinline__ int checked_page(const int* __restrict__ brow, int pi, int max_pages, int num_pages) {
  const int pg = (pi >= 0 && pi < max_pages) ? brow[pi] : -1;
  if (pg < 0 || pg >= num_pages) {
    atomicCAS(&g_attn_err_word, 0u, kSiteBadPage);
    return 0;
  }
  return pg;
}

__global__ void __launch_bounds__(1024) decode_plan_kernel(const int* __restrict__ kv_lens, int B, int hkv, int mode,
                                                           int target, int fast_units_wanted, int max_tokens,
                                                           DecodePlan plan) {
  pdl_wait();
  pdl_trigger();
  __shared__ int part[1024];
  const int t = threadIdx.x;
  if (t == 0) *plan.counter = 0;
  const int per = (B + 1023) / 1024;
  const int b0 = min(B, t * per), b1 = min(B, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) {
    int L = kv_lens[b];
    if (L < 0 || L > max_tokens) {
      atomicCAS(&g_attn_err_word, 0u, kSiteBadLength);
      L = L < 0 ? 0 : max_tokens;
    }
    plan.len[b] = L;
    const bool inv = (mode == BI_MODE_INVARIANT) || (mode == BI_MODE_PROTECTED && b == target);
    int ul, n;
    if (inv) {
      ul = kSplit;
      n = (L + kSplit - 1) / kSplit;
    } else if (fast_units_wanted <= 0) {
      ul = kSplit;  // tuned FAST: the invariant splits, combined left to right
      n = (L + kSplit - 1) / kSplit;
    } else {
      const int pages = (L + kPage - 1) / kPage;
      int want = min(max(1, fast_units_wanted), min(kMaxFastUnits, max(1, pages)));
      ul = kPage * ((pages + want - 1) / want);
      n = (L + ul - 1) / ul;
    }
    if (L <= 0) n = 0;
    plan.mode[b] = inv ? kPlanInvariant : kPlanFast;
    plan.ulen[b] = ul;
    plan.nunits[b] = n;
    local += n;
  }
  part[t] = local;
  __syncthreads();
  // inclusive Hillis-Steele scan over the 1024 thread totals (integers: order-free)
  for (int off = 1; off < 1024; off <<= 1) {
    const int v = (t >= off) ? part[t - off] : 0;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  int run = part[t] - local;
  for (int b = b0; b < b1; ++b) {
    plan.prefix[b] = run;
    for (int u = 0; u < plan.nunits[b]; ++u) plan.unit_row[run + u] = b;
    run += plan.nunits[b];
  }
  if (t == 1023) plan.prefix[B] = part[1023];
}

__device__ __forceinline__ int find_row(const int* prefix, int n, int u) {
  // largest b with prefix[b] <= u (prefix is non-decreasing, prefix[n] > u)
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Decode split kernel: a persistent CTA of one 128-thread consumer group plus a
// producer warp.  The producer streams every split's K and V (in quarters of
// 64 positions = 4 pages of one kv head, one bulk copy per page) into a ring of
// shared-memory stages; the consumers run split_reduce on each split as soon as
// its quarters land.  A unit (one request, one kv head, one planned range) is
// one 256-position split under the invariant plan, or several consecutive
// 256-position blocks combined left to right under the FAST plan.
// Ring-size rule: the four consumer warps may wait on the four key quarters of
// a split at once, so a stage's previous use must belong to an earlier phase
// (stages >= 4); with fewer, a wait on the next use of a stage can be satisfied
// by the completed parity of the use before it, and the ring's accounting
// breaks.  (A 3-stage build did exactly that.)
constexpr int kDecodeStages = 4;
static_assert(kDecodeStages >= 4, "the four quarters of a phase may be waited on together");
constexpr int kDecodeThreads = kGroupThreads + 32;

// Work items reach the consumers through a 2-slot ring filled by the producer
// one item ahead: the item's descriptor and its G query rows (one bulk copy),
// so the consumer warps never wait on global loads for their indexing or q.
constexpr int kItemSlots = 2;

template <int HD, int G>
struct DecodeSmem {
  // TMA tensor copies land here with the 128-byte swizzle, which wants 1024-byte aligned pages: the ring is the
  // first member and the dynamic shared memory window starts 1024-byte aligned (checked at kernel entry).  No
  // alignment attribute on the struct: padding it to 1024 bytes would cost the third CTA per SM.
  __align__(128) unsigned char ring[kDecodeStages][PageLayout<HD>::kQuarterBytes];
  SplitSmem<HD, G> sm;
  __align__(16) __nv_bfloat16 qbuf[kItemSlots][G * HD];
  int4 item[kItemSlots];  // {unit u, kv head g, first position, end position}
  unsigned long long full[kDecodeStages];
  unsigned long long empty[kDecodeStages];
  unsigned long long item_full[kItemSlots];
  unsigned long long item_empty[kItemSlots];
  int abort_flag;
};

// One TMA tensor copy of a page of one kv head: box {64 dims, 16 positions, HD/64
// halves} of the cache viewed as [pages * kv heads][16][HD/64][64], landing as
// [half][position][64 dims] with the 128-byte swizzle.
// A page of keys or values is read once per pass, so its copies carry an L2
// evict-first hint: the cache stream does not push out of L2 what is reused
// soon after (the split states that the merge kernel reads back, the
// activations between the layer's kernels).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_page(uint32_t dst, const CUtensorMap* map, uint32_t bar, int page_head) {
  const uint64_t pol = l2_evict_first_policy();
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(0), "r"(0), "r"(page_head), "l"(pol)
      : "memory");
}

template <int HD, int G, int PL>
__global__ void __launch_bounds__(kDecodeThreads, 3) decode_split_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const __nv_bfloat16* __restrict__ q, const float* __restrict__ qf, const int* __restrict__ block_table, int B,
    int hq, int hkv, int max_pages, int num_pages, float scale_log2, DecodePlan plan, Partials part,
    int plan_ready) {
  // PL = 1: bf16 queries, staged with the item; PL = 3: fp32 queries qf
  // (fp32-activation layers; q unused), which the consumers read from global
  // memory (the item ring then carries the descriptor only).
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    // the swizzled TMA copies need 1024-byte aligned pages; report instead of copying misaligned
    if (threadIdx.x == 0) atomicCAS(&g_attn_err_word, 0u, kSiteSmemAlign);
    return;
  }
  DecodeSmem<HD, G>& S = *reinterpret_cast<DecodeSmem<HD, G>*>(smem_raw);
  const uint32_t full0 = smem_u32(&S.full[0]);
  const uint32_t empty0 = smem_u32(&S.empty[0]);
  const uint32_t ifull0 = smem_u32(&S.item_full[0]);
  const uint32_t iempty0 = smem_u32(&S.item_empty[0]);
  volatile int* abort_flag = &S.abort_flag;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDecodeStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(ifull0 + 8 * i, 1);                 // producer's arrive + the q bytes
      mbar_init(iempty0 + 8 * i, kGroupThreads / 32);  // one arrive per consumer warp
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // plan_ready: the plan was built by a kernel that finished before the
  // previous one started (the layers after the first of a decode step).  The
  // producer then issues the key quarters of its first item before waiting for
  // the previous kernel, as far as they hold no page of the request's newest
  // position (the one that kernel stores); `pre` counts them.
  int pre = 0;
  uint32_t pre_issued = 0;
  if (plan_ready && threadIdx.x >= kGroupThreads) {
    const int lane = threadIdx.x - kGroupThreads;
    const int it = static_cast<int>(blockIdx.x);
    if (it < plan.prefix[B] * hkv) {
      const int u = it / hkv, g = it % hkv;
      const int b = plan.unit_row[u];
      const int L = plan.len[b], ul = plan.ulen[b];
      const int bs = (u - plan.prefix[b]) * ul;  // the first block of the item
      const int valid = min(kSplit, min(L, bs + ul) - bs);
      const int newest_page_start = ((L - 1) / kPage) * kPage;
      while (pre < 4 && 64 * pre < valid && bs + 64 * pre + 64 <= newest_page_start) ++pre;
      const int* brow = block_table + static_cast<size_t>(b) * max_pages;
      const int npages = (min(valid, 64 * pre) + kPage - 1) / kPage;
      const int pg = lane < npages ? checked_page(brow, bs / kPage + lane, max_pages, num_pages) : 0;
      for (int j = 0; j < pre; ++j) {
        const int nv = min(64, valid - 64 * j);
        const int npg = (nv + kPage - 1) / kPage;
        const uint32_t fb = full0 + 8 * j;  // fresh stages: nothing to wait for
        const int page = __shfl_sync(0xffffffffu, pg, (j * 4 + lane) & 31);
        if (lane == 0) mbar_expect_tx(fb, static_cast<uint32_t>(npg * kPage * HD * 2));
        __syncwarp();
        if (lane < npg) tma_page(smem_u32(&S.ring[j][lane * PageLayout<HD>::kPageBytes]), &kmap, fb, page * hkv + g);
        pre_issued |= 1u << j;
      }
    }
  }
  pdl_wait();
  pdl_trigger();
  const int total = plan.prefix[B] * hkv;

  if (threadIdx.x >= kGroupThreads) {
    // ---------------------------------------------------------------- producer warp
    // Lane 0 claims each stage (waits for it to be free, arms its barrier with
    // the byte count); lanes 0..3 then issue one page copy each, so the copies
    // of a stage are in flight together.
    const int plane = threadIdx.x - kGroupThreads;
    int n = 0;
    uint32_t issued = pre_issued, ipar = 0;  // quarters issued before the wait: stages 0.., phase 0
    int skip = pre;
    // Work items: each CTA's first is its own index, the rest are claimed from
    // a counter shared by the launch's CTAs (the next one as soon as the current
    // one's copies are all issued), so a CTA that finishes early takes more;
    // which CTA reduces an item changes nothing in its arithmetic.
    auto claim = [&]() -> int {
      int it = 0;
      if (plane == 0) it = static_cast<int>(gridDim.x) + atomicAdd(plan.counter, 1);
      return __shfl_sync(0xffffffffu, it, 0);
    };
    // item k's descriptor and q go to slot k % 2; an item is announced while
    // the item before it is still being streamed; a claim past the last item
    // is announced as an end marker (u = -1).  Returns the item's request row
    // (every lane), which the loop below reuses.
    int ann = 0;
    uint32_t ann_issued = 0;
    auto announce = [&](int it) -> int {
      const int u = it < total ? it / hkv : 0;
      const int g = it % hkv;
      const int b = it < total ? plan.unit_row[u] : 0;
      if (plane == 0) {
        const int slot = ann % kItemSlots;
        const uint32_t ph = static_cast<uint32_t>((ann / kItemSlots) & 1);
        wait_bounded(iempty0 + 8 * slot, ph ^ 1u, abort_flag, 14);
        if (it >= total) {
          S.item[slot] = make_int4(-1, 0, 0, 0);
          mbar_arrive(ifull0 + 8 * slot);  // release: the descriptor store
          ann_issued &= ~(1u << slot);
        } else {
          const int ul = plan.ulen[b];
          const int us = (u - plan.prefix[b]) * ul;
          S.item[slot] = make_int4(u, g, us, min(plan.len[b], us + ul));
          if (qf != nullptr) {
            mbar_arrive(ifull0 + 8 * slot);  // release: the descriptor store
          } else {
            mbar_expect_tx(ifull0 + 8 * slot, static_cast<uint32_t>(G * HD * 2));  // release: the descriptor store
            bulk_g2s(smem_u32(&S.qbuf[slot][0]), q + (static_cast<size_t>(b) * hq + g * G) * HD, G * HD * 2,
                     ifull0 + 8 * slot);
            ann_issued |= 1u << slot;
          }
        }
      }
      ++ann;
      return b;
    };
    int item = static_cast<int>(blockIdx.x);
    int b = announce(item);
    while (item < total) {
      const int u = item / hkv;
      const int g = item % hkv;
      const int s = u - plan.prefix[b];
      const int L = plan.len[b];
      const int ul = plan.ulen[b];
      const int ustart = s * ul;
      const int uend = min(L, ustart + ul);
      const int* brow = block_table + static_cast<size_t>(b) * max_pages;
      for (int bs = ustart; bs < uend; bs += kSplit) {
        const int valid = min(kSplit, uend - bs);
        // the block's (up to 16) page indices, one per lane, fetched together
        // before its copies rather than one dependent load per quarter
        const int npages = (valid + kPage - 1) / kPage;
        const int pg = plane < npages ? checked_page(brow, bs / kPage + plane, max_pages, num_pages) : 0;
        for (int j = 0; j < 8; ++j, ++n) {
          if (skip > 0) {  // issued before the wait
            --skip;
            continue;
          }
          const int st = n % kDecodeStages;
          const uint32_t ph = static_cast<uint32_t>((n / kDecodeStages) & 1);
          const int q0 = (j & 3) * 64;
          const int nv = max(0, min(64, valid - q0));
          const int npg = (nv + kPage - 1) / kPage;
          const uint32_t fb = full0 + 8 * st;
          const int page = __shfl_sync(0xffffffffu, pg, ((j & 3) * 4 + plane) & 31);
          if (plane == 0) {
            wait_bounded(empty0 + 8 * st, ph ^ 1u, abort_flag, 13);
            mbar_expect_tx(fb, static_cast<uint32_t>(npg * kPage * HD * 2));
          }
          __syncwarp();
          if (plane < npg)
            tma_page(smem_u32(&S.ring[st][plane * PageLayout<HD>::kPageBytes]), (j < 4) ? &kmap : &vmap, fb,
                     page * hkv + g);
          issued |= 1u << st;
          ipar = (ipar & ~(1u << st)) | (ph << st);
        }
      }
      // the next item is claimed once this one's copies are all issued, not
      // before: a CTA then holds at most one item that no copy has started
      // for, which keeps the launch's last items from queueing behind busy CTAs
      item = claim();
      b = announce(item);
    }
    // keep the CTA resident until every copy it issued has landed
    if (plane == 0) {
      for (int i = 0; i < kDecodeStages; ++i)
        if (issued & (1u << i)) wait_drain(full0 + 8 * i, (ipar >> i) & 1u);
      // the q copies of the last announced items
      for (int k = max(0, ann - kItemSlots); k < ann; ++k)
        if (ann_issued & (1u << (k % kItemSlots)))
          wait_drain(ifull0 + 8 * (k % kItemSlots), static_cast<uint32_t>((k / kItemSlots) & 1));
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  constexpr int OPT = outputs_per_thread(HD, G);
  const int tid = threadIdx.x;
  int n0 = 0;
  // items in the order the producer announces them, up to its end marker (a
  // CTA never gets more than `total`; a wait that gave up ends the loop too)
  for (int icount = 0; icount <= total; ++icount) {
    const int islot = icount % kItemSlots;
    const bool ok = wait_bounded(ifull0 + 8 * islot, static_cast<uint32_t>((icount / kItemSlots) & 1), abort_flag, 15);
    const int4 desc = S.item[islot];
    // one decision for the whole group (its warps meet at named barriers below)
    if (group_any(0, !ok || desc.x < 0)) break;
    const int u = desc.x;
    const int g = desc.y;
    const int ustart = desc.z;
    const int uend = desc.w;
    QFrags<HD, PL> qfr;
    if constexpr (PL == 1) {
      load_qfrags<HD, G>(&S.qbuf[islot][0], qfr);
    } else {
      const int b = plan.unit_row[u];
      load_qfrags<HD, G>(qf + (static_cast<size_t>(b) * hq + g * G) * HD, qfr);
    }
    __syncwarp();
    if ((tid & 31) == 0) mbar_arrive(iempty0 + 8 * islot);  // descriptor and q are in registers
    float rm[G], rl[G], ro[OPT];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      rm[hh] = -INFINITY;
      rl[hh] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < OPT; ++j) ro[j] = 0.f;
    bool first = true;
    for (int bs = ustart; bs < uend; bs += kSplit, n0 += 8) {
      const int valid = min(kSplit, uend - bs);
      RingKV<HD> kv{&S.ring[0][0], full0, empty0, n0, kDecodeStages, abort_flag};
      float bo[OPT];
      split_reduce<HD, G, PL>(qfr, kv, valid, scale_log2, S.sm, 0, bo);
#pragma unroll
      for (int j = 0; j < OPT; ++j) {
        const int k = tid + kGroupThreads * j;
        if (k < G * HD) {
          const int hh = k / HD;
          if (first) {
            ro[j] = bo[j];
          } else {
            float mm = rm[hh], ll = rl[hh];
            merge_state(mm, ll, ro[j], S.sm.m[hh], S.sm.l[hh], bo[j]);
          }
        }
      }
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        if (first) {
          rm[hh] = S.sm.m[hh];
          rl[hh] = S.sm.l[hh];
        } else {
          float oo = 0.f;
          merge_state(rm[hh], rl[hh], oo, S.sm.m[hh], S.sm.l[hh], 0.f);
        }
      }
      first = false;
      group_sync(0);  // the group scratch is reused by the next split
    }
    const size_t pidx = static_cast<size_t>(u) * hq + g * G;
#pragma unroll
    for (int j = 0; j < OPT; ++j) {
      const int k = tid + kGroupThreads * j;
      if (k < G * HD) part.o[(pidx + k / HD) * HD + (k % HD)] = ro[j];
    }
    if (tid < G) {
      part.m[pidx + tid] = rm[tid];
      part.l[pidx + tid] = rl[tid];
    }
  }
}


// Merge of the split states of each (request, query head) in a second kernel.
__global__ void decode_merge_kernel(const Partials part, DecodePlan plan, ActDst out, int B, int hq, int hkv,
                                    int hd) {
  // The next kernel (the O projection) may launch at once: its CTAs then take
  // the SMs that the split kernel's last CTAs free and fetch their first weight
  // stages while this merge still waits; its own wait still covers this kernel.
  pdl_trigger();
  pdl_wait();
  // the split kernel has finished: its work counter starts from zero for the next launch
  if (blockIdx.x == 0 && threadIdx.x == 0) *plan.counter = 0;
  const int b = blockIdx.x / hkv;
  const int g = blockIdx.x % hkv;
  const int G = hq / hkv;
  const int q4 = hd / 4;  // threads per head: four dims each
  const int hh = threadIdx.x / q4;
  const int d0 = 4 * (threadIdx.x % q4);
  if (b >= B || hh >= G) return;
  const int h = g * G + hh;
  float m, l;
  float4 o;
  merge_row(part, plan.prefix[b], plan.nunits[b], plan.mode[b] == kPlanInvariant, hq, hd, h, d0, m, l, o);
  store_out4(out, (static_cast<size_t>(b) * hq + h) * hd + d0, l, o);
}

// ------------------------------------------------------------------ prefill
// Units are (q-block of up to 16 tokens of one request, split); the q-block's
// tokens that see the split reduce it one after another with the same split
// function as decode, reading the split's K/V from shared memory.
//
// INVARIANT splits of a token at position p: [256s, 256s+256) ∩ [0, p].
// FAST splits (the non-invariant scheme in which cached and new tokens are
// reduced separately): cached keys [0, pos0) cut at multiples of 256 from 0,
// then new keys [pos0, p] cut at pos0 + multiples of 256.
struct PrefillPlan {
  int* tok_prefix;   // [T+1] exclusive prefix of per-token split counts
  int* qb_req;       // [NQB]
  int* qb_tok0;      // [NQB]
  int* qb_ntok;      // [NQB]
  int* qb_prefix;    // [NQB+1] exclusive prefix of per-q-block unit counts
  int* counts;       // [2]: NQB, total units
  int* req_mode;     // [B]
};

__device__ __forceinline__ int n_splits_token(bool inv, int pos0, int p) {
  if (inv) return p / kSplit + 1;
  return (pos0 + kSplit - 1) / kSplit + (p - pos0) / kSplit + 1;
}

// split index s of a token of request (pos0) -> [start, end) of keys, clipped to p
__device__ __forceinline__ void split_range(bool inv, int pos0, int s, int p, int& start, int& end) {
  if (inv) {
    start = s * kSplit;
    end = min(p + 1, start + kSplit);
    return;
  }
  const int nc = (pos0 + kSplit - 1) / kSplit;
  if (s < nc) {
    start = s * kSplit;
    end = min(pos0, start + kSplit);
  } else {
    start = pos0 + (s - nc) * kSplit;
    end = min(p + 1, start + kSplit);
  }
}

__global__ void __launch_bounds__(1024) prefill_plan_kernel(const int* __restrict__ q_start,
                                                            const int* __restrict__ q_pos0, int B, int T, int mode,
                                                            int target, PrefillPlan plan) {
  pdl_wait();
  pdl_trigger();
  __shared__ int part[1024];

  const int t = threadIdx.x;
  // phase 1: per-token split counts -> tok_prefix (tokens in order)
  {
    const int per = (T + 1023) / 1024;
    const int t0 = min(T, t * per), t1 = min(T, t0 + per);
    int local = 0;
    int b = 0;
    for (int tok = t0; tok < t1; ++tok) {
      if (tok == t0) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (q_start[mid] <= tok) lo = mid; else hi = mid - 1;
        }
        b = lo;
      }
      while (q_start[b + 1] <= tok) ++b;
      const bool inv = (mode == BI_MODE_INVARIANT) || (mode == BI_MODE_PROTECTED && b == target);
      const int p = q_pos0[b] + (tok - q_start[b]);
      local += n_splits_token(inv, q_pos0[b], p);
    }
    part[t] = local;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      const int v = (t >= off) ? part[t - off] : 0;
      __syncthreads();
      part[t] += v;
      __syncthreads();
    }
    int run = part[t] - local;
    for (int tok = t0; tok < t1; ++tok) {
      int lo = 0, hi = B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (q_start[mid] <= tok) lo = mid; else hi = mid - 1;
      }
      const int bb = lo;
      const bool inv = (mode == BI_MODE_INVARIANT) || (mode == BI_MODE_PROTECTED && bb == target);
      const int p = q_pos0[bb] + (tok - q_start[bb]);
      plan.tok_prefix[tok] = run;
      run += n_splits_token(inv, q_pos0[bb], p);
    }
    if (t == 1023) plan.tok_prefix[T] = part[1023];
    __syncthreads();
  }
  // phase 2: q-blocks of each request (sequential over requests in thread 0,
  // then a parallel fill); counts per request are small integers.
  if (t == 0) {
    int nqb = 0, units = 0;
    for (int b = 0; b < B; ++b) {
      const bool inv = (mode == BI_MODE_INVARIANT) || (mode == BI_MODE_PROTECTED && b == target);
      plan.req_mode[b] = inv ? kPlanInvariant : kPlanFast;
      const int n = q_start[b + 1] - q_start[b];
      for (int j = 0; j < n; j += kPrefillQBlock) {
        const int cnt = min(kPrefillQBlock, n - j);
        const int plast = q_pos0[b] + j + cnt - 1;
        plan.qb_req[nqb] = b;
        plan.qb_tok0[nqb] = q_start[b] + j;
        plan.qb_ntok[nqb] = cnt;
        plan.qb_prefix[nqb] = units;
        units += n_splits_token(inv, q_pos0[b], plast);
        ++nqb;
      }
    }
    plan.qb_prefix[nqb] = units;
    plan.counts[0] = nqb;
    plan.counts[1] = units;

  }
}

template <int HD, int G>
struct PrefillSmem {
  __align__(16) unsigned char k[4 * PageLayout<HD>::kQuarterBytes];  // the split's keys, page layout of the ring
  __align__(16) unsigned char v[4 * PageLayout<HD>::kQuarterBytes];
  SplitSmem<HD, G> grp[kPrefillGroups];
};

template <int HD, int G, int PL>
__global__ void __launch_bounds__(kGroupThreads* kPrefillGroups) prefill_split_kernel(
    const __nv_bfloat16* __restrict__ q, const float* __restrict__ qf, const __nv_bfloat16* __restrict__ kc,
    const __nv_bfloat16* __restrict__ vc, const int* __restrict__ block_table, const int* __restrict__ q_pos0,
    const int* __restrict__ q_start, int hq, int hkv, int max_pages, int num_pages, float scale_log2,
    PrefillPlan plan, Partials part) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  PrefillSmem<HD, G>& sm = *reinterpret_cast<PrefillSmem<HD, G>*>(smem_raw);
  constexpr int OPT = outputs_per_thread(HD, G);
  const int group = threadIdx.x / kGroupThreads;
  const int tid = threadIdx.x % kGroupThreads;
  const int c = (tid & 31) & 7;
  const int nqb = plan.counts[0];
  const int total = plan.counts[1] * hkv;
  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    const int u = item / hkv;
    const int g = item % hkv;
    const int qb = find_row(plan.qb_prefix, nqb, u);
    const int s = u - plan.qb_prefix[qb];
    const int b = plan.qb_req[qb];
    const int tok0 = plan.qb_tok0[qb];
    const int ntok = plan.qb_ntok[qb];
    const int pos0 = q_pos0[b];
    const int p_first = pos0 + (tok0 - q_start[b]);
    const int p_last = p_first + ntok - 1;
    const bool inv = plan.req_mode[b] == kPlanInvariant;
    int st, en;
    split_range(inv, pos0, s, p_last, st, en);
    // stage keys/values [st, en) of kv head g
    const int rows = en - st;
    constexpr int CH = HD / 8;  // 16-byte chunks per row
    __syncthreads();
    for (int idx = threadIdx.x; idx < rows * CH; idx += blockDim.x) {
      const int r = idx / CH, ch = idx % CH;
      const int pos = st + r;
      const int pg = checked_page(block_table + static_cast<size_t>(b) * max_pages, pos / kPage, max_pages, num_pages);
      const size_t off = ((static_cast<size_t>(pg) * hkv + g) * kPage + (pos % kPage)) * HD + ch * 8;
      const int so = (r >> 6) * PageLayout<HD>::kQuarterBytes + PageLayout<HD>::chunk(r & 63, ch);
      *reinterpret_cast<uint4*>(&sm.k[so]) = *reinterpret_cast<const uint4*>(kc + off);
      *reinterpret_cast<uint4*>(&sm.v[so]) = *reinterpret_cast<const uint4*>(vc + off);
    }
    __syncthreads();
    SmemKV<HD> kv{&sm.k[0], &sm.v[0]};
    for (int qi = group; qi < ntok; qi += kPrefillGroups) {
      const int tok = tok0 + qi;
      const int p = p_first + qi;
      if (s >= n_splits_token(inv, pos0, p)) continue;  // this split lies after the token
      int st_t, en_t;
      split_range(inv, pos0, s, p, st_t, en_t);
      const int valid = en_t - st_t;  // >= 1; same origin st as the staged rows
      float bo[OPT];
      QFrags<HD, PL> qfr;
      if constexpr (PL == 1) load_qfrags<HD, G>(q + (static_cast<size_t>(tok) * hq + g * G) * HD, qfr);
      else load_qfrags<HD, G>(qf + (static_cast<size_t>(tok) * hq + g * G) * HD, qfr);
      split_reduce<HD, G, PL>(qfr, kv, valid, scale_log2, sm.grp[group], group, bo);
      const size_t pidx = (static_cast<size_t>(plan.tok_prefix[tok]) + s) * hq + g * G;
#pragma unroll
      for (int j = 0; j < OPT; ++j) {
        const int k = tid + kGroupThreads * j;
        if (k < G * HD) part.o[(pidx + k / HD) * HD + (k % HD)] = bo[j];
      }
      if (tid < G) {
        part.m[pidx + tid] = sm.grp[group].m[tid];
        part.l[pidx + tid] = sm.grp[group].l[tid];
      }
      group_sync(group);  // group scratch reused by the next token
    }
  }
}

__global__ void prefill_merge_kernel(const Partials part, PrefillPlan plan, const int* __restrict__ q_start,
                                     const int* __restrict__ q_pos0, int B, ActDst out, int hq, int hkv, int hd) {
  pdl_wait();
  pdl_trigger();
  const int tok = blockIdx.x / hkv;
  const int g = blockIdx.x % hkv;
  const int G = hq / hkv;
  const int q4 = hd / 4;  // threads per head: four dims each
  const int hh = threadIdx.x / q4;
  const int d0 = 4 * (threadIdx.x % q4);
  if (hh >= G) return;
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (q_start[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int h = g * G + hh;
  const int n = plan.tok_prefix[tok + 1] - plan.tok_prefix[tok];
  float m, l;
  float4 o;
  merge_row(part, plan.tok_prefix[tok], n, plan.req_mode[b] == kPlanInvariant, hq, hd, h, d0, m, l, o);
  store_out4(out, (static_cast<size_t>(tok) * hq + h) * hd + d0, l, o);
}

// ------------------------------------------------------------------ host side
bi_status check_dims(const bi_attn_dims* dm) {
  BI_REQUIRE(dm != nullptr, BI_ERR_INVALID_ARG, "attention: null dims");
  BI_REQUIRE(dm->head_dim == 64 || dm->head_dim == 128, BI_ERR_UNSUPPORTED, "attention: head_dim %d (64 or 128)",
             dm->head_dim);
  BI_REQUIRE(dm->num_kv_heads >= 1 && dm->num_q_heads >= dm->num_kv_heads &&
                 dm->num_q_heads % dm->num_kv_heads == 0,
             BI_ERR_INVALID_ARG, "attention: heads %d/%d", dm->num_q_heads, dm->num_kv_heads);
  const int G = dm->num_q_heads / dm->num_kv_heads;
  BI_REQUIRE(G == 1 || G == 2 || G == 4, BI_ERR_UNSUPPORTED, "attention: %d query heads per kv head (1, 2 or 4)", G);
  BI_REQUIRE(dm->page_size == kPage, BI_ERR_UNSUPPORTED, "attention: page_size %d (must be %d)", dm->page_size, kPage);
  BI_REQUIRE(dm->max_pages >= 1 && dm->num_pages >= 1, BI_ERR_INVALID_ARG, "attention: max_pages/num_pages");
  BI_REQUIRE(dm->scale > 0.f && dm->scale == dm->scale, BI_ERR_INVALID_ARG, "attention: scale must be > 0");
  const int64_t max_tokens = static_cast<int64_t>(dm->max_pages) * kPage;
  BI_REQUIRE((max_tokens + kSplit - 1) / kSplit <= (int64_t(1) << BI_MERGE_DEPTH), BI_ERR_UNSUPPORTED,
             "attention: max_pages*16 beyond the merge depth");
  return BI_OK;
}

int max_units_per_request(const bi_attn_dims* dm) {
  const int inv = (dm->max_pages * kPage + kSplit - 1) / kSplit;
  return std::max(inv, kMaxFastUnits);
}

struct DecodeWs {
  DecodePlan plan;
  Partials part;
  size_t bytes;
};

// Plan arrays of a decode batch (small; reusable by every layer of a step).
size_t carve_decode_plan(void* base, int B, int hkv, size_t units, DecodePlan* plan) {
  WsCarver cv(base, 0);
  plan->len = cv.take<int>(B);
  plan->mode = cv.take<int>(B);
  plan->ulen = cv.take<int>(B);
  plan->nunits = cv.take<int>(B);
  plan->prefix = cv.take<int>(B + 1);
  plan->counter = cv.take<int>(1);
  plan->unit_row = cv.take<int>(units);
  return align_up(cv.used, 256);
}

size_t carve_decode_parts(void* base, size_t units, const bi_attn_dims* dm, Partials* part) {
  WsCarver cv(base, 0);
  part->m = cv.take<float>(units * dm->num_q_heads);
  part->l = cv.take<float>(units * dm->num_q_heads);
  part->o = cv.take<float>(units * dm->num_q_heads * dm->head_dim);
  return align_up(cv.used, 256);
}

DecodeWs carve_decode(void* ws, size_t, int B, const bi_attn_dims* dm) {
  DecodeWs r;
  const size_t units = static_cast<size_t>(B) * max_units_per_request(dm);
  const size_t pb = carve_decode_plan(ws, B, dm->num_kv_heads, units, &r.plan);
  const size_t qb = carve_decode_parts(ws ? static_cast<char*>(ws) + pb : nullptr, units, dm, &r.part);
  r.bytes = pb + qb;
  return r;
}

struct PrefillWs {
  PrefillPlan plan;
  Partials part;
  size_t bytes;
};

int64_t max_prefill_qblocks(int B, int T) { return static_cast<int64_t>(B) + T / kPrefillQBlock + 1; }

PrefillWs carve_prefill(void* ws, size_t cap, int B, int T, const bi_attn_dims* dm) {
  WsCarver cv(ws, cap);
  PrefillWs r;
  const int64_t nqb = max_prefill_qblocks(B, T);
  r.plan.tok_prefix = cv.take<int>(T + 1);
  r.plan.qb_req = cv.take<int>(nqb);
  r.plan.qb_tok0 = cv.take<int>(nqb);
  r.plan.qb_ntok = cv.take<int>(nqb);
  r.plan.qb_prefix = cv.take<int>(nqb + 1);
  r.plan.counts = cv.take<int>(2);
  r.plan.req_mode = cv.take<int>(B);
  // per token at most ceil(max_tokens/256) + 1 splits (FAST adds one cut at pos0)
  const size_t per_tok = (static_cast<size_t>(dm->max_pages) * kPage + kSplit - 1) / kSplit + 1;
  const size_t units = static_cast<size_t>(T) * per_tok;
  r.part.m = cv.take<float>(units * dm->num_q_heads);
  r.part.l = cv.take<float>(units * dm->num_q_heads);
  r.part.o = cv.take<float>(units * dm->num_q_heads * dm->head_dim);
  r.bytes = cv.used;
  return r;
}

// Dynamic shared memory of the decode split kernel (three CTAs per SM at head_dim 128).
template <int HD, int G>
constexpr size_t decode_smem() { return sizeof(DecodeSmem<HD, G>); }

template <int HD, int G, int PL>
bi_status decode_grid(int* grid) {
  const size_t smem = decode_smem<HD, G>();
  const void* fn = reinterpret_cast<const void*>(decode_split_kernel<HD, G, PL>);
  BI_CUDA_TRY(ensure_smem_limit(fn, static_cast<int>(smem)));
  *grid = occupancy_per_sm(fn, kDecodeThreads, smem) * num_sms();
  return BI_OK;
}

// Tensor map of a paged K or V cache [pages][kv heads][16][HD] bf16 for the
// decode loader: viewed as [pages * kv heads][16 positions][HD/64 halves][64]
// (strides 16*HD*2, HD*2 and 128 bytes), box {64, 16, HD/64, 1} = one page of
// one kv head, 128-byte swizzle.  Cached per (pointer, shape, device).
PFN_cuTensorMapEncodeTiled_v12000 attn_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

std::mutex g_cache_map_mutex;
std::vector<std::pair<std::tuple<const void*, int, int, int, int>, CUtensorMap>> g_cache_maps;

bi_status cache_map(const void* cache, int num_pages, int hkv, int hd, CUtensorMap* out) {
  int dev = 0;
  BI_CUDA_TRY(cudaGetDevice(&dev));
  const auto key = std::make_tuple(cache, num_pages, hkv, hd, dev);
  {
    std::lock_guard<std::mutex> lock(g_cache_map_mutex);
    for (const auto& e : g_cache_maps)
      if (e.first == key) {
        *out = e.second;
        return BI_OK;
      }
  }
  auto fn = attn_encode_fn();
  BI_REQUIRE(fn != nullptr, BI_ERR_CUDA, "attention: cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[4] = {64, 16, static_cast<cuuint64_t>(hd / 64),
                        static_cast<cuuint64_t>(num_pages) * static_cast<cuuint64_t>(hkv)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(hd) * 2, 128, static_cast<cuuint64_t>(16 * hd * 2)};
  cuuint32_t box[4] = {64, 16, static_cast<cuuint32_t>(hd / 64), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  BI_REQUIRE(r == CUDA_SUCCESS, BI_ERR_CUDA, "attention: cuTensorMapEncodeTiled failed for the KV cache (%d)",
             static_cast<int>(r));
  std::lock_guard<std::mutex> lock(g_cache_map_mutex);
  if (g_cache_maps.size() > 1024) g_cache_maps.clear();
  g_cache_maps.emplace_back(key, *out);
  return BI_OK;
}

// Tuning of the non-invariant decode schedule (bi_fast_attention_plan): 0 =
// the occupancy-chosen unit count below; 1 = fixed 256-token units (the
// invariant splits) combined left to right.
std::atomic<int> g_fast_attn_plan{0};

// Units per request the FAST plan asks for (the plan kernel caps it at 64 and
// at the request's page count): about four work items per SM over the batch;
// 0 asks the plan kernel for fixed 256-token units.
int fast_units_wanted(int B, int hkv) {
  if (g_fast_attn_plan.load() == 1) return 0;
  return std::max(1, (4 * num_sms() + B * hkv - 1) / (B * hkv));
}

template <int HD, int G>
bi_status decode_launch(const void* q, const void* kc, const void* vc, const int32_t* bt, const int32_t* kv_lens,
                        int B, const bi_attn_dims* dm, const ActDst& out, bi_mode mode, int target, const DecodeWs& w,
                        cudaStream_t s, bool make_plan = true) {
  // fp32-activation layers: fp32 queries (the consumers read them from global memory)
  const bool qf = dm->act_f32 != 0;
  if (mode == BI_MODE_INVARIANT_KSPLIT) mode = BI_MODE_INVARIANT;  // the split-K variant changes the GEMM only
  if (make_plan) {
    const int fast_units = fast_units_wanted(B, dm->num_kv_heads);
    BI_TIMED(::bi::kTagAttnPlan, s,
             BI_PDL_CHECK(launch_pdl(decode_plan_kernel, dim3(1), dim3(1024), 0, s, kv_lens, B, dm->num_kv_heads,
                                     static_cast<int>(mode), target, fast_units, dm->max_pages * kPage, w.plan)));
    BI_LAUNCH_CHECK();
  }
  const float sl2 = dm->scale * kLog2e;
  CUtensorMap kmap, vmap;
  BI_TRY(cache_map(kc, dm->num_pages, dm->num_kv_heads, HD, &kmap));
  BI_TRY(cache_map(vc, dm->num_pages, dm->num_kv_heads, HD, &vmap));
  int grid = 0;
  const size_t dsmem = decode_smem<HD, G>();
  if (qf) {
    BI_TRY((decode_grid<HD, G, 3>(&grid)));
    BI_TIMED(::bi::kTagAttnDecodeSplit, s,
             BI_PDL_CHECK(launch_pdl(decode_split_kernel<HD, G, 3>, dim3(grid), dim3(kDecodeThreads), dsmem, s,
                                     kmap, vmap, nullptr, static_cast<const float*>(q), bt, B, dm->num_q_heads,
                                     dm->num_kv_heads, dm->max_pages, dm->num_pages, sl2, w.plan, w.part,
                                     make_plan ? 0 : 1)));
  } else {
    BI_TRY((decode_grid<HD, G, 1>(&grid)));
    BI_TIMED(::bi::kTagAttnDecodeSplit, s,
             BI_PDL_CHECK(launch_pdl(decode_split_kernel<HD, G, 1>, dim3(grid), dim3(kDecodeThreads), dsmem, s,
                                     kmap, vmap, static_cast<const __nv_bfloat16*>(q), nullptr, bt, B,
                                     dm->num_q_heads, dm->num_kv_heads, dm->max_pages, dm->num_pages, sl2, w.plan,
                                     w.part, make_plan ? 0 : 1)));
  }
  BI_LAUNCH_CHECK();
  BI_TIMED(::bi::kTagAttnDecodeMerge, s,
           BI_PDL_CHECK(launch_pdl(decode_merge_kernel, dim3(B * dm->num_kv_heads), dim3(G * HD / 4), 0, s, w.part,
                                   w.plan, out, B, dm->num_q_heads, dm->num_kv_heads, HD)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

template <int HD, int G>
bi_status prefill_launch(const void* q, const void* kc, const void* vc, const int32_t* bt, const int32_t* q_start,
                         const int32_t* q_pos0, int B, int T, const bi_attn_dims* dm, const ActDst& out,
                         bi_mode mode, int target, const PrefillWs& w, cudaStream_t s) {
  const bool qf = dm->act_f32 != 0;  // fp32 queries
  if (mode == BI_MODE_INVARIANT_KSPLIT) mode = BI_MODE_INVARIANT;  // the split-K variant changes the GEMM only
  BI_TIMED(::bi::kTagAttnPlan, s, BI_PDL_CHECK(launch_pdl(prefill_plan_kernel, dim3(1), dim3(1024), 0, s, q_start, q_pos0, B, T, static_cast<int>(mode), target, w.plan)));
  BI_LAUNCH_CHECK();
  const size_t smem = sizeof(PrefillSmem<HD, G>);
  const float sl2 = dm->scale * kLog2e;
  auto go = [&](auto kern) -> bi_status {
    BI_CUDA_TRY(ensure_smem_limit(reinterpret_cast<const void*>(kern), static_cast<int>(smem)));
    BI_TIMED(::bi::kTagAttnPrefillSplit, s,
             BI_PDL_CHECK(launch_pdl(kern, dim3(num_sms()), dim3(kGroupThreads * kPrefillGroups), smem, s,
                                     qf ? nullptr : static_cast<const __nv_bfloat16*>(q),
                                     qf ? static_cast<const float*>(q) : nullptr,
                                     static_cast<const __nv_bfloat16*>(kc), static_cast<const __nv_bfloat16*>(vc), bt,
                                     q_pos0, q_start, dm->num_q_heads, dm->num_kv_heads, dm->max_pages,
                                     dm->num_pages, sl2, w.plan, w.part)));
    BI_LAUNCH_CHECK();
    return BI_OK;
  };
  // the same split function as decode (same bits): one query term (bf16) or three (fp32)
  BI_TRY(qf ? go(prefill_split_kernel<HD, G, 3>) : go(prefill_split_kernel<HD, G, 1>));
  BI_TIMED(::bi::kTagAttnPrefillMerge, s, BI_PDL_CHECK(launch_pdl(prefill_merge_kernel, dim3(T * dm->num_kv_heads), dim3(G * HD / 4), 0, s, w.part, w.plan, q_start, q_pos0, B,
                                                               out, dm->num_q_heads, dm->num_kv_heads, HD)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

#define BI_ATTN_DISPATCH(FN, ...)                                           \
  do {                                                                      \
    const int G_ = dims->num_q_heads / dims->num_kv_heads;                  \
    if (dims->head_dim == 128) {                                            \
      if (G_ == 1) return FN<128, 1>(__VA_ARGS__);                          \
      if (G_ == 2) return FN<128, 2>(__VA_ARGS__);                          \
      return FN<128, 4>(__VA_ARGS__);                                       \
    }                                                                       \
    if (G_ == 1) return FN<64, 1>(__VA_ARGS__);                             \
    if (G_ == 2) return FN<64, 2>(__VA_ARGS__);                             \
    return FN<64, 4>(__VA_ARGS__);                                          \
  } while (0)

}  // namespace attn

bi_status decode_attention_impl(const void* q, const void* kc, const void* vc, const int32_t* bt,
                                const int32_t* kv_lens, int32_t B, const bi_attn_dims* dims, void* out, bi_mode mode,
                                int32_t target, void* ws, size_t ws_bytes, cudaStream_t s) {
  clear_error();
  BI_TRY(attn::check_dims(dims));
  BI_REQUIRE(B >= 0, BI_ERR_INVALID_ARG, "bi_decode_attention: B=%d", B);
  BI_REQUIRE(mode_valid(mode), BI_ERR_INVALID_ARG, "mode %d",
             static_cast<int>(mode));
  BI_REQUIRE(mode != BI_MODE_PROTECTED || target < B, BI_ERR_INVALID_ARG, "target_request %d >= B %d", target, B);
  if (B == 0) return BI_OK;
  BI_REQUIRE(q && kc && vc && bt && kv_lens && out, BI_ERR_INVALID_ARG, "bi_decode_attention: null pointer");
  BI_REQUIRE(aligned16(q) && aligned16(kc) && aligned16(vc) && aligned16(out), BI_ERR_INVALID_ARG,
             "bi_decode_attention: q/caches/out must be 16-byte aligned");
  attn::DecodeWs w = attn::carve_decode(ws, ws_bytes, B, dims);
  BI_REQUIRE(ws != nullptr && w.bytes <= ws_bytes, BI_ERR_WORKSPACE, "bi_decode_attention: workspace %zu < %zu",
             ws_bytes, w.bytes);
  const ActDst od{out, 0, dims->act_f32 ? kActF32 : kActBF16};
  BI_ATTN_DISPATCH(attn::decode_launch, q, kc, vc, bt, kv_lens, B, dims, od, mode,
                   mode == BI_MODE_PROTECTED ? target : -1, w, s);
}

bi_status prefill_attention_impl(const void* q, const void* kc, const void* vc, const int32_t* bt,
                                 const int32_t* q_start, const int32_t* q_pos0, int32_t B, int32_t T,
                                 const bi_attn_dims* dims, void* out, bi_mode mode, int32_t target, void* ws,
                                 size_t ws_bytes, cudaStream_t s) {
  clear_error();
  BI_TRY(attn::check_dims(dims));
  BI_REQUIRE(B >= 0 && T >= 0 && (B > 0 || T == 0), BI_ERR_INVALID_ARG, "bi_prefill_attention: B=%d T=%d", B, T);
  BI_REQUIRE(mode_valid(mode), BI_ERR_INVALID_ARG, "mode %d",
             static_cast<int>(mode));
  BI_REQUIRE(mode != BI_MODE_PROTECTED || target < B, BI_ERR_INVALID_ARG, "target_request %d >= B %d", target, B);
  if (T == 0) return BI_OK;
  BI_REQUIRE(q && kc && vc && bt && q_start && q_pos0 && out, BI_ERR_INVALID_ARG, "bi_prefill_attention: null pointer");
  BI_REQUIRE(aligned16(q) && aligned16(kc) && aligned16(vc) && aligned16(out), BI_ERR_INVALID_ARG,
             "bi_prefill_attention: q/caches/out must be 16-byte aligned");
  attn::PrefillWs w = attn::carve_prefill(ws, ws_bytes, B, T, dims);
  BI_REQUIRE(ws != nullptr && w.bytes <= ws_bytes, BI_ERR_WORKSPACE, "bi_prefill_attention: workspace %zu < %zu",
             ws_bytes, w.bytes);
  const ActDst od{out, 0, dims->act_f32 ? kActF32 : kActBF16};
  BI_ATTN_DISPATCH(attn::prefill_launch, q, kc, vc, bt, q_start, q_pos0, B, T, dims, od, mode,
                   mode == BI_MODE_PROTECTED ? target : -1, w, s);
}

// Prefill attention inside the layer: output written as `out` says (three
// bf16 planes for fp32-activation layers).
bi_status prefill_attention_layer(const void* q, const void* kc, const void* vc, const int32_t* bt,
                                  const int32_t* q_start, const int32_t* q_pos0, int32_t B, int32_t T,
                                  const bi_attn_dims* dims, const ActDst& out, bi_mode mode, int32_t target, void* ws,
                                  size_t ws_bytes, cudaStream_t s) {
  BI_TRY(attn::check_dims(dims));
  if (T == 0) return BI_OK;
  attn::PrefillWs w = attn::carve_prefill(ws, ws_bytes, B, T, dims);
  BI_REQUIRE(ws != nullptr && w.bytes <= ws_bytes, BI_ERR_WORKSPACE, "prefill attention: workspace %zu < %zu",
             ws_bytes, w.bytes);
  BI_ATTN_DISPATCH(attn::prefill_launch, q, kc, vc, bt, q_start, q_pos0, B, T, dims, out, mode,
                   mode == BI_MODE_PROTECTED ? target : -1, w, s);
}

// ------------------------------------------------------------------ decode without a caller workspace
// Some callers cannot allocate device memory when they call attention: a plugin
// inside a host framework whose caching allocator owns all of the GPU's memory,
// or a serving loop that must never call cudaMalloc (it can synchronise the
// device).  bi_decode_attention_noalloc serves them from a fixed scratch array
// that lives in this library's device data for as long as the library is loaded.
namespace attn {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per GPU that loads the library
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
// device address of the scratch, per (device, CUDA context): a context created
// after a device reset gets its own lookup
std::vector<std::pair<std::pair<int, void*>, void*>> g_noalloc_address;

// The current CUDA context (the driver's cuCtxGetCurrent, reached through the
// runtime's entry-point query), or null if it cannot be read.
void* current_context() {
  using Fn = int (*)(void**);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(p);
  });
  void* ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != 0) return nullptr;
  return ctx;
}

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device and context (with that device current) and cached.
bi_status noalloc_scratch_address(void** out) {
  int dev = 0;
  BI_CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  const auto key = std::make_pair(dev, current_context());
  for (const auto& e : g_noalloc_address)
    if (e.first == key && key.second != nullptr) {
      *out = e.second;
      return BI_OK;
    }
  void* p = nullptr;
  BI_CUDA_TRY(cudaGetSymbolAddress(&p, g_noalloc_scratch));  // also makes the device's context current
  g_noalloc_address.emplace_back(std::make_pair(dev, current_context()), p);
  *out = p;
  return BI_OK;
}

// Scratch layout of one call: the same plan and partial-state arrays as the
// workspace path, with the partial states sized for the units `mode` can plan:
// INVARIANT one per 256 tokens of the longest allowed request; FAST at most
// f = min(64, fast_units_wanted) per request (the value decode_launch passes to
// the plan kernel, computed by the same function); PROTECTED f per request
// plus the target's invariant units.
DecodeWs carve_decode_noalloc(void* base, int B, const bi_attn_dims* dm, bi_mode mode, int target) {
  DecodeWs r;
  const size_t inv = static_cast<size_t>((dm->max_pages * kPage + kSplit - 1) / kSplit);
  const int fw = fast_units_wanted(B, dm->num_kv_heads);
  const size_t f = fw <= 0 ? inv : static_cast<size_t>(std::min(kMaxFastUnits, fw));
  size_t units;
  if (mode_invariant(mode)) units = static_cast<size_t>(B) * inv;
  else if (mode == BI_MODE_PROTECTED && target >= 0) units = static_cast<size_t>(B - 1) * f + std::max(inv, f);
  else units = static_cast<size_t>(B) * f;
  const size_t pb = carve_decode_plan(base, B, dm->num_kv_heads, units, &r.plan);
  const size_t qb = carve_decode_parts(base ? static_cast<char*>(base) + pb : nullptr, units, dm, &r.part);
  r.bytes = pb + qb;
  return r;
}

}  // namespace attn

bi_status decode_attention_noalloc_impl(const void* q, const void* kc, const void* vc, const int32_t* bt,
                                        const int32_t* kv_lens, int32_t B, const bi_attn_dims* dims, void* out,
                                        bi_mode mode, int32_t target, cudaStream_t s) {
  clear_error();
  BI_TRY(attn::check_dims(dims));
  BI_REQUIRE(B >= 0, BI_ERR_INVALID_ARG, "bi_decode_attention_noalloc: B=%d", B);
  BI_REQUIRE(mode_valid(mode), BI_ERR_INVALID_ARG, "mode %d",
             static_cast<int>(mode));
  BI_REQUIRE(mode != BI_MODE_PROTECTED || target < B, BI_ERR_INVALID_ARG, "target_request %d >= B %d", target, B);
  if (B == 0) return BI_OK;
  BI_REQUIRE(q && kc && vc && bt && kv_lens && out, BI_ERR_INVALID_ARG, "bi_decode_attention_noalloc: null pointer");
  BI_REQUIRE(aligned16(q) && aligned16(kc) && aligned16(vc) && aligned16(out), BI_ERR_INVALID_ARG,
             "bi_decode_attention_noalloc: q/caches/out must be 16-byte aligned");
  const int tgt = mode == BI_MODE_PROTECTED ? target : -1;
  const size_t need = attn::carve_decode_noalloc(nullptr, B, dims, mode, tgt).bytes;
  BI_REQUIRE(need <= attn::kNoAllocScratchBytes, BI_ERR_UNSUPPORTED,
             "bi_decode_attention_noalloc: this batch needs %zu bytes of scratch but the fixed scratch holds %zu "
             "bytes; use bi_decode_attention with a caller workspace",
             need, attn::kNoAllocScratchBytes);
  void* base = nullptr;
  BI_TRY(attn::noalloc_scratch_address(&base));
  attn::DecodeWs w = attn::carve_decode_noalloc(base, B, dims, mode, tgt);
  const ActDst od{out, 0, dims->act_f32 ? kActF32 : kActBF16};
  BI_ATTN_DISPATCH(attn::decode_launch, q, kc, vc, bt, kv_lens, B, dims, od, mode, tgt, w, s);
}

// Decode attention for the layer loop: the plan lives in `plan_ws` (sized by
// decode_plan_bytes) and is built only when make_plan is set, so the layers of
// one step share it; the partial states live in `part_ws`.
size_t decode_plan_bytes(int32_t B, const bi_attn_dims* dims) {
  attn::DecodePlan p;
  return attn::carve_decode_plan(nullptr, B, dims->num_kv_heads,
                                 static_cast<size_t>(B) * attn::max_units_per_request(dims), &p);
}

size_t decode_parts_bytes(int32_t B, const bi_attn_dims* dims) {
  attn::Partials p;
  return attn::carve_decode_parts(nullptr, static_cast<size_t>(B) * attn::max_units_per_request(dims), dims, &p);
}

bi_status decode_attention_layer(const void* q, const void* kc, const void* vc, const int32_t* bt,
                                 const int32_t* kv_lens, int32_t B, const bi_attn_dims* dims, const ActDst& out,
                                 bi_mode mode, int32_t target, void* plan_ws, bool make_plan, void* part_ws,
                                 size_t part_bytes, cudaStream_t s) {
  BI_TRY(attn::check_dims(dims));
  BI_REQUIRE(B >= 1 && plan_ws && part_ws && part_bytes >= decode_parts_bytes(B, dims), BI_ERR_WORKSPACE,
             "decode attention: workspace");
  attn::DecodeWs w;
  attn::carve_decode_plan(plan_ws, B, dims->num_kv_heads, static_cast<size_t>(B) * attn::max_units_per_request(dims),
                          &w.plan);
  attn::carve_decode_parts(part_ws, static_cast<size_t>(B) * attn::max_units_per_request(dims), dims, &w.part);
  BI_ATTN_DISPATCH(attn::decode_launch, q, kc, vc, bt, kv_lens, B, dims, out, mode,
                   mode == BI_MODE_PROTECTED ? target : -1, w, s, make_plan);
}

size_t decode_attention_ws(int32_t B, const bi_attn_dims* dims) {
  if (B <= 0 || attn::check_dims(dims) != BI_OK) return 0;
  return attn::carve_decode(nullptr, 0, B, dims).bytes;
}

size_t prefill_attention_ws(int32_t B, int32_t T, const bi_attn_dims* dims) {
  if (B <= 0 || T <= 0 || attn::check_dims(dims) != BI_OK) return 0;
  return attn::carve_prefill(nullptr, 0, B, T, dims).bytes;
}

int take_attn_device_error(cudaStream_t s, int32_t* code) {
  unsigned v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, attn::g_attn_err_word, sizeof(v), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return 1;
  if (cudaStreamSynchronize(s) != cudaSuccess) return 1;
  if (v != 0) {
    unsigned zero = 0;
    if (cudaMemcpyToSymbolAsync(attn::g_attn_err_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
      return 1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return 1;
  }
  *code = static_cast<int32_t>(v);
  return 0;
}

}  // namespace bi

extern "C" bi_status bi_fast_attention_plan(int32_t plan) {
  bi::clear_error();
  BI_REQUIRE(plan == 0 || plan == 1, BI_ERR_INVALID_ARG, "bi_fast_attention_plan: plan %d", plan);
  bi::attn::g_fast_attn_plan.store(plan);
  return BI_OK;
}

extern "C" size_t bi_decode_attention_workspace(int32_t B, const bi_attn_dims* dims, bi_mode) {
  return bi::decode_attention_ws(B, dims);
}

extern "C" bi_status bi_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_table, const int32_t* kv_lens, int32_t B,
                                         const bi_attn_dims* dims, void* out, bi_mode mode, int32_t target_request,
                                         void* workspace, size_t ws_bytes, bi_stream s) {
  return bi::decode_attention_impl(q, k_cache, v_cache, block_table, kv_lens, B, dims, out, mode, target_request,
                                   workspace, ws_bytes, reinterpret_cast<cudaStream_t>(s));
}

extern "C" bi_status bi_decode_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                 const int32_t* block_table, const int32_t* kv_lens, int32_t B,
                                                 const bi_attn_dims* dims, void* out, bi_mode mode,
                                                 int32_t target_request, bi_stream s) {
  return bi::decode_attention_noalloc_impl(q, k_cache, v_cache, block_table, kv_lens, B, dims, out, mode,
                                           target_request, reinterpret_cast<cudaStream_t>(s));
}

extern "C" size_t bi_prefill_attention_workspace(int32_t B, int32_t T, const bi_attn_dims* dims, bi_mode) {
  return bi::prefill_attention_ws(B, T, dims);
}

extern "C" bi_status bi_prefill_attention(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_table, const int32_t* q_start, const int32_t* q_pos0,
                                          int32_t B, int32_t T, const bi_attn_dims* dims, void* out, bi_mode mode,
                                          int32_t target_request, void* workspace, size_t ws_bytes, bi_stream s) {
  return bi::prefill_attention_impl(q, k_cache, v_cache, block_table, q_start, q_pos0, B, T, dims, out, mode,
                                    target_request, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(s));
}
