// Batch-invariant bf16 GEMM on the sm_103a tensor cores (tcgen05 + TMEM, fed by TMA).
//
// C[i][j] = sum_k A[i][k] * W[j][k]  (+ residual[i][j]), fp32 accumulation.
// (devpress digest of "Defeating Nondeterminism in LLM Inference", section 3.2:
// a matmul is pointwise products plus a reduction over k; it stays batch
// invariant when every output tile reduces its whole K range inside one core
// with one kernel configuration for every M, i.e. no split-K.  "Batch-Invariant
// Kernel" notes, section GEMM: the K split may depend on K only.)
//
// Reduction geometry, identical for every M, N and CTA shape:
//   * tcgen05.mma.cta_group::1.kind::f16 with M=128, K=16, bf16 operands from
//     shared memory (128-byte swizzled, K-major), fp32 accumulator in tensor memory;
//   * the K range is consumed in 64-wide k-tiles in ascending order, four
//     instructions of K=16 per k-tile in ascending order; the first
//     instruction of an output tile overwrites the accumulator, all others add.
// An output element therefore sees the same instruction sequence with the
// same operands whatever M is and whichever CTA computes it.  The
// instruction's N extent (the CTA tile width, 32-256 columns) and the
// persistent tile-to-CTA mapping are scheduling choices that never touch an
// element's arithmetic; the row-0 M sweeps check this bitwise across widths.
//
// Roles in a CTA of 192 threads: warp 0 issues TMA loads, warp 1 owns the
// tensor memory and issues the MMAs (one thread), warps 2-5 drain the
// accumulator (tcgen05.ld) and store.  Shared-memory stages and two
// tensor-memory accumulators are handed between roles with mbarriers.  Every
// wait is bounded: when one runs out the kernel records a site code in a
// device error word, stops all roles, waits (bounded) for its own copies and
// MMAs, frees its tensor memory and returns.
//
// FAST mode (the non-invariant schedule used to measure the cost of
// invariance): when there are fewer tiles than SMs the K range is split over
// several CTAs and the fp32 partials are added in a second pass, so an
// element's rounding depends on M.  PROTECTED: tiles holding target rows are
// never split.  INVARIANT_KSPLIT: a K split fixed by the weight shape (N, K).
//
// fp32 activations (planes = 3): A holds fp32 activations as three bf16 planes
// hi, mid, lo whose sum is the fp32 value (common.cuh); every k16 step issues
// the instruction once per plane, in plane order, on the same B operand, so
// C = sum_k (hi + mid + lo)[i][k] * W[j][k] with exact products and fp32
// accumulation.  The order is fixed per element, so this is as batch invariant
// as the one-plane GEMM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <tuple>
#include <vector>
#include <unordered_map>

#include "common.cuh"

namespace bi {
namespace gemm {

constexpr int kBM = 128;        // instruction / tile rows
constexpr int kBN = 64;         // instruction columns
constexpr int kBK = 64;         // k-tile (128 bytes of bf16: one swizzle row)
constexpr int kUK = 16;         // instruction K
constexpr int kProducerWarps = 1;
constexpr int kMmaWarp = kProducerWarps;
constexpr int kThreads = (kProducerWarps + 1 + 4) * 32;  // SM-pair kernel
// one-SM kernel: two epilogue warps per tensor-memory lane quarter, each taking
// half of a tile's columns (or half of each SwiGLU chunk's outputs)
constexpr int kEpiWarpsTc = 8;
constexpr int kThreadsTc = (kProducerWarps + 1 + kEpiWarpsTc) * 32;
constexpr int kATileBytes = kBM * kBK * 2;  // 16 KiB
constexpr int kSmemLimit = 227 * 1024;     // dynamic shared memory per CTA
constexpr int kMaxStages = 16;
constexpr int kOverreadSlack = kATileBytes;  // see the A-tile note below
constexpr int kMaxSplitK = 16;

__device__ unsigned int g_err_word = 0;

enum OutKind : int { kOutBF16 = 0, kOutF32 = 1 };

struct Args {
  int M, N, K;
  int a_rows;       // rows of A per TMA box (16, 32, 64 or 128)
  int m64;          // 1 (M <= 64): instructions of M = 64, accumulator row r in tensor-memory lane 32 (r / 16) + r % 16
  int kbs;          // k-blocks per stage (one TMA box spans them when map3d)
  int map3d;        // tensor maps are [kblock][rows][64] views (K % 64 == 0)
  int stage_bytes;  // kbs x (A box + TN rows of B)
  int stages;
  int m_tiles, n_tiles;  // n_tiles counts CTA-wide column tiles (TN wide)
  int splits;            // K splits of the other tiles, one CTA unit each (partials summed by a second pass)
  int tm0, tm1;          // m-tiles [tm0, tm1) are computed whole by one unit each
  int seq;               // ... as `seq` K-split partials merged inside the CTA (1: one pass over K)
  int units;             // total work units
  int kb_total;          // k-tiles in K
  int prefetch_w;        // 1: W is constant while the previous kernel runs (weights of a forward pass), so
                         // the first stages' W copies may be issued before waiting for that kernel
  void* C;
  const __nv_bfloat16* R;  // residual or null
  float* partial;          // [splits][M][N] fp32 (split units only)
  int out_kind;
  int plane_rows;          // rows of each A plane (three planes for fp32 A; the kernel's PL)
  const float* Rf;         // fp32 residual (fp32 output) or null
  int swiglu;                  // 1: gate|up GEMM with SwiGLU in the epilogue: a tile's first TN/2 B rows are
                               // gate rows nt*TN/2.., the next TN/2 the up rows F + nt*TN/2.. of the same outputs;
                               // the epilogue writes act[row][nt*TN/2 + j] = swiglu(bf16(gate), bf16(up))
  int F;                       // ... output width (half of N)
  __nv_bfloat16* act;          // ... output [M][F]
  unsigned long long wait_ns;  // limit of every bounded wait (2 s; shorter only under the test hook below)
  int drop_first_stage;        // test hook: CTA 0 issues no copies for its first stage (its waits then run out)
};

// ------------------------------------------------------------------ PTX wrappers
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

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Bounded wait, slow path.  Returns false (after recording `site`) when the
// limit runs out or another role has already aborted.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, int site,
                                       uint64_t limit_ns) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u) {
      if (*abort_flag) return false;
      const uint64_t now = global_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_ns) {
        atomicCAS(&g_err_word, 0u, static_cast<unsigned>(site));
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag, int site,
                                             uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, site, limit_ns);
}

// Time-bounded wait that ignores the abort flag (used while draining after an abort).
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity) && global_ns() - t0 < kWaitLimitNs) {
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z,
                                            int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Weight copies of a GEMM with one row tile read every weight byte once per
// pass: they carry an L2 evict-first cache policy, so the weight stream does not
// push out of L2 the activations that the next kernels read.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 int z, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 int z, int w, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// An MMA and a commit issued by one elected lane of a warp whose lanes all
// execute the call with the same operands: the warp's control flow and the
// descriptors stay uniform, and a small-N MMA issues in about 40 cycles instead
// of about 55 from a single-lane branch (measured on this GB300 with a probe of
// back-to-back M=128, N=32 instructions).
__device__ __forceinline__ void tc_mma_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), descriptor
// version 1, base offset 0 (tiles are 1024-byte aligned).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;    // leading byte offset (unused with this swizzle)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;  // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;           // version
  d |= static_cast<uint64_t>(2) << 61;           // 128-byte swizzle
  return d;
}

// Instruction descriptor: fp32 accumulator, bf16 A and B, both K-major, M = m (128 or 64), N = n.
// An M = 64 instruction costs the tensor pipe less than an M = 128 one at decode widths (N <= 64: about 31
// against 40 cycles per instruction issued back to back, measured on this GB300); every accumulator element
// is the same chain of K = 16 steps either way.
__host__ __device__ constexpr uint32_t idesc_for(int n, int m = kBM) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// unit -> (m tile, n tile, split index, split count)
__device__ __forceinline__ void unit_coords(const Args& a, int u, int& mt, int& nt, int& s, int& nsplit, int& seq) {
  const int prot = a.tm1 - a.tm0;
  const int per_col = prot + (a.m_tiles - prot) * a.splits;
  nt = u / per_col;
  int r = u % per_col;
  seq = 1;
  const int before = a.tm0 * a.splits;
  if (r < before) {
    mt = r / a.splits;
    s = r % a.splits;
    nsplit = a.splits;
  } else if (r < before + prot) {
    mt = a.tm0 + (r - before);
    s = 0;
    nsplit = 1;
    seq = a.seq;
  } else {
    r -= before + prot;
    mt = a.tm1 + r / a.splits;
    s = r % a.splits;
    nsplit = a.splits;
  }
}

// K-split s of n: k-tiles [floor(s*T/n), floor((s+1)*T/n)), T = k-tiles in K.
// The partition depends on (T, n) only; with n <= T every part is non-empty.
__host__ __device__ __forceinline__ void k_range(int kb_total, int s, int nsplit, int& kb0, int& kb1) {
  kb0 = static_cast<int>((static_cast<int64_t>(s) * kb_total) / nsplit);
  kb1 = static_cast<int>((static_cast<int64_t>(s + 1) * kb_total) / nsplit);
}

// Shared memory: [barrier block 1 KiB][stage 0]..[stage n-1][slack].  A stage
// holds kbs A boxes of a_rows rows then kbs B boxes of TN rows (one per k-block).
//
// A-tile note: the instruction always reads 128 rows of A (16 KiB) from the
// stage start.  When M <= 64 only the first a_rows rows are loaded; the
// instruction's rows a_rows..127 then read whatever follows in shared memory
// (the B tile, the next stage, or the trailing slack, never outside the
// allocation) and produce accumulator rows that are never stored.  Each output
// row depends only on its own A row, so the rows that are stored are computed
// exactly as with a full tile; the saved shared memory holds more weight bytes
// in flight at decode sizes.
constexpr int kBarBlock = 1024;

__host__ __device__ constexpr size_t smem_bytes(int stages, int stage_bytes, int a_rows) {
  return 1024 /* alignment slack */ + kBarBlock + static_cast<size_t>(stages) * stage_bytes +
         (a_rows < kBM ? kOverreadSlack : 0);
}

// PL: planes of A (1: bf16 A; 3: fp32 A as three bf16 planes).  A compile-time
// count keeps the one-plane kernel free of the plane loops on its latency path.
template <int TN, int PL>
__global__ void __launch_bounds__(kThreadsTc, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                                                              const __grid_constant__ CUtensorMap tmW, const Args a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // two accumulators of TN columns, plus the running sum of merged units when
  // it fits (TN <= 128); allocations are powers of two
  constexpr int kTmemCols = TN == 32 ? 128 : TN == 64 ? 256 : 512;
  const int kStages = a.stages;
  const int kStageBytes = a.stage_bytes;
  const int kbs = a.kbs;
  const int a_tile = a.a_rows * kBK * 2;      // one k-block of A
  const int b_tile = TN * kBK * 2;            // one k-block of B
  const int a_plane = kbs * a_tile;           // one plane of A in a stage
  const int a_bytes = PL * a_plane;           // A part of a stage
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  unsigned char* tiles = smem + kBarBlock;
  // bars: full[kMaxStages], empty[kMaxStages], tfull[2], tempty[2], drain
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kMaxStages;
  const uint32_t tfull0 = empty0 + 8 * kMaxStages;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain_bar = tempty0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, kEpiWarpsTc);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything below reads or writes memory shared with the previous kernel,
  // except the weight copies of the first stages when a.prefetch_w is set: the
  // producer issues those first (their stages are fresh, so no empty-wait is
  // needed) and only then waits, so weight latency overlaps the previous kernel.
  // B part of a stage: the tile's TN weight rows (for the SwiGLU GEMM TN/2 gate
  // rows then the TN/2 up rows of the same outputs, one box of a row-pair map)
  // (one row tile: every weight byte is read once, see l2_evict_first_policy)
  const bool w_once = a.m_tiles == 1;
  const uint64_t w_pol = l2_evict_first_policy();
  auto load_w = [&](uint32_t dst, uint32_t bar, int nt, int kb) {
    if (a.swiglu) {
      if (a.map3d) tma_load_4d_hint(dst, &tmW, bar, 0, nt * (TN / 2), 0, kb, w_pol);
      else tma_load_3d_hint(dst, &tmW, bar, kb * kBK, nt * (TN / 2), 0, w_pol);
    } else if (a.map3d) {
      if (w_once) tma_load_3d_hint(dst, &tmW, bar, 0, nt * TN, kb, w_pol);
      else tma_load_3d(dst, &tmW, bar, 0, nt * TN, kb);
    } else {
      if (w_once) tma_load_2d_hint(dst, &tmW, bar, kb * kBK, nt * TN, w_pol);
      else tma_load_2d(dst, &tmW, bar, kb * kBK, nt * TN);
    }
  };
  int pre_stages = 0;  // stages whose W copy (and transaction count) was issued early
  if (warp < kProducerWarps && lane == 0 && a.prefetch_w && blockIdx.x < a.units) {
    int mt, nt, s, ns, seq, kb0, kb1;
    unit_coords(a, blockIdx.x, mt, nt, s, ns, seq);
    if (seq > 1) k_range(a.kb_total, 0, seq, kb0, kb1);
    else k_range(a.kb_total, s, ns, kb0, kb1);
    for (int kb = kb0; kb < kb1 && pre_stages < kStages; kb += kbs, ++pre_stages) {
      const uint32_t fb = full0 + 8 * pre_stages;
      const uint32_t sa = smem_u32(tiles + pre_stages * kStageBytes);
      mbar_expect_tx(fb, static_cast<uint32_t>(kStageBytes));
      load_w(sa + a_bytes, fb, nt, kb);
    }
  }
  pdl_wait();
  pdl_trigger();

  if (warp < kProducerWarps) {
    // ------------------------------------------------------------ TMA producer
    // One thread issues A then B of every stage in consumption order.
    if (lane == 0) {
      // the stages whose weight copies went out before the wait (first use, parity 0)
      uint32_t issued_mask = pre_stages >= 32 ? ~0u : ((1u << pre_stages) - 1u), issued_par = 0;
      bool ok = true;
      int st = 0;        // stage slot and its phase parity, advanced in the same
      uint32_t ph = 0;   // sequence as the MMA warp's
      for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        int mt, nt, s, ns, seq;
        unit_coords(a, u, mt, nt, s, ns, seq);
        for (int q = 0; q < seq && ok; ++q) {
          int kb0, kb1;
          if (seq > 1) k_range(a.kb_total, q, seq, kb0, kb1);
          else k_range(a.kb_total, s, ns, kb0, kb1);
          for (int kb = kb0; kb < kb1; kb += kbs) {
            const uint32_t fb = full0 + 8 * st;
            const uint32_t sa = smem_u32(tiles + st * kStageBytes);
            if (pre_stages > 0) {
              // W of this stage is already on its way (issued before the wait): add A only
              --pre_stages;
#pragma unroll
              for (int pl = 0; pl < PL; ++pl) {
                if (a.map3d) tma_load_3d(sa + pl * a_plane, &tmA, fb, 0, pl * a.plane_rows + mt * kBM, kb);
                else tma_load_2d(sa + pl * a_plane, &tmA, fb, kb * kBK, pl * a.plane_rows + mt * kBM);
              }
            } else {
              if (!wait_bounded(empty0 + 8 * st, ph ^ 1u, abort_flag, 1, a.wait_ns)) {
                ok = false;
                break;
              }
              if (a.drop_first_stage && blockIdx.x == 0 && u == static_cast<int>(blockIdx.x) && kb == kb0 &&
                  q == 0) {
                // test hook: this stage's barrier is never armed and nothing lands in it, so the MMA
                // thread's wait for it runs out (the stage is not counted as issued: nothing to drain)
                if (++st == kStages) {
                  st = 0;
                  ph ^= 1u;
                }
                continue;
              }
              mbar_expect_tx(fb, static_cast<uint32_t>(kStageBytes));
              if (a.map3d) {
#pragma unroll
                for (int pl = 0; pl < PL; ++pl)
                  tma_load_3d(sa + pl * a_plane, &tmA, fb, 0, pl * a.plane_rows + mt * kBM, kb);
                load_w(sa + a_bytes, fb, nt, kb);
              } else {
#pragma unroll
                for (int pl = 0; pl < PL; ++pl)
                  tma_load_2d(sa + pl * a_plane, &tmA, fb, kb * kBK, pl * a.plane_rows + mt * kBM);
                load_w(sa + a_bytes, fb, nt, kb);
              }
            }
            issued_mask |= 1u << st;
            issued_par = (issued_par & ~(1u << st)) | (ph << st);
            if (++st == kStages) {
              st = 0;
              ph ^= 1u;
            }
          }
        }
      }
      // Let every copy issued land before shared memory is released.  After a
      // normal run the MMA warp has already waited on each of them, so these
      // return at once; after an abort (which another role may raise after this
      // loop has ended) they keep the CTA alive until its copies are done.
      for (int i = 0; i < kStages; ++i)
        if (issued_mask & (1u << i)) wait_drain(full0 + 8 * i, (issued_par >> i) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Every pass over a K range (a whole tile, one split unit, or one of the
    // in-CTA partials of a merged unit) goes into the next of the two
    // accumulators and is handed to the epilogue on its own.  The whole warp
    // runs the loop; one elected lane issues each MMA and commit.  Every lane
    // waits on the barriers itself and the warp goes on only if all of them saw
    // the phase complete, so the loop stays uniform even when a wait runs out.
    {
      auto wait_all = [&](uint32_t bar, uint32_t par, int site) -> bool {
        const bool r = wait_bounded(bar, par, abort_flag, site, a.wait_ns);
        return __all_sync(0xffffffffu, r);
      };
      const uint64_t desc0 = sw128_desc(smem_u32(tiles));
      const uint32_t kIdescW = a.m64 ? idesc_for(TN, 64) : idesc_for(TN);
      int st = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      bool any = false;
      for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        int mt, nt, s, ns, seq;
        unit_coords(a, u, mt, nt, s, ns, seq);
        for (int q = 0; q < seq && ok; ++q) {
          int kb0, kb1;
          if (seq > 1) k_range(a.kb_total, q, seq, kb0, kb1);
          else k_range(a.kb_total, s, ns, kb0, kb1);
          if (!wait_all(tempty0 + 8 * acc, acc_ph ^ 1u, 2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * TN);
          for (int kb = kb0; kb < kb1; kb += kbs) {
            if (!wait_all(full0 + 8 * st, ph, 3)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // descriptors of this stage: start addresses advance in 16-byte units
            const uint64_t sdesc = desc0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
            const int nkb = min(kbs, kb1 - kb);  // k-blocks of this stage inside the range
            for (int j = 0; j < nkb; ++j) {
              const uint64_t adesc = sdesc + static_cast<uint64_t>((j * a_tile) >> 4);
              const uint64_t bdesc = sdesc + static_cast<uint64_t>((a_bytes + j * b_tile) >> 4);
              const uint32_t first = (kb + j == kb0) ? 1u : 0u;
              if constexpr (PL == 1) {
#pragma unroll
                for (int k = 0; k < kBK / kUK; ++k) {
                  // the first instruction of a pass overwrites the accumulator, all others add;
                  // one instruction spans the tile's TN columns: the B rows of a stage are
                  // contiguous 128-byte swizzle rows, 1024 bytes per 8-row group
                  const uint32_t accum = (k > 0 || !first) ? 1u : 0u;
                  tc_mma_elect(d0, adesc + static_cast<uint64_t>(2 * k), bdesc + static_cast<uint64_t>(2 * k),
                               kIdescW, accum);
                }
              } else {
                // fp32 A: per k16 step the planes hi, mid, lo in order, same B operand
#pragma unroll
                for (int k = 0; k < kBK / kUK; ++k) {
#pragma unroll
                  for (int pl = 0; pl < PL; ++pl) {
                    const uint32_t accum = (k > 0 || pl > 0 || !first) ? 1u : 0u;
                    tc_mma_elect(d0, adesc + static_cast<uint64_t>(((pl * a_plane) >> 4) + 2 * k),
                                 bdesc + static_cast<uint64_t>(2 * k), kIdescW, accum);
                  }
                }
              }
            }
            tc_commit_elect(empty0 + 8 * st);  // stage free once these MMAs have read it
            any = true;
            if (++st == kStages) {
              st = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit_elect(tfull0 + 8 * acc);
          if (++acc == 2) {
            acc = 0;
            acc_ph ^= 1u;
          }
        }
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0) && any) {
        // a commit arrives once every MMA issued above has completed
        tc_commit_elect(drain_bar);
        wait_drain(drain_bar, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (8 warps)
    // Thread = one accumulator row (tensor-memory lane), 32 columns per load;
    // the two warps of a lane quarter take alternate 32-column chunks.
    // Merged units: partial q is added into a running sum kept in a third
    // tensor-memory buffer, sum = ((0 + P0) + P1) + ..., rounded once at the end;
    // the second-pass reduction of split units adds the same partials in the
    // same order, so both give the same bits.
    // With M = 64 instructions the accumulator holds 16 rows per lane quarter
    // (lanes 32 w .. 32 w + 15); the warp's other lanes load and store nothing.
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int half = (warp - kProducerWarps - 1) >> 2;  // 0 or 1: which of the quarter's two warps
    const bool lane_live = !a.m64 || lane < 16;
    const int row_in_tile = a.m64 ? quarter * 16 + lane : quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t sum_base = lane_base + 2 * TN;  // running-sum buffer (merged units only)
    int acc = 0;
    uint32_t acc_ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
      int mt, nt, s, ns, seq;
      unit_coords(a, u, mt, nt, s, ns, seq);
      const int row = mt * kBM + row_in_tile;
      const bool row_ok = lane_live && row < a.M;
      for (int q = 0; q < seq; ++q) {
        if (!wait_bounded(tfull0 + 8 * acc, acc_ph, abort_flag, 4, a.wait_ns)) {
          ok = false;
          break;
        }
        __syncwarp();  // lanes leave the wait at different times; tcgen05.ld needs the whole warp
        tc_fence_after();
        const uint32_t tbase = lane_base + acc * TN;
        const bool last = q == seq - 1;
        if constexpr (TN % 64 == 0) {
          if (a.swiglu) {
            // gate chunk ch and up chunk ch of the tile give 32 outputs of a row: each accumulator value is
            // rounded to bf16 as the plain GEMM stores it, then the SwiGLU kernel's own function.  Both warps
            // of the lane quarter load the chunk pair and each computes half of the outputs.  With M = 64
            // instructions the quarter's 16 rows sit in lanes 0..15, so lanes 16..31 take the upper 16 columns
            // of the row of lane - 16 (shuffled over): every lane computes 8 outputs per chunk.
#pragma unroll 1
            for (int ch = 0; ch < TN / 64; ++ch) {
              uint32_t g[32], v[32];
              tc_ld32(tbase + ch * 32, g);
              tc_ld32(tbase + TN / 2 + ch * 32, v);
              const int col0 = nt * (TN / 2) + ch * 32;
              if (a.m64) {
                // this warp's 8 of the lane's 16 outputs: columns 8 half .. 8 half + 7 of its 16
                const int src = lane & 15;
                const bool upper = lane >= 16;
                float o[8];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                  // register indices stay compile-time: pick between the two halves' values
                  const uint32_t ga = half ? g[8 + e] : g[e], gb = half ? g[9 + e] : g[e + 1];
                  const uint32_t va = half ? v[8 + e] : v[e], vb = half ? v[9 + e] : v[e + 1];
                  const uint32_t gA = half ? g[24 + e] : g[16 + e], gB = half ? g[25 + e] : g[17 + e];
                  const uint32_t vA = half ? v[24 + e] : v[16 + e], vB = half ? v[25 + e] : v[17 + e];
                  const uint32_t g0 = __shfl_sync(0xffffffffu, gA, src);
                  const uint32_t g1 = __shfl_sync(0xffffffffu, gB, src);
                  const uint32_t v0 = __shfl_sync(0xffffffffu, vA, src);
                  const uint32_t v1 = __shfl_sync(0xffffffffu, vB, src);
                  const uint32_t gp = pack_bf16x2(__uint_as_float(upper ? g0 : ga), __uint_as_float(upper ? g1 : gb));
                  const uint32_t up = pack_bf16x2(__uint_as_float(upper ? v0 : va), __uint_as_float(upper ? v1 : vb));
                  o[e] = swiglu1(bf16_lo(gp), bf16_lo(up));
                  o[e + 1] = swiglu1(bf16_hi(gp), bf16_hi(up));
                }
                const int orow = mt * kBM + quarter * 16 + src;
                const int c0 = col0 + (upper ? 16 : 0) + 8 * half;
                if (orow < a.M && c0 < a.F)
                  *reinterpret_cast<uint4*>(a.act + static_cast<size_t>(orow) * a.F + c0) = pack8(o);
              } else {
                if (!row_ok || col0 >= a.F) continue;
                __nv_bfloat16* dst = a.act + static_cast<size_t>(row) * a.F + col0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int q8 = 2 * half + h;
                  if (col0 + 8 * q8 >= a.F) break;
                  float o[8];
#pragma unroll
                  for (int e = 0; e < 8; e += 2) {
                    const int i0 = 8 * h + e;  // compile-time; the other half's values sit 16 further on
                    const uint32_t gp = pack_bf16x2(__uint_as_float(half ? g[16 + i0] : g[i0]),
                                                    __uint_as_float(half ? g[17 + i0] : g[i0 + 1]));
                    const uint32_t up = pack_bf16x2(__uint_as_float(half ? v[16 + i0] : v[i0]),
                                                    __uint_as_float(half ? v[17 + i0] : v[i0 + 1]));
                    o[e] = swiglu1(bf16_lo(gp), bf16_lo(up));
                    o[e + 1] = swiglu1(bf16_hi(gp), bf16_hi(up));
                  }
                  *reinterpret_cast<uint4*>(dst + 8 * q8) = pack8(o);
                }
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
            if (++acc == 2) {
              acc = 0;
              acc_ph ^= 1u;
            }
            continue;
          }
        }
#pragma unroll 1
        for (int ch = half; ch < TN / 32; ch += 2) {
          uint32_t r[32];
          tc_ld32(tbase + ch * 32, r);
          if (seq > 1) {
            if constexpr (TN <= 128) {
              uint32_t t[32];
              if (q > 0) tc_ld32(sum_base + ch * 32, t);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                r[e] = __float_as_uint(__fadd_rn(q > 0 ? __uint_as_float(t[e]) : 0.f, __uint_as_float(r[e])));
              if (!last) {
                tc_st32(sum_base + ch * 32, r);
                continue;
              }
            }
          }
          const int col0 = nt * TN + ch * 32;
          if (!row_ok || col0 >= a.N) continue;
          if (ns > 1) {
            float* dst = a.partial + (static_cast<size_t>(s) * a.M + row) * a.N + col0;
#pragma unroll
            for (int g = 0; g < 8; ++g)
              if (col0 + 4 * g < a.N)
                *reinterpret_cast<float4*>(dst + 4 * g) =
                    make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
          } else if (a.out_kind == kOutF32) {
            float* dst = static_cast<float*>(a.C) + static_cast<size_t>(row) * a.N + col0;
            // fp32 residual: fp32-activation layers only
            const float* res = (PL > 1 && a.Rf) ? a.Rf + static_cast<size_t>(row) * a.N + col0 : nullptr;
#pragma unroll
            for (int g = 0; g < 8; ++g)
              if (col0 + 4 * g < a.N) {
                float4 v = make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                       __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
                if (res) {
                  const float4 rv = *reinterpret_cast<const float4*>(res + 4 * g);
                  v.x = __fadd_rn(v.x, rv.x); v.y = __fadd_rn(v.y, rv.y);
                  v.z = __fadd_rn(v.z, rv.z); v.w = __fadd_rn(v.w, rv.w);
                }
                *reinterpret_cast<float4*>(dst + 4 * g) = v;
              }
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.C) + static_cast<size_t>(row) * a.N + col0;
            const __nv_bfloat16* res = a.R ? a.R + static_cast<size_t>(row) * a.N + col0 : nullptr;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              if (col0 + 8 * g >= a.N) break;
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(r[8 * g + e]);
              if (res) {
                float rv[8];
                unpack8(*reinterpret_cast<const uint4*>(res + 8 * g), rv);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = __fadd_rn(f[e], rv[e]);
              }
              *reinterpret_cast<uint4*>(dst + 8 * g) = pack8(f);
            }
          }
        }
        if (seq > 1 && !last) asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          acc_ph ^= 1u;
        }
      }
    }
  }

  // Normal exit: the epilogue has consumed the last accumulator commit, so every
  // MMA has completed and every load was consumed.  After an abort the producer
  // and the MMA warp drained their own work above.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------ two-SM tiles (INVARIANT, M > 128)
// A cluster of two CTAs (an SM pair) computes 256 x TN2 output tiles (TN2 = 256,
// 224, 192 or 128; 224 makes N = 4096 exactly 19 column tiles, so 4 row tiles fill
// the 76 pairs of a 152-SM part in whole waves, and 192 makes N = 14336 75 column
// tiles, one wave for 256 rows) with tcgen05.mma.cta_group::2
// (instruction M = 256, N = TN2, K = 16).  CTA rank r
// loads A rows [256 i + 128 r, +128) and B rows [TN2 j + r TN2/2, +TN2/2) of
// every k-tile into its own shared memory; the even CTA issues the MMAs, which
// read both CTAs' operands and accumulate rows 128 r .. of the tile in CTA r's
// tensor memory.  Per SM a k-tile moves 16 KiB of A and TN2/2 rows of B, two
// thirds of what a one-SM 128 x 256 tile moves for the same flops, which is
// what lets the copy engines keep the tensor cores busy.  Per element the
// instruction sequence (ascending k-tiles, four K = 16 steps each, the first
// overwriting the accumulator) is the one of the one-SM kernel, so the bits
// are the same.
//
// Synchronisation (every wait bounded; a wait that runs out records a site
// code and the kernel winds down):
//   * full[s] lives in the even CTA and counts both CTAs' copy bytes (armed by
//     the even CTA's producer); the odd CTA's copies signal it remotely;
//   * the MMA commits arrive on empty[s] and tfull[a] of both CTAs (multicast);
//   * both CTAs' epilogue warps arrive on the even CTA's tempty[a];
//   * a handshake barrier in each CTA, armed by the other CTA, orders the
//     pair's tensor-memory allocation before the first MMA and keeps each CTA
//     alive at the end until the other no longer addresses it.
// The kernel waits for its predecessor before doing anything (no prologue
// overlaps another kernel), is launched without programmatic serialisation,
// and lets its successor start only when it exits.
constexpr int kPairTmemCols = 512;   // two accumulators of up to 256 columns
constexpr int kPairStagesMax = 16;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// address of the same shared variable in CTA `cta` of this cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(cta));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait on a barrier that the other CTA of the pair arrives on; records `site` when it runs out.
__device__ __noinline__ bool wait_pair(uint32_t bar, uint32_t parity, int site, uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (global_ns() - t0 > limit_ns) {
      atomicCAS(&g_err_word, 0u, static_cast<unsigned>(site));
      return false;
    }
  }
  return true;
}
// Time-bounded wait that records `site` when it runs out (end-of-kernel drains).
__device__ __noinline__ void wait_drain_rec(uint32_t bar, uint32_t parity, int site) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicCAS(&g_err_word, 0u, static_cast<unsigned>(site));
      return;
    }
  }
}
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int x,
                                                 int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
// The pair's MMA and commit, issued by one elected lane of a warp whose lanes all
// make the call (see tc_mma_elect).  The commit arrives on the barrier at this
// shared offset in the CTAs of `mask` (bit r = rank r) once every MMA issued so
// far has completed.
__device__ __forceinline__ void tc_mma_pair_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair_elect(uint32_t bar, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(bar),
      "h"(mask)
      : "memory");
}
// Instruction descriptor of the pair: fp32 accumulator, bf16 A and B, K-major, M = 256, N = n.
__host__ __device__ constexpr uint32_t idesc_pair(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(256 >> 4) << 24);
}

template <int TN2>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, const Args a) {
  static_assert(TN2 == 256 || TN2 == 224 || TN2 == 192 || TN2 == 128, "pair tile widths");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int kStages = a.stages;
  constexpr int a_tile = kBM * kBK * 2;             // this CTA's 128 A rows of a k-tile
  constexpr int kStageBytes = a_tile + (TN2 / 2) * kBK * 2;  // + its TN2/2 B rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  unsigned char* tiles = smem + kBarBlock;
  // bars: full[16], empty[16], tfull[2], tempty[2], drain, sync; then the tensor-memory slot and the abort word
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kPairStagesMax;
  const uint32_t tfull0 = empty0 + 8 * kPairStagesMax;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain_bar = tempty0 + 16;
  const uint32_t sync_bar = drain_bar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kPairStagesMax + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int nclusters = static_cast<int>(gridDim.x >> 1);

  pdl_wait();  // nothing below overlaps the previous kernel
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full0 + 8 * i, 1);  // the even CTA's producer; bytes of both CTAs
      mbar_init(empty0 + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, 8);  // four epilogue warps in each CTA
    }
    mbar_init(drain_bar, 1);
    mbar_init(sync_bar, 1);  // phase 0: the other CTA's allocation is done; phase 1: it has finished
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
  }
  // Both CTAs' barriers are initialised before either addresses the other's.
  // Nothing above can block, and the two CTAs of a cluster run together.
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (warp == kMmaWarp) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kPairTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  bool pair_ok = true;
  if (threadIdx.x == 0) {
    // handshake 1: both CTAs hold the pair's tensor memory before the first MMA
    mbar_arrive_cluster(peer_addr(sync_bar, rank ^ 1u));
    pair_ok = wait_pair(sync_bar, 0, 30, a.wait_ns);
    uint32_t peer_base = 0;
    if (pair_ok) {
      asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(peer_base) : "r"(peer_addr(smem_u32(tmem_slot), rank ^ 1u))
                   : "memory");
      if (peer_base != *tmem_slot) {
        atomicCAS(&g_err_word, 0u, 31u);
        pair_ok = false;
      }
    }
    if (!pair_ok) *abort_flag = 1;
  }
  __syncthreads();
  const uint32_t tmem_base = *tmem_slot;
  const int m_tiles2 = (a.M + 255) / 256;
  // no work at all when the handshake failed (both CTAs fail it together or time out)
  const int units = *abort_flag ? 0 : m_tiles2 * a.n_tiles;

  if (warp < kProducerWarps) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t issued_mask = 0, issued_par = 0;
      const uint32_t full_leader0 = peer_addr(full0, 0);
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = cid; u < units && ok; u += nclusters) {
        const int nt = u / m_tiles2, mt2 = u % m_tiles2;
        const int arow = mt2 * 256 + static_cast<int>(rank) * kBM;
        const int brow = nt * TN2 + static_cast<int>(rank) * (TN2 / 2);
        for (int kb = 0; kb < a.kb_total; ++kb) {
          if (!wait_bounded(empty0 + 8 * st, ph ^ 1u, abort_flag, 21, a.wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(tiles + st * kStageBytes);
          if (leader) mbar_expect_tx(full0 + 8 * st, static_cast<uint32_t>(2 * kStageBytes));
          tma_load_2d_pair(sa, &tmA, full_leader0 + 8 * st, kb * kBK, arow);
          tma_load_2d_pair(sa + a_tile, &tmW, full_leader0 + 8 * st, kb * kBK, brow);
          issued_mask |= 1u << st;
          issued_par = (issued_par & ~(1u << st)) | (ph << st);
          if (++st == kStages) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      if (leader) {
        // the copies of both CTAs complete on these barriers
        for (int i = 0; i < kStages; ++i)
          if (issued_mask & (1u << i)) wait_drain_rec(full0 + 8 * i, (issued_par >> i) & 1u, 25);
      }
      // the even CTA's commits for the last use of each stage arrive in this
      // CTA's shared memory: let them land before the CTA may leave
      if (!*abort_flag)
        for (int i = 0; i < kStages; ++i)
          if (issued_mask & (1u << i)) wait_drain_rec(empty0 + 8 * i, (issued_par >> i) & 1u, 26);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    // The whole warp runs the loop and an elected lane issues (as in the one-SM
    // kernel); the warp goes on only if all lanes saw each barrier phase complete.
    if (leader) {
      auto wait_all = [&](uint32_t bar, uint32_t par, int site) -> bool {
        const bool r = wait_bounded(bar, par, abort_flag, site, a.wait_ns);
        return __all_sync(0xffffffffu, r);
      };
      const uint64_t desc0 = sw128_desc(smem_u32(tiles));
      constexpr uint32_t kIdesc = idesc_pair(TN2);
      int st = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      uint32_t acc_used = 0, acc_par = 0;  // accumulators committed, and the parity of their last commit
      bool ok = true;
      bool any = false;
      for (int u = cid; u < units && ok; u += nclusters) {
        if (!wait_all(tempty0 + 8 * acc, acc_ph ^ 1u, 22)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * TN2);
        for (int kb = 0; kb < a.kb_total; ++kb) {
          if (!wait_all(full0 + 8 * st, ph, 23)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = desc0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
          const uint64_t bdesc = adesc + static_cast<uint64_t>(a_tile >> 4);
#pragma unroll
          for (int k = 0; k < kBK / kUK; ++k)
            tc_mma_pair_elect(d0, adesc + static_cast<uint64_t>(2 * k), bdesc + static_cast<uint64_t>(2 * k), kIdesc,
                              (k > 0 || kb > 0) ? 1u : 0u);
          tc_commit_pair_elect(empty0 + 8 * st, 3);
          any = true;
          if (++st == kStages) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_elect(tfull0 + 8 * acc, 3);
        acc_used |= 1u << acc;
        acc_par = (acc_par & ~(1u << acc)) | (acc_ph << acc);
        if (++acc == 2) {
          acc = 0;
          acc_ph ^= 1u;
        }
      }
      const bool aborted = __any_sync(0xffffffffu, *abort_flag != 0);
      if (aborted && any) {
        tc_commit_pair_elect(drain_bar, 1);
        wait_drain(drain_bar, 0);
      }
      // both CTAs' epilogues release each accumulator on this CTA's tempty: let
      // their last arrivals land before this CTA may leave
      if (!aborted)
        for (int i = 0; i < 2; ++i)
          if (acc_used & (1u << i)) wait_drain_rec(tempty0 + 8 * i, (acc_par >> i) & 1u, 27);
    }
  } else {
    // ------------------------------------------------------------ epilogue (4 warps, both CTAs)
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t tempty_leader0 = peer_addr(tempty0, 0);
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int u = cid; u < units; u += nclusters) {
      const int nt = u / m_tiles2, mt2 = u % m_tiles2;
      if (!wait_bounded(tfull0 + 8 * acc, acc_ph, abort_flag, 24, a.wait_ns)) break;
      __syncwarp();  // lanes leave the wait at different times; tcgen05.ld needs the whole warp
      tc_fence_after();
      const int row = mt2 * 256 + static_cast<int>(rank) * kBM + row_in_tile;
      const bool row_ok = row < a.M;
      const uint32_t tbase = lane_base + acc * TN2;
#pragma unroll 1
      for (int ch = 0; ch < TN2 / 32; ++ch) {
        uint32_t r[32];
        tc_ld32(tbase + ch * 32, r);
        const int col0 = nt * TN2 + ch * 32;
        if (!row_ok || col0 >= a.N) continue;
        if (a.out_kind == kOutF32) {
          float* dst = static_cast<float*>(a.C) + static_cast<size_t>(row) * a.N + col0;
#pragma unroll
          for (int g = 0; g < 8; ++g)
            if (col0 + 4 * g < a.N)
              *reinterpret_cast<float4*>(dst + 4 * g) =
                  make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                              __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
        } else {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.C) + static_cast<size_t>(row) * a.N + col0;
          const __nv_bfloat16* res = a.R ? a.R + static_cast<size_t>(row) * a.N + col0 : nullptr;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            if (col0 + 8 * g >= a.N) break;
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(r[8 * g + e]);
            if (res) {
              float rv[8];
              unpack8(*reinterpret_cast<const uint4*>(res + 8 * g), rv);
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __fadd_rn(f[e], rv[e]);
            }
            *reinterpret_cast<uint4*>(dst + 8 * g) = pack8(f);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_ph ^= 1u;
      }
    }
  }

  // Teardown: every MMA has completed once this CTA's epilogue consumed the
  // last accumulator; handshake 2 keeps the pair's shared and tensor memory
  // alive until the other CTA is done with them.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && pair_ok) {
    mbar_arrive_cluster(peer_addr(sync_bar, rank ^ 1u));
    wait_pair(sync_bar, 1, 32, kWaitLimitNs);
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kPairTmemCols)
                 : "memory");
  }
}

// Second pass of split-K: element (i, j) of an unprotected tile is the
// left-to-right sum ((0 + P_0) + P_1) + ... of its split partials (+ residual),
// rounded once.  A thread owns four columns of one row; the partials are
// fetched four splits at a time so their loads are in flight together, and
// added in split order.
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, void* C, const __nv_bfloat16* __restrict__ R,
                                     const float* __restrict__ Rf, int M, int N, int splits, int skip_r0, int skip_r1,
                                     int out_kind) {
  pdl_wait();
  pdl_trigger();
  const int64_t chunks = static_cast<int64_t>(N) / 4;
  const int64_t n = static_cast<int64_t>(M) * chunks;
  const size_t plane = static_cast<size_t>(M) * N;
  for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < n;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(k / chunks);
    const int col = static_cast<int>(k % chunks) * 4;
    if (row >= skip_r0 && row < skip_r1) continue;
    const float* p = partial + static_cast<size_t>(row) * N + col;
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = 0;
    for (; s + 4 <= splits; s += 4) {
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __ldcs(reinterpret_cast<const float4*>(p + (s + j) * plane));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f.x = __fadd_rn(f.x, v[j].x); f.y = __fadd_rn(f.y, v[j].y);
        f.z = __fadd_rn(f.z, v[j].z); f.w = __fadd_rn(f.w, v[j].w);
      }
    }
    for (; s < splits; ++s) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(p + s * plane));
      f.x = __fadd_rn(f.x, v.x); f.y = __fadd_rn(f.y, v.y); f.z = __fadd_rn(f.z, v.z); f.w = __fadd_rn(f.w, v.w);
    }
    const size_t o = static_cast<size_t>(row) * N + col;
    if (out_kind == kOutF32) {
      if (Rf) {
        const float4 rv = *reinterpret_cast<const float4*>(Rf + o);
        f.x = __fadd_rn(f.x, rv.x); f.y = __fadd_rn(f.y, rv.y); f.z = __fadd_rn(f.z, rv.z); f.w = __fadd_rn(f.w, rv.w);
      }
      *reinterpret_cast<float4*>(static_cast<float*>(C) + o) = f;
    } else {
      if (R) {
        const uint2 rr = *reinterpret_cast<const uint2*>(R + o);
        f.x = __fadd_rn(f.x, bf16_lo(rr.x)); f.y = __fadd_rn(f.y, bf16_hi(rr.x));
        f.z = __fadd_rn(f.z, bf16_lo(rr.y)); f.w = __fadd_rn(f.w, bf16_hi(rr.y));
      }
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(C) + o) =
          make_uint2(pack_bf16x2(f.x, f.y), pack_bf16x2(f.z, f.w));
    }
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

struct MapKey {
  const void* ptr;
  int64_t rows, K;
  int box_rows;
  int kbs;  // 0: 2D map; >0: 3D [kblock][rows][64] view with boxes spanning kbs k-blocks
  int halves;  // 1: the matrix taken as two stacked [rows][K] halves, one box from each
  int dev;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && K == o.K && box_rows == o.box_rows && kbs == o.kbs &&
           halves == o.halves && dev == o.dev;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    size_t h = reinterpret_cast<size_t>(k.ptr);
    h ^= static_cast<size_t>(k.rows) * 0x9E3779B97F4A7C15ull;
    h ^= static_cast<size_t>(k.K) * 0xC2B2AE3D27D4EB4Full;
    h ^= static_cast<size_t>(k.box_rows * 131 + k.dev + k.kbs * 7919 + k.halves * 104729);
    return h;
  }
};

std::mutex g_map_mutex;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

// Tensor map of a [rows][K] bf16 row-major matrix, 128-byte swizzle, out-of-range
// elements read as zero.  2D (kbs == 0): box 64 (K) x box_rows.  3D (kbs > 0, K a
// multiple of 64): the matrix viewed as [K/64][rows][64] (k-block stride 128
// bytes), box 64 x box_rows x kbs, so one copy brings kbs consecutive k-blocks,
// each landing as its own swizzled box_rows x 128-byte tile.
// halves == 1: the matrix is [2][rows][K] (two stacked matrices) and every box
// takes box_rows rows of the first half followed by the same rows of the
// second, landing as one 2*box_rows-row tile (one more map dimension of extent
// 2 and stride rows*K elements).
bi_status tensor_map(const void* ptr, int64_t rows, int64_t K, int box_rows, int kbs, CUtensorMap* out,
                     int halves = 0) {
  int dev = 0;
  cudaGetDevice(&dev);
  MapKey key{ptr, rows, K, box_rows, kbs, halves, dev};
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *out = it->second;
      return BI_OK;
    }
  }
  auto fn = encode_fn();
  BI_REQUIRE(fn != nullptr, BI_ERR_CUDA, "bi_gemm: cuTensorMapEncodeTiled is not available from the driver");
  CUresult r;
  if (halves != 0) {
    const cuuint64_t half = static_cast<cuuint64_t>(rows) * K * 2;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(kbs == 0 ? K : kBK), static_cast<cuuint64_t>(rows), 2,
                          static_cast<cuuint64_t>(K / kBK)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(K) * 2, half, static_cast<cuuint64_t>(kBK) * 2};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows), 2,
                         static_cast<cuuint32_t>(kbs)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    r = fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kbs == 0 ? 3 : 4, const_cast<void*>(ptr), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else if (kbs == 0) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    r = fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kBK), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(K / kBK)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(kBK) * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows),
                         static_cast<cuuint32_t>(kbs)};
    cuuint32_t estr[3] = {1, 1, 1};
    r = fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  BI_REQUIRE(r == CUDA_SUCCESS, BI_ERR_CUDA, "bi_gemm: cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  std::lock_guard<std::mutex> lock(g_map_mutex);
  if (g_maps.size() > 4096) g_maps.clear();
  g_maps[key] = *out;
  return BI_OK;
}

// SM count used by the planner; with no device (workspace queries on a host
// without a GPU) it assumes 152.
int plan_sms() {
  const int n = num_sms();
  return n > 0 ? n : 152;
}

struct Plan {
  int TN;  // CTA tile width in columns: 32, 64, 128, 192 or 256
  int a_rows, kbs, map3d, stage_bytes, stages;
  int splits;
  int tm0, tm1, seq;
  int m_tiles, n_tiles, units, kb_total;
  int pair;  // 0: one-SM tiles; else the width of the SM-pair tiles (256 x pair)
};

// Clusters of two CTAs of the pair kernel that can be resident at once on the
// current device (cached per device); 76 when there is no device.
template <int TN2>
int pair_clusters_for() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 76;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= static_cast<int>(cache.size())) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    const void* fn = reinterpret_cast<const void*>(gemm_pair_kernel<TN2>);
    int n = 0;
    if (ensure_smem_limit(fn, kSmemLimit) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * 76);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kSmemLimit;
      if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
    }
    cache[dev] = n > 0 ? n : std::max(1, plan_sms() / 2);
  }
  return cache[dev];
}

int pair_clusters(int tn2) {
  if (num_sms() <= 0) return 76;
  switch (tn2) {
    case 256: return pair_clusters_for<256>();
    case 224: return pair_clusters_for<224>();
    case 192: return pair_clusters_for<192>();
    default: return pair_clusters_for<128>();
  }
}

// Relative time of one k-tile per CTA (one-SM tile of `tn` columns) or per CTA
// pair (256 x tn2 tile), as measured on GB300 for compute-sized GEMMs: the
// copy engines, not the tensor cores, set the pace of the narrower tiles.
double ktile_cost_single(int tn) { return tn >= 256 ? 645.0 : tn >= 128 ? 625.0 : tn >= 64 ? 500.0 : 450.0; }
double ktile_cost_pair(int tn2) { return tn2 >= 256 ? 540.0 : tn2 >= 224 ? 495.0 : tn2 >= 192 ? 470.0 : 420.0; }

// Part count of the K-only split (INVARIANT_KSPLIT): enough parts that a
// decode-sized GEMM (one 128-row tile, 256-column tiles) gives about one unit
// per SM of a 152-SM part, at least 4 k-tiles per part, at most kMaxSplitK.
// A constant target (not the device's SM count) keeps the bits the same on
// every device.
constexpr int kKsplitUnits = 152;
int ksplit_count(int64_t N, int64_t K) {
  const int64_t kb_total = (K + kBK - 1) / kBK;
  const int64_t tiles = (N + 4 * kBN - 1) / (4 * kBN);
  int64_t ks = std::max<int64_t>(1, kKsplitUnits / std::max<int64_t>(1, tiles));
  ks = std::min<int64_t>(ks, kMaxSplitK);
  ks = std::min<int64_t>(ks, std::max<int64_t>(1, kb_total / 4));
  return static_cast<int>(ks);
}

int choose_width(int64_t M, int64_t N, int max_tn) {
  const int sms = plan_sms();
  const int64_t mt = (M + kBM - 1) / kBM;
  double best = -1.0;
  int btn = 64;
  const int widths[3] = {256, 128, 64};
  const double penalty[3] = {1.0, 0.92, 0.80};  // operand bytes per flop grow as the tile narrows
  for (int i = 0; i < 3; ++i) {
    const int tn = widths[i];
    if (tn > max_tn) continue;
    const int64_t tiles = mt * ((N + tn - 1) / tn);
    const int64_t waves = (tiles + sms - 1) / sms;
    const double eff = static_cast<double>(tiles) / static_cast<double>(waves * sms) * penalty[i];
    if (eff > best + 1e-9) {
      best = eff;
      btn = tn;
    }
  }
  return btn;
}

// Decode-sized M (one 128-row tile): the GEMM streams the weights and every
// CTA also reads the whole A block of its K range, so take the width that
// minimises (waves of units) x (bytes a CTA reads per unit ~ TN + a_rows).
int choose_width_small_m(int64_t N, int splits, int a_rows) {
  const int sms = plan_sms();
  int btn = 64;
  int64_t best = INT64_MAX;
  for (int tn : {256, 192, 128, 64, 32}) {
    const int64_t units = ((N + tn - 1) / tn) * splits;
    const int64_t waves = (units + sms - 1) / sms;
    const int64_t cost = waves * (tn + a_rows);
    if (cost < best) {
      best = cost;
      btn = tn;
    }
  }
  return btn;
}

// Tuning of the non-invariant schedule (bi_fast_gemm_plan): per (M, N, K,
// planes), 1 = FAST takes the tile plan of INVARIANT (no split-K) instead of
// its own split-K rule.  A host-side table, set by a caller that has timed both.
std::mutex g_fast_mutex;
std::map<std::tuple<int64_t, int64_t, int64_t, int>, int> g_fast_plan;

int fast_plan_hint(int64_t M, int64_t N, int64_t K, int planes) {
  std::lock_guard<std::mutex> lock(g_fast_mutex);
  auto it = g_fast_plan.find(std::make_tuple(M, N, K, planes));
  return it == g_fast_plan.end() ? 0 : it->second;
}

// planes: 1 for bf16 A, 3 for fp32 A held as three bf16 planes (each plane
// adds an A box to every stage).
Plan make_plan(int64_t M, int64_t N, int64_t K, bi_mode mode, int64_t tb, int64_t te, int planes = 1,
               bool allow_pair = true) {
  Plan p;
  p.a_rows = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : kBM;
  p.m_tiles = static_cast<int>((M + kBM - 1) / kBM);
  p.kb_total = static_cast<int>((K + kBK - 1) / kBK);
  p.splits = 1;
  p.tm0 = p.tm1 = 0;
  p.seq = 1;
  // A protected target in the only m-tile makes the whole launch INVARIANT.
  if (mode == BI_MODE_PROTECTED && te > tb && p.m_tiles == 1) mode = BI_MODE_INVARIANT;
  // FAST tuned to the invariant tile plan for this shape
  if (mode == BI_MODE_FAST && fast_plan_hint(M, N, K, planes) == 1) mode = BI_MODE_INVARIANT;
  int max_tn = 256;
  if (mode == BI_MODE_INVARIANT_KSPLIT) {
    const int ks = ksplit_count(N, K);
    if (p.m_tiles == 1) {
      p.splits = ks;  // parts on separate CTAs, added by the second pass
    } else if (ks > 1) {
      p.tm0 = 0;      // every tile merged in its CTA
      p.tm1 = p.m_tiles;
      p.seq = ks;
      max_tn = 128;   // the running sum needs a third accumulator-sized buffer
    }
  }
  int fast_tn = 0;
  if (mode == BI_MODE_FAST || mode == BI_MODE_PROTECTED) {
    // FAST: split K when there are fewer tiles than SMs (the split count
    // follows M); PROTECTED: the target's tiles are not split.  Its tile is
    // the widest of 256/128/64 columns that still gives every SM a tile (else
    // 64), as a conventional GEMM picks it.
    fast_tn = 64;
    if (M <= kBM) {
      for (int tn : {256, 128, 64})
        if ((N + tn - 1) / tn >= plan_sms()) {
          fast_tn = tn;
          break;
        }
    } else {
      fast_tn = choose_width(M, N, 256);
    }
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * ((N + fast_tn - 1) / fast_tn);
    const int sms = plan_sms();
    int sk = static_cast<int>(std::min<int64_t>(kMaxSplitK, std::max<int64_t>(1, sms / std::max<int64_t>(1, tiles))));
    p.splits = std::max(1, std::min(sk, p.kb_total));
    if (mode == BI_MODE_PROTECTED && te > tb) {
      p.tm0 = static_cast<int>(tb / kBM);
      p.tm1 = static_cast<int>((te - 1) / kBM) + 1;
    }
  }
  if (fast_tn) p.TN = fast_tn;
  else p.TN = M <= kBM ? choose_width_small_m(N, p.splits, planes * p.a_rows) : choose_width(M, N, max_tn);
  p.pair = 0;
  if (mode == BI_MODE_INVARIANT && planes == 1 && M > kBM && allow_pair) {
    // SM-pair tiles when the model says they finish sooner than the one-SM tiles
    const int sms = plan_sms();
    const int64_t single_units = static_cast<int64_t>(p.m_tiles) * ((N + p.TN - 1) / p.TN);
    double best = static_cast<double>((single_units + sms - 1) / sms) * ktile_cost_single(p.TN);
    for (int tn2 : {256, 224, 192, 128}) {
      const int64_t units = ((M + 255) / 256) * ((N + tn2 - 1) / tn2);
      const int cl = pair_clusters(tn2);
      const double t = static_cast<double>((units + cl - 1) / cl) * ktile_cost_pair(tn2);
      if (t < best * 0.97) {
        best = t;
        p.pair = tn2;
      }
    }
  }
  if (p.pair) {
    p.TN = p.pair;
    p.a_rows = kBM;
    p.kbs = 1;
    p.map3d = 0;
    p.stage_bytes = kBM * kBK * 2 + (p.pair / 2) * kBK * 2;
    p.stages = std::min(kPairStagesMax, (kSmemLimit - 1024 - kBarBlock) / p.stage_bytes);
    p.n_tiles = static_cast<int>((N + p.pair - 1) / p.pair);
    p.units = static_cast<int>(((M + 255) / 256) * p.n_tiles);
    return p;
  }
  // Each stage costs the copy engine and the barrier round trip a roughly fixed
  // time, so at decode sizes a stage spans several k-blocks (one 3D box per
  // operand, up to 8 k-blocks), but it also waits for its whole stage before the
  // MMAs start, so the ring keeps at least three stages.  Measured on GB300,
  // 64x4096x12288: 4 k-blocks x 4 stages (48 KiB each) 31.0 us against 8 x 2
  // (96 KiB) 33.7 us; 1x4096x12288: 8 x 4 (48 KiB) 27.0 us against 4 x 8 31.0 us
  // and 2 k-blocks per stage 42 us at either size.  (A 3D copy costs more than a
  // 2D box of the same bytes, so the 3D view is used only when a copy spans
  // several k-blocks.)
  p.kbs = (K % kBK == 0 && M <= kBM) ? std::min(8, std::max(1, 256 / p.TN)) : 1;
  const int budget = kSmemLimit - 1024 - kBarBlock - (p.a_rows < kBM ? kOverreadSlack : 0);
  const int kblock_bytes = (planes * p.a_rows + p.TN) * kBK * 2;
  const int min_stages = 3;
  while (p.kbs > 1 && budget / (p.kbs * kblock_bytes) < min_stages) p.kbs /= 2;
  p.map3d = p.kbs > 1 ? 1 : 0;
  p.stage_bytes = p.kbs * kblock_bytes;
  p.stages = std::min(kMaxStages, budget / p.stage_bytes);
  p.n_tiles = static_cast<int>((N + p.TN - 1) / p.TN);
  const int prot = p.tm1 - p.tm0;
  p.units = p.n_tiles * (prot + (p.m_tiles - prot) * p.splits);
  return p;
}

template <int TN2>
bi_status launch_pair(const CUtensorMap& ma, const CUtensorMap& mw, const Args& args, cudaStream_t s) {
  const void* fn = reinterpret_cast<const void*>(gemm_pair_kernel<TN2>);
  BI_CUDA_TRY(ensure_smem_limit(fn, kSmemLimit));
  const size_t smem = 1024 + kBarBlock + static_cast<size_t>(args.stages) * args.stage_bytes;
  const int grid = 2 * std::min(args.units, pair_clusters(TN2));
  // no programmatic serialisation: the pair kernel starts after its predecessor has finished
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  BI_TIMED(::bi::kTagGemm, s, BI_PDL_CHECK(cudaLaunchKernelEx(&cfg, gemm_pair_kernel<TN2>, ma, mw, args)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

template <int TN, int PL>
bi_status launch_w(const CUtensorMap& ma, const CUtensorMap& mw, const Args& args, cudaStream_t s) {
  BI_CUDA_TRY(ensure_smem_limit(reinterpret_cast<const void*>(gemm_tc_kernel<TN, PL>), kSmemLimit));
  const size_t smem = smem_bytes(args.stages, args.stage_bytes, args.a_rows);
  const int grid = std::min(args.units, num_sms());
  BI_TIMED(::bi::kTagGemm, s, BI_PDL_CHECK(launch_pdl(gemm_tc_kernel<TN, PL>, dim3(grid), dim3(kThreadsTc), smem, s, ma, mw, args)));
  BI_LAUNCH_CHECK();
  return BI_OK;
}

}  // namespace gemm

int take_gemm_device_error(cudaStream_t s, int32_t* code) {
  unsigned v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, gemm::g_err_word, sizeof(v), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return 1;
  if (cudaStreamSynchronize(s) != cudaSuccess) return 1;
  if (v != 0) {
    unsigned zero = 0;
    if (cudaMemcpyToSymbolAsync(gemm::g_err_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return 1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return 1;
  }
  *code = static_cast<int32_t>(v);
  return 0;
}

size_t gemm_ws(int64_t M, int64_t N, int64_t K, bi_mode mode, int planes) {
  if (mode == BI_MODE_INVARIANT || M <= 0 || N <= 0 || K <= 0) return 0;
  // PROTECTED: the largest need with or without a target
  int splits = gemm::make_plan(M, N, K, mode, 0, 0, planes).splits;
  if (mode == BI_MODE_PROTECTED) splits = std::max(splits, gemm::make_plan(M, N, K, mode, 0, 1, planes).splits);
  if (splits <= 1) return 0;
  return static_cast<size_t>(splits) * M * N * sizeof(float);
}

size_t gemm_ws(int64_t M, int64_t N, int64_t K, bi_mode mode) { return gemm_ws(M, N, K, mode, 1); }

namespace {

// Test hook state (bi_debug_arm_gemm_stall): the next GEMM launch of this host
// thread drops its first stage's copies in CTA 0 and uses a short wait limit.
thread_local unsigned long long t_stall_wait_ns = 0;

// Shared body of the bf16-A and fp32-A (planes) GEMMs.  A: [M][K] bf16, or
// three bf16 planes [3][M][K] when planes == 3.  R: bf16 residual (bf16 out);
// Rf: fp32 residual (fp32 out).
bi_status gemm_core(const void* A, int planes, const void* Wt, void* C, const void* R, const float* Rf, int64_t M,
                    int64_t N, int64_t K, bi_dtype out_dtype, bi_mode mode, int32_t target_row,
                    int32_t target_count, void* ws, size_t ws_bytes, cudaStream_t s, bool weights_constant) {
  BI_REQUIRE(M >= 0 && N >= 0 && K >= 8, BI_ERR_INVALID_ARG, "bi_gemm: M=%lld N=%lld K=%lld",
             static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K));
  BI_REQUIRE(K % 8 == 0 && N % 8 == 0, BI_ERR_UNSUPPORTED, "bi_gemm: K (%lld) and N (%lld) must be multiples of 8",
             static_cast<long long>(K), static_cast<long long>(N));
  BI_REQUIRE(planes * M < (int64_t(1) << 31) && N < (int64_t(1) << 31) && K < (int64_t(1) << 31), BI_ERR_UNSUPPORTED,
             "bi_gemm: sizes beyond int32");
  BI_REQUIRE(out_dtype == BI_BF16 || out_dtype == BI_F32, BI_ERR_UNSUPPORTED, "bi_gemm: out dtype %d",
             static_cast<int>(out_dtype));
  BI_REQUIRE(mode_valid(mode), BI_ERR_INVALID_ARG, "bi_gemm: mode %d",
             static_cast<int>(mode));
  BI_REQUIRE(R == nullptr || out_dtype == BI_BF16, BI_ERR_UNSUPPORTED, "bi_gemm: residual needs bf16 output");
  BI_REQUIRE(Rf == nullptr || out_dtype == BI_F32, BI_ERR_UNSUPPORTED, "bi_gemm: fp32 residual needs fp32 output");
  int64_t tb = 0, te = 0;
  if (mode == BI_MODE_PROTECTED && target_row >= 0) {
    BI_REQUIRE(target_count >= 1 && target_row + static_cast<int64_t>(target_count) <= M, BI_ERR_INVALID_ARG,
               "bi_gemm: target rows [%d, %d) outside [0, %lld)", target_row, target_row + target_count,
               static_cast<long long>(M));
    tb = target_row;
    te = target_row + static_cast<int64_t>(target_count);
  }
  if (M == 0 || N == 0) return BI_OK;
  BI_REQUIRE(A && Wt && C, BI_ERR_INVALID_ARG, "bi_gemm: null pointer");
  BI_REQUIRE(aligned16(A) && aligned16(Wt) && aligned16(C) && (R == nullptr || aligned16(R)) &&
                 (Rf == nullptr || aligned16(Rf)),
             BI_ERR_INVALID_ARG, "bi_gemm: pointers must be 16-byte aligned");
  // the stall test hook exists in the one-SM kernel only
  gemm::Plan p = gemm::make_plan(M, N, K, mode, tb, te, planes, t_stall_wait_ns == 0);
  BI_REQUIRE(p.seq == 1 || p.TN <= 128, BI_ERR_UNSUPPORTED, "bi_gemm: internal plan error (merged units at width %d)",
             p.TN);
  BI_REQUIRE(p.stages >= 2, BI_ERR_UNSUPPORTED, "bi_gemm: internal plan error (%d stages)", p.stages);
  gemm::Args args{};
  args.M = static_cast<int>(M);
  args.a_rows = p.a_rows;
  args.m64 = M <= 64 ? 1 : 0;
  args.kbs = p.kbs;
  args.map3d = p.map3d;
  args.stage_bytes = p.stage_bytes;
  args.stages = p.stages;
  args.N = static_cast<int>(N);
  args.K = static_cast<int>(K);
  args.m_tiles = p.m_tiles;
  args.n_tiles = p.n_tiles;
  args.splits = p.splits;
  args.tm0 = p.tm0;
  args.tm1 = p.tm1;
  args.seq = p.seq;
  args.prefetch_w = weights_constant ? 1 : 0;
  args.units = p.units;
  args.kb_total = p.kb_total;
  args.C = C;
  args.R = static_cast<const __nv_bfloat16*>(R);
  args.Rf = Rf;
  args.plane_rows = static_cast<int>(M);
  args.out_kind = out_dtype == BI_F32 ? gemm::kOutF32 : gemm::kOutBF16;
  args.partial = nullptr;
  args.wait_ns = gemm::kWaitLimitNs;
  args.drop_first_stage = 0;
  if (t_stall_wait_ns != 0) {
    args.wait_ns = t_stall_wait_ns;
    args.drop_first_stage = 1;
    args.prefetch_w = 0;
    t_stall_wait_ns = 0;
  }
  if (p.splits > 1) {
    const size_t need = static_cast<size_t>(p.splits) * M * N * sizeof(float);
    BI_REQUIRE(ws != nullptr && ws_bytes >= need && aligned16(ws), BI_ERR_WORKSPACE,
               "bi_gemm: workspace %zu < %zu bytes", ws_bytes, need);
    args.partial = static_cast<float*>(ws);
  }
  CUtensorMap ma, mw;
  if (p.pair) {
    BI_TRY(gemm::tensor_map(A, M, K, gemm::kBM, 0, &ma));
    BI_TRY(gemm::tensor_map(Wt, N, K, p.pair / 2, 0, &mw));
    switch (p.pair) {
      case 256: return gemm::launch_pair<256>(ma, mw, args, s);
      case 224: return gemm::launch_pair<224>(ma, mw, args, s);
      case 192: return gemm::launch_pair<192>(ma, mw, args, s);
      default: return gemm::launch_pair<128>(ma, mw, args, s);
    }
  }
  // the planes form one [planes*M][K] matrix; plane p's rows start at p*M
  BI_TRY(gemm::tensor_map(A, planes * M, K, p.a_rows, p.map3d ? p.kbs : 0, &ma));
  BI_TRY(gemm::tensor_map(Wt, N, K, p.TN, p.map3d ? p.kbs : 0, &mw));
  bi_status st;
  if (planes == 1) {
    if (p.TN == 256) st = gemm::launch_w<256, 1>(ma, mw, args, s);
    else if (p.TN == 192) st = gemm::launch_w<192, 1>(ma, mw, args, s);
    else if (p.TN == 128) st = gemm::launch_w<128, 1>(ma, mw, args, s);
    else if (p.TN == 64) st = gemm::launch_w<64, 1>(ma, mw, args, s);
    else st = gemm::launch_w<32, 1>(ma, mw, args, s);
  } else {
    if (p.TN == 256) st = gemm::launch_w<256, 3>(ma, mw, args, s);
    else if (p.TN == 192) st = gemm::launch_w<192, 3>(ma, mw, args, s);
    else if (p.TN == 128) st = gemm::launch_w<128, 3>(ma, mw, args, s);
    else if (p.TN == 64) st = gemm::launch_w<64, 3>(ma, mw, args, s);
    else st = gemm::launch_w<32, 3>(ma, mw, args, s);
  }
  if (st != BI_OK) return st;
  if (p.splits > 1) {
    const int64_t n = M * (N / 4);
    const int64_t grid = std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(num_sms()) * 8);
    const int skip0 = p.tm0 * gemm::kBM, skip1 = static_cast<int>(std::min<int64_t>(M, int64_t(p.tm1) * gemm::kBM));
    BI_TIMED(::bi::kTagSplitkReduce, s, BI_PDL_CHECK(launch_pdl(gemm::splitk_reduce_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, args.partial, C, args.R, args.Rf, args.M, args.N,
                                                                          p.splits, skip0, skip1, args.out_kind)));
    BI_LAUNCH_CHECK();
  }
  return BI_OK;
}

// fp32 [rows][cols] -> three bf16 planes [3][rows][cols] (cols % 4 == 0).
__global__ void split_planes_kernel(const float* __restrict__ x, uint16_t* __restrict__ y, int64_t n4, size_t plane) {
  pdl_wait();
  pdl_trigger();
  for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < n4;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = *reinterpret_cast<const float4*>(x + 4 * k);
    store_planes4(y + 4 * k, plane, v.x, v.y, v.z, v.w);
  }
}

size_t planes_bytes(int64_t M, int64_t K) { return align_up(static_cast<size_t>(3) * M * K * 2, 256); }

}  // namespace

bi_status gemm_impl(const void* A, const void* Wt, void* C, const void* R, int64_t M, int64_t N, int64_t K,
                    bi_dtype out_dtype, bi_mode mode, int32_t target_row, int32_t target_count, void* ws,
                    size_t ws_bytes, cudaStream_t s, bool weights_constant) {
  clear_error();
  return gemm_core(A, 1, Wt, C, R, nullptr, M, N, K, out_dtype, mode, target_row, target_count, ws, ws_bytes, s,
                   weights_constant);
}

bi_status swiglu_impl(const void* gu, void* out, int64_t T, int64_t F, cudaStream_t s);  // pointwise.cu

// Gate|up GEMM with SwiGLU in its epilogue: act[M][F] = swiglu(A Wgu^T) for Wgu
// [2F][K] (gate rows then up rows).  Runs only where the plan of the plain
// [M][2F] GEMM is one-SM tiles, one split, one unit per tile and a tile width
// that is a multiple of 64; then every product is the plain GEMM's own (the
// same per-element k order) and the output equals that GEMM followed by the
// SwiGLU kernel, bit for bit.  *used says whether it ran; when it is false
// nothing was launched and the caller runs the two kernels.
bi_status gemm_swiglu_impl(const void* A, const void* Wgu, void* act, int64_t M, int64_t F, int64_t K, bi_mode mode,
                           int32_t target_row, int32_t target_count, cudaStream_t s, bool* used,
                           bool weights_constant) {
  *used = false;
  if (M <= 0 || F <= 0 || K < 8 || K % 8 != 0 || F % 8 != 0 || M > gemm::kBM || t_stall_wait_ns != 0) return BI_OK;
  if (!mode_valid(mode) || M >= (int64_t(1) << 31) || 2 * F >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return BI_OK;
  if (!aligned16(A) || !aligned16(Wgu) || !aligned16(act)) return BI_OK;
  int64_t tb = 0, te = 0;
  if (mode == BI_MODE_PROTECTED && target_row >= 0) {
    if (target_count < 1 || target_row + static_cast<int64_t>(target_count) > M) return BI_OK;
    tb = target_row;
    te = target_row + static_cast<int64_t>(target_count);
  }
  const gemm::Plan p = gemm::make_plan(M, 2 * F, K, mode, tb, te, 1, true);
  if (p.pair || p.splits != 1 || p.seq != 1 || p.TN % 64 != 0 || p.stages < 2) return BI_OK;
  gemm::Args args{};
  args.M = static_cast<int>(M);
  args.a_rows = p.a_rows;
  args.m64 = M <= 64 ? 1 : 0;
  args.kbs = p.kbs;
  args.map3d = p.map3d;
  args.stage_bytes = p.stage_bytes;
  args.stages = p.stages;
  args.N = static_cast<int>(2 * F);
  args.K = static_cast<int>(K);
  args.m_tiles = p.m_tiles;
  args.n_tiles = p.n_tiles;
  args.splits = 1;
  args.tm0 = p.tm0;
  args.tm1 = p.tm1;
  args.seq = 1;
  args.prefetch_w = weights_constant ? 1 : 0;
  args.units = p.units;
  args.kb_total = p.kb_total;
  args.plane_rows = static_cast<int>(M);
  args.out_kind = gemm::kOutBF16;
  args.swiglu = 1;
  args.F = static_cast<int>(F);
  args.act = static_cast<__nv_bfloat16*>(act);
  args.wait_ns = gemm::kWaitLimitNs;
  CUtensorMap ma, mw;
  BI_TRY(gemm::tensor_map(A, M, K, p.a_rows, p.map3d ? p.kbs : 0, &ma));
  BI_TRY(gemm::tensor_map(Wgu, F, K, p.TN / 2, p.map3d ? p.kbs : 0, &mw, 1));
  bi_status st;
  if (p.TN == 256) st = gemm::launch_w<256, 1>(ma, mw, args, s);
  else if (p.TN == 192) st = gemm::launch_w<192, 1>(ma, mw, args, s);
  else if (p.TN == 128) st = gemm::launch_w<128, 1>(ma, mw, args, s);
  else st = gemm::launch_w<64, 1>(ma, mw, args, s);
  if (st == BI_OK) *used = true;
  return st;
}

// fp32-activation layers: A already split into three bf16 planes [3][M][K] by
// the kernel that produced it; fp32 output, optional fp32 residual.
bi_status gemm_planes_impl(const void* A_planes, const void* Wt, float* C, const float* Rf, int64_t M, int64_t N,
                           int64_t K, bi_mode mode, int32_t target_row, int32_t target_count, void* ws,
                           size_t ws_bytes, cudaStream_t s, bool weights_constant) {
  return gemm_core(A_planes, 3, Wt, C, nullptr, Rf, M, N, K, BI_F32, mode, target_row, target_count, ws, ws_bytes, s,
                   weights_constant);
}

size_t gemm_f32a_ws(int64_t M, int64_t N, int64_t K, bi_mode mode) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return planes_bytes(M, K) + gemm_ws(M, N, K, mode, 3);
}

bi_status gemm_f32a_impl(const float* A, const void* Wt, float* C, const float* Rf, int64_t M, int64_t N, int64_t K,
                         bi_mode mode, int32_t target_row, int32_t target_count, void* ws, size_t ws_bytes,
                         cudaStream_t s) {
  clear_error();
  BI_REQUIRE(M >= 0 && N >= 0 && K >= 8 && K % 8 == 0, BI_ERR_INVALID_ARG, "bi_gemm_f32a: M=%lld N=%lld K=%lld",
             static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K));
  BI_REQUIRE(mode_valid(mode), BI_ERR_INVALID_ARG, "bi_gemm_f32a: mode %d", static_cast<int>(mode));
  if (M == 0 || N == 0) return BI_OK;
  BI_REQUIRE(A && aligned16(A), BI_ERR_INVALID_ARG, "bi_gemm_f32a: null or misaligned A");
  const size_t pb = planes_bytes(M, K);
  BI_REQUIRE(ws != nullptr && aligned16(ws) && ws_bytes >= gemm_f32a_ws(M, N, K, mode), BI_ERR_WORKSPACE,
             "bi_gemm_f32a: workspace %zu < %zu bytes", ws_bytes, gemm_f32a_ws(M, N, K, mode));
  uint16_t* planes = static_cast<uint16_t*>(ws);
  const int64_t n4 = M * K / 4;
  const int64_t grid = std::min<int64_t>((n4 + 255) / 256, static_cast<int64_t>(num_sms()) * 8);
  BI_TIMED(::bi::kTagSplitPlanes, s, BI_PDL_CHECK(launch_pdl(split_planes_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, A, planes, n4, static_cast<size_t>(M * K))));
  BI_LAUNCH_CHECK();
  return gemm_core(planes, 3, Wt, C, nullptr, Rf, M, N, K, BI_F32, mode, target_row, target_count,
                   static_cast<char*>(ws) + pb, ws_bytes - pb, s, false);
}

}  // namespace bi

extern "C" size_t bi_gemm_workspace(int64_t M, int64_t N, int64_t K, bi_mode mode) {
  return bi::gemm_ws(M, N, K, mode);
}

extern "C" size_t bi_gemm_f32a_workspace(int64_t M, int64_t N, int64_t K, bi_mode mode) {
  return bi::gemm_f32a_ws(M, N, K, mode);
}

extern "C" bi_status bi_gemm_f32a(const float* A, const void* W, float* C, const float* residual, int64_t M,
                                  int64_t N, int64_t K, bi_mode mode, int32_t target_row, int32_t target_count,
                                  void* workspace, size_t ws_bytes, bi_stream s) {
  return bi::gemm_f32a_impl(A, W, C, residual, M, N, K, mode, target_row, target_count, workspace, ws_bytes,
                            reinterpret_cast<cudaStream_t>(s));
}

extern "C" bi_status bi_fast_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t plan) {
  bi::clear_error();
  BI_REQUIRE(M > 0 && N > 0 && K > 0 && (plan == 0 || plan == 1), BI_ERR_INVALID_ARG,
             "bi_fast_gemm_plan: M=%lld N=%lld K=%lld plan=%d", static_cast<long long>(M), static_cast<long long>(N),
             static_cast<long long>(K), plan);
  std::lock_guard<std::mutex> lock(bi::gemm::g_fast_mutex);
  for (int planes : {1, 3}) {
    const auto key = std::make_tuple(M, N, K, planes);
    if (plan == 0) bi::gemm::g_fast_plan.erase(key);
    else bi::gemm::g_fast_plan[key] = plan;
  }
  return BI_OK;
}

extern "C" bi_status bi_debug_arm_gemm_stall(int64_t wait_ns) {
  bi::clear_error();
  BI_REQUIRE(wait_ns >= 1000000 && wait_ns <= 2000000000, BI_ERR_INVALID_ARG,
             "bi_debug_arm_gemm_stall: wait limit %lld ns outside [1e6, 2e9]", static_cast<long long>(wait_ns));
  bi::t_stall_wait_ns = static_cast<unsigned long long>(wait_ns);
  return BI_OK;
}

extern "C" int32_t bi_gemm_ksplit(int64_t N, int64_t K) {
  if (N <= 0 || K <= 0) return 1;
  return bi::gemm::ksplit_count(N, K);
}

extern "C" bi_status bi_gemm(const void* A, const void* W, void* C, const void* residual, int64_t M, int64_t N,
                             int64_t K, bi_dtype out_dtype, bi_mode mode, int32_t target_row, int32_t target_count,
                             void* workspace, size_t ws_bytes, bi_stream s) {
  return bi::gemm_impl(A, W, C, residual, M, N, K, out_dtype, mode, target_row, target_count, workspace, ws_bytes,
                       reinterpret_cast<cudaStream_t>(s), false);
}

extern "C" size_t bi_gemm_swiglu_workspace(int64_t M, int64_t F, int64_t K, bi_mode mode) {
  if (M <= 0 || F <= 0 || K <= 0) return 0;
  return bi::align_up(static_cast<size_t>(M) * 2 * F * 2, 256) + bi::gemm_ws(M, 2 * F, K, mode);
}

extern "C" bi_status bi_gemm_swiglu(const void* A, const void* W_gate_up, void* act, int64_t M, int64_t F, int64_t K,
                                    bi_mode mode, int32_t target_row, int32_t target_count, void* workspace,
                                    size_t ws_bytes, bi_stream s) {
  bi::clear_error();
  BI_REQUIRE(M >= 0 && F >= 0 && K >= 8, BI_ERR_INVALID_ARG, "bi_gemm_swiglu: M=%lld F=%lld K=%lld",
             static_cast<long long>(M), static_cast<long long>(F), static_cast<long long>(K));
  BI_REQUIRE(K % 8 == 0 && F % 8 == 0, BI_ERR_UNSUPPORTED, "bi_gemm_swiglu: K (%lld) and F (%lld) must be multiples of 8",
             static_cast<long long>(K), static_cast<long long>(F));
  BI_REQUIRE(bi::mode_valid(mode), BI_ERR_INVALID_ARG, "bi_gemm_swiglu: mode %d", static_cast<int>(mode));
  if (mode == BI_MODE_PROTECTED && target_row >= 0)
    BI_REQUIRE(target_count >= 1 && target_row + static_cast<int64_t>(target_count) <= M, BI_ERR_INVALID_ARG,
               "bi_gemm_swiglu: target rows [%d, %d) outside [0, %lld)", target_row, target_row + target_count,
               static_cast<long long>(M));
  if (M == 0 || F == 0) return BI_OK;
  BI_REQUIRE(A && W_gate_up && act, BI_ERR_INVALID_ARG, "bi_gemm_swiglu: null pointer");
  BI_REQUIRE(bi::aligned16(A) && bi::aligned16(W_gate_up) && bi::aligned16(act), BI_ERR_INVALID_ARG,
             "bi_gemm_swiglu: pointers must be 16-byte aligned");
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  bool used = false;
  BI_TRY(bi::gemm_swiglu_impl(A, W_gate_up, act, M, F, K, mode, target_row, target_count, st, &used, false));
  if (used) return BI_OK;
  const size_t gu_bytes = bi::align_up(static_cast<size_t>(M) * 2 * F * 2, 256);
  const size_t need = bi_gemm_swiglu_workspace(M, F, K, mode);
  BI_REQUIRE(workspace != nullptr && bi::aligned16(workspace) && ws_bytes >= need, BI_ERR_WORKSPACE,
             "bi_gemm_swiglu: workspace %zu < %zu bytes", ws_bytes, need);
  void* gu = workspace;
  void* sub = static_cast<char*>(workspace) + gu_bytes;
  BI_TRY(bi::gemm_impl(A, W_gate_up, gu, nullptr, M, 2 * F, K, BI_BF16, mode, target_row, target_count,
                       ws_bytes > gu_bytes ? sub : nullptr, ws_bytes - gu_bytes, st, false));
  return bi::swiglu_impl(gu, act, M, F, st);
}
