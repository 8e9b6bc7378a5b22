// Shared host/device helpers of libbi.  Compiled for sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <string>
#include <utility>

#include "../../include/bi.h"

namespace bi {

// ------------------------------------------------------------------ host-side error reporting
void set_error(const char* fmt, ...);
void clear_error();
int num_sms();  // SM count of the current device (cached per device)
// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device); thread-safe.
cudaError_t ensure_smem_limit(const void* kernel, int bytes);
// Resident CTAs per SM of `kernel` at `threads` threads and `smem` bytes of
// dynamic shared memory on the current device (after ensure_smem_limit),
// cached per (kernel, device); 1 if the query fails.
int occupancy_per_sm(const void* kernel, int threads, size_t smem);

#define BI_REQUIRE(cond, code, ...)     \
  do {                                  \
    if (!(cond)) {                      \
      ::bi::set_error(__VA_ARGS__);     \
      return code;                      \
    }                                   \
  } while (0)

#define BI_CUDA_TRY(expr)                                                                        \
  do {                                                                                           \
    cudaError_t e_ = (expr);                                                                     \
    if (e_ != cudaSuccess) {                                                                     \
      ::bi::set_error("%s failed: %s (%s:%d)", #expr, cudaGetErrorString(e_), __FILE__, __LINE__); \
      return BI_ERR_CUDA;                                                                        \
    }                                                                                            \
  } while (0)

#define BI_LAUNCH_CHECK()                                                                        \
  do {                                                                                           \
    cudaError_t e_ = cudaGetLastError();                                                         \
    if (e_ != cudaSuccess) {                                                                     \
      ::bi::set_error("kernel launch failed: %s (%s:%d)", cudaGetErrorString(e_), __FILE__, __LINE__); \
      return BI_ERR_CUDA;                                                                        \
    }                                                                                            \
  } while (0)

#define BI_TRY(expr)              \
  do {                            \
    bi_status st_ = (expr);       \
    if (st_ != BI_OK) return st_; \
  } while (0)

// Kernel tags of the optional launch timer (names in api.cu, same order).
enum KernelTag : int {
  kTagRmsnorm = 0,
  kTagRmsnormSplit,
  kTagGemm,
  kTagSplitkReduce,
  kTagAttnPlan,
  kTagAttnDecodeSplit,
  kTagAttnDecodeMerge,
  kTagAttnPrefillSplit,
  kTagAttnPrefillMerge,
  kTagQkvRope,
  kTagSwiglu,
  kTagEmbed,
  kTagTopk,
  kTagBatchIndex,
  kTagGather,
  kTagRopeTable,
  kTagSplitPlanes,
  kTagCount
};
extern volatile int g_profiling;
int prof_begin(int tag, cudaStream_t s);  // -1 when not recording
void prof_end(int slot, cudaStream_t s);

// Launch a kernel, bracketed by timing events when the launch timer is on.
#define BI_TIMED(tag, stream, ...)                                            \
  do {                                                                        \
    const int prof_slot_ = ::bi::g_profiling ? ::bi::prof_begin((tag), (stream)) : -1; \
    __VA_ARGS__;                                                              \
    if (prof_slot_ >= 0) ::bi::prof_end(prof_slot_, (stream));                \
  } while (0)

// Programmatic dependent launch: every library kernel is launched with
// programmatic stream serialisation, so it may start while its predecessor in
// the stream is still running.  Each kernel calls pdl_wait() before it reads
// or writes memory that the predecessor touches (griddepcontrol.wait returns
// once the predecessor grid has completed and its writes are visible), and
// pdl_trigger() to let its own successor start launching early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launch errors surface through cudaGetLastError (checked by BI_LAUNCH_CHECK).
#define BI_PDL_CHECK(expr) (void)(expr)

// Modes whose reduction geometry never depends on the batch.
inline bool mode_invariant(bi_mode m) { return m == BI_MODE_INVARIANT || m == BI_MODE_INVARIANT_KSPLIT; }
inline bool mode_valid(bi_mode m) { return m >= BI_MODE_INVARIANT && m <= BI_MODE_INVARIANT_KSPLIT; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Bump allocator over a caller-owned workspace (host-side bookkeeping only).
struct WsCarver {
  char* base;
  size_t cap;
  size_t used = 0;
  WsCarver(void* b, size_t c) : base(static_cast<char*>(b)), cap(c) {}
  template <typename T>
  T* take(size_t count) {
    used = align_up(used, 256);
    T* p = reinterpret_cast<T*>(base ? base + used : nullptr);
    used += count * sizeof(T);
    return p;
  }
  bool ok() const { return used <= cap; }
};

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// fp32 -> bf16 with round-to-nearest-even (the hardware conversion).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint16_t to_bf16_bits(float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
  f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
  f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

// SwiGLU of one (gate, up) pair: silu(g) * u = g / (1 + e^-g) * u, each
// operation rounded once (the one definition the SwiGLU kernels and the
// gate|up GEMM's fused epilogue share, so both give the same bits).
__device__ __forceinline__ float swiglu1(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// ------------------------------------------------------------------ fp32 activations as three bf16 planes
// An fp32 value a is the sum hi + mid + lo of three bf16 values, hi = bf16(a),
// mid = bf16(a - hi), lo = a - hi - mid: each fp32 difference is exact (it only
// removes leading significant bits), and the last remainder has at most 8
// significant bits, so it is a bf16 value itself whenever it stays in bf16's
// normal range (|a| >= 2^-110; below that it is rounded to 2^-133).  An fp32
// activation tensor [rows][cols] that feeds a GEMM is stored as three bf16
// planes [3][rows][cols]; a bf16 x bf16 product is exact in fp32, so the GEMM
// over the planes with fp32 accumulation multiplies the fp32 activations by
// the bf16 weights without rounding the activations.
__device__ __forceinline__ void split3(float a, float& hi, float& mid, float& lo) {
  hi = __bfloat162float(__float2bfloat16_rn(a));
  const float r = __fsub_rn(a, hi);
  mid = __bfloat162float(__float2bfloat16_rn(r));
  lo = __fsub_rn(r, mid);
}

// Four consecutive values into the three planes at p, p + plane, p + 2 plane
// (p 8-byte aligned).
__device__ __forceinline__ void store_planes4(uint16_t* p, size_t plane, float a, float b, float c, float d) {
  float h[4], m[4], l[4];
  split3(a, h[0], m[0], l[0]);
  split3(b, h[1], m[1], l[1]);
  split3(c, h[2], m[2], l[2]);
  split3(d, h[3], m[3], l[3]);
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]));
  *reinterpret_cast<uint2*>(p + plane) = make_uint2(pack_bf16x2(m[0], m[1]), pack_bf16x2(m[2], m[3]));
  *reinterpret_cast<uint2*>(p + 2 * plane) = make_uint2(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]));
}

// Where a producing kernel writes activations: bf16, fp32, or fp32 as three
// bf16 planes (`plane` elements apart) for a GEMM that consumes them.
enum ActKind : int { kActBF16 = 0, kActF32 = 1, kActPlanes = 2 };
struct ActDst {
  void* p;
  size_t plane;  // elements between planes (kActPlanes)
  int kind;
};

// Four consecutive values at element offset off (a multiple of 4).
__device__ __forceinline__ void act_store4(const ActDst& d, size_t off, float a, float b, float c, float e) {
  if (d.kind == kActF32) {
    *reinterpret_cast<float4*>(static_cast<float*>(d.p) + off) = make_float4(a, b, c, e);
  } else if (d.kind == kActPlanes) {
    store_planes4(static_cast<uint16_t*>(d.p) + off, d.plane, a, b, c, e);
  } else {
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(d.p) + off) = make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, e));
  }
}

// Loads that bypass L1 allocation for streamed-once data.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

}  // namespace bi
