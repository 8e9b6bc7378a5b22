// Library-wide C entry points: status strings, error detail, device facts.
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <vector>

#include "common.cuh"

namespace bi {

namespace {
thread_local std::string g_last_error;
std::mutex g_sm_mutex;
std::vector<int> g_sm_count;  // per device, 0 = not queried yet
}  // namespace

void set_error(const char* fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

void clear_error() { g_last_error.clear(); }

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(g_sm_mutex);
  if (dev >= static_cast<int>(g_sm_count.size())) g_sm_count.resize(dev + 1, 0);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

namespace {
std::mutex g_attr_mutex;
std::set<std::tuple<const void*, int, int>> g_smem_set;          // (kernel, device, bytes) already raised
std::map<std::tuple<const void*, int, int, size_t>, int> g_occ;  // (kernel, device, threads, smem) -> CTAs/SM
}  // namespace

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  const auto key = std::make_tuple(kernel, dev, bytes);
  if (g_smem_set.count(key)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g_smem_set.insert(key);
  return e;
}

int occupancy_per_sm(const void* kernel, int threads, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  const auto key = std::make_tuple(kernel, dev, threads, smem);
  auto it = g_occ.find(key);
  if (it != g_occ.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) n = 1;
  g_occ[key] = n;
  return n;
}

// Defined next to the kernels that own a device error word.
int take_gemm_device_error(cudaStream_t s, int32_t* code);
int take_attn_device_error(cudaStream_t s, int32_t* code);
int take_pointwise_device_error(cudaStream_t s, int32_t* code);

// ------------------------------------------------------------------ launch timer
volatile int g_profiling = 0;

namespace {
const char* const kTagNames[kTagCount] = {
    "rmsnorm",          "rmsnorm_split",       "gemm",        "splitk_reduce", "attn_plan",   "attn_decode_split",
    "attn_decode_merge", "attn_prefill_split", "attn_prefill_merge", "qkv_rope_store", "swiglu", "embed",
    "topk",             "batch_index",         "gather_rows", "rope_table",
    "split_planes"};

struct ProfState {
  std::mutex mu;
  std::vector<cudaEvent_t> events;  // 2 per slot
  std::vector<int> tags;            // per used slot
  int capacity = 0;
};
ProfState g_prof;
}  // namespace

int prof_begin(int tag, cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  if (!g_profiling) return -1;
  const int slot = static_cast<int>(g_prof.tags.size());
  if (slot >= g_prof.capacity) return -1;
  if (cudaEventRecord(g_prof.events[2 * slot], s) != cudaSuccess) return -1;
  g_prof.tags.push_back(tag);
  return slot;
}

void prof_end(int slot, cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  if (slot >= 0 && slot < g_prof.capacity) cudaEventRecord(g_prof.events[2 * slot + 1], s);
}

}  // namespace bi

extern "C" bi_status bi_profile_start(int32_t max_launches) {
  bi::clear_error();
  BI_REQUIRE(max_launches >= 1 && max_launches <= (1 << 22), BI_ERR_INVALID_ARG, "bi_profile_start: %d launches",
             max_launches);
  std::lock_guard<std::mutex> lock(bi::g_prof.mu);
  for (cudaEvent_t e : bi::g_prof.events) cudaEventDestroy(e);
  bi::g_prof.events.clear();
  bi::g_prof.tags.clear();
  bi::g_prof.capacity = 0;
  bi::g_prof.events.resize(2 * static_cast<size_t>(max_launches));
  for (auto& e : bi::g_prof.events) BI_CUDA_TRY(cudaEventCreate(&e));
  bi::g_prof.capacity = max_launches;
  bi::g_profiling = 1;
  return BI_OK;
}

extern "C" bi_status bi_profile_stop(void) {
  bi::g_profiling = 0;
  return BI_OK;
}

extern "C" bi_status bi_profile_read(const char* kernel, int32_t* launches, double* total_ms) {
  bi::clear_error();
  BI_REQUIRE(kernel && launches && total_ms, BI_ERR_INVALID_ARG, "bi_profile_read: null pointer");
  int tag = -1;
  for (int i = 0; i < bi::kTagCount; ++i)
    if (std::string(kernel) == bi::kTagNames[i]) tag = i;
  BI_REQUIRE(tag >= 0, BI_ERR_INVALID_ARG, "bi_profile_read: unknown kernel '%s'", kernel);
  std::lock_guard<std::mutex> lock(bi::g_prof.mu);
  int n = 0;
  double tot = 0.0;
  for (size_t i = 0; i < bi::g_prof.tags.size(); ++i) {
    if (bi::g_prof.tags[i] != tag) continue;
    BI_CUDA_TRY(cudaEventSynchronize(bi::g_prof.events[2 * i + 1]));
    float ms = 0.f;
    BI_CUDA_TRY(cudaEventElapsedTime(&ms, bi::g_prof.events[2 * i], bi::g_prof.events[2 * i + 1]));
    tot += ms;
    ++n;
  }
  *launches = n;
  *total_ms = tot;
  return BI_OK;
}

extern "C" const char* bi_profile_kernel_name(int32_t i) {
  return (i >= 0 && i < bi::kTagCount) ? bi::kTagNames[i] : nullptr;
}

extern "C" int32_t bi_profile_kernel_count(void) { return bi::kTagCount; }

extern "C" const char* bi_status_string(bi_status st) {
  switch (st) {
    case BI_OK: return "BI_OK";
    case BI_ERR_INVALID_ARG: return "BI_ERR_INVALID_ARG";
    case BI_ERR_UNSUPPORTED: return "BI_ERR_UNSUPPORTED";
    case BI_ERR_WORKSPACE: return "BI_ERR_WORKSPACE";
    case BI_ERR_CUDA: return "BI_ERR_CUDA";
    case BI_ERR_TIMEOUT: return "BI_ERR_TIMEOUT";
  }
  return "BI_ERR_UNKNOWN";
}

extern "C" const char* bi_last_error_message(void) { return bi::g_last_error.c_str(); }

extern "C" int32_t bi_version(void) { return 100; }

extern "C" int32_t bi_num_sms(void) { return bi::num_sms(); }

extern "C" bi_status bi_device_error(int32_t* code, bi_stream s) {
  bi::clear_error();
  BI_REQUIRE(code != nullptr, BI_ERR_INVALID_ARG, "bi_device_error: null code pointer");
  *code = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  BI_CUDA_TRY(cudaStreamSynchronize(st));
  int32_t cg = 0, ca = 0, cp = 0;
  if (bi::take_gemm_device_error(st, &cg) != 0 || bi::take_attn_device_error(st, &ca) != 0 ||
      bi::take_pointwise_device_error(st, &cp) != 0) {
    bi::set_error("bi_device_error: reading the device error words failed");
    return BI_ERR_CUDA;
  }
  const int32_t c = cg != 0 ? cg : ca != 0 ? ca : cp;
  *code = c;
  if (c == 0) return BI_OK;
  if (c == 18) {
    bi::set_error("decode attention: its dynamic shared memory was not 1024-byte aligned; nothing was computed");
    return BI_ERR_UNSUPPORTED;
  }
  if (c >= 16) {
    bi::set_error("a kernel met an out-of-range KV length, block-table entry or position (site code %d)", c);
    return BI_ERR_INVALID_ARG;
  }
  bi::set_error("an in-kernel wait ran out (site code %d)", c);
  return BI_ERR_TIMEOUT;
}
