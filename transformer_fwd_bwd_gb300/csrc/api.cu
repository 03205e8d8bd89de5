// Status reporting, the device error flag, device facts, the launch counter and the
// optional per-GEMM timing.
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace {
thread_local char g_msg[512] = "";
constexpr int kMaxDevices = 64;
// One flag word per device; the host reaches it through cudaGetSymbolAddress.
__device__ uint32_t g_errflag;
uint32_t* g_flag_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_mu;
std::atomic<uint64_t> g_launches{0};
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

// GEMM timing: while enabled, each GEMM launch gets a record and a region of a device buffer
// in which every CTA of the GEMM kernel (and of a K split's reduce kernel) stores %globaltimer
// when it starts work (after its programmatic-launch wait) and when it has finished.
struct GemmRecord {
  double flops;
  int shape[8];
  int grid, rgrid;  // CTAs of the GEMM kernel and of the reduce kernel (0: none)
};
std::mutex g_prof_mu;
unsigned long long* g_ts_buf = nullptr;  // capacity × kProfSlots × 2 words
int g_ts_dev = -1;
size_t g_prof_cap = 0;
std::vector<GemmRecord> g_records;
bool g_prof_on = false;
}  // namespace

namespace xt {

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int check_launch(const char* what) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(XT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return XT_OK;
}

static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

uint32_t* errflag() {
  int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_flag_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_errflag) != cudaSuccess) return nullptr;
    g_flag_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_flag_ptr[dev];
}

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

int num_sms() {
  int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = v > 0 ? v : 1;
  }
  return g_sms[dev];
}

bool gemm_profile_begin(double flops, const int* shape, unsigned long long** ts, void** token) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on || !g_ts_buf || g_records.size() >= g_prof_cap) return false;
  GemmRecord r{flops, {}, 0, 0};
  for (int i = 0; i < 8; ++i) r.shape[i] = shape[i];
  *ts = g_ts_buf + g_records.size() * size_t(kProfSlots) * 2;
  g_records.push_back(r);
  *token = reinterpret_cast<void*>(g_records.size());
  return true;
}

void gemm_profile_grids(void* token, int grid, int rgrid) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  const size_t i = reinterpret_cast<size_t>(token);
  if (i >= 1 && i <= g_records.size()) {
    g_records[i - 1].grid = grid;
    g_records[i - 1].rgrid = rgrid;
  }
}

}  // namespace xt

extern "C" {

uint64_t xt_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int xt_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
  return XT_OK;
}

uint64_t xt_get_wait_limit_ns(void) { return g_wait_ns.load(std::memory_order_relaxed); }

int xt_profile_gemm(int capacity) {
  XT_REQUIRE(capacity >= 0, "xt_profile_gemm: negative capacity");
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_records.clear();
  g_prof_on = capacity > 0;
  if (!g_prof_on) return XT_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return xt::check_launch("xt_profile_gemm");
  if (g_ts_buf && (g_ts_dev != dev || g_prof_cap < size_t(capacity))) {
    cudaFree(g_ts_buf);
    g_ts_buf = nullptr;
  }
  if (!g_ts_buf) {
    const size_t bytes = size_t(capacity) * xt::kProfSlots * 2 * sizeof(unsigned long long);
    if (cudaMalloc(&g_ts_buf, bytes) != cudaSuccess) {
      g_ts_buf = nullptr;
      g_prof_on = false;
      return xt::check_launch("xt_profile_gemm");
    }
    g_ts_dev = dev;
    g_prof_cap = size_t(capacity);
  }
  return XT_OK;
}

int xt_profile_gemm_read(double* flops, float* ms, int* shapes, int max_records, int* n) {
  XT_REQUIRE(n != nullptr, "xt_profile_gemm_read: n is NULL");
  std::lock_guard<std::mutex> lk(g_prof_mu);
  const int cnt = int(g_records.size());
  *n = cnt;
  if (cnt == 0) return XT_OK;
  if (cudaDeviceSynchronize() != cudaSuccess) return xt::check_launch("xt_profile_gemm_read");
  std::vector<unsigned long long> ts(size_t(cnt) * xt::kProfSlots * 2);
  if (cudaMemcpy(ts.data(), g_ts_buf, ts.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost) != cudaSuccess)
    return xt::check_launch("xt_profile_gemm_read");
  for (int i = 0; i < cnt && i < max_records; ++i) {
    const GemmRecord& r = g_records[i];
    const unsigned long long* t = ts.data() + size_t(i) * xt::kProfSlots * 2;
    unsigned long long t0 = ~0ull, t1 = 0;
    for (int c = 0; c < r.grid; ++c) {
      if (t[2 * c] < t0) t0 = t[2 * c];
      if (t[2 * c + 1] > t1) t1 = t[2 * c + 1];
    }
    for (int c = 0; c < r.rgrid; ++c) {
      const unsigned long long e = t[2 * (xt::kProfGemmSlots + c) + 1];
      if (e > t1) t1 = e;
    }
    if (flops) flops[i] = r.flops;
    if (ms) ms[i] = t1 > t0 ? float(double(t1 - t0) * 1e-6) : 0.f;
    if (shapes)
      for (int j = 0; j < 8; ++j) shapes[8 * i + j] = r.shape[j];
  }
  return XT_OK;
}

const char* xt_last_error(void) { return g_msg; }

const char* xt_version(void) { return "xt 0.1 (sm_103a)"; }

int xt_get_device_errors(uint32_t* out, void* stream) {
  XT_REQUIRE(out != nullptr, "xt_get_device_errors: out is NULL");
  uint32_t* f = xt::errflag();
  if (!f) return xt::fail(XT_ERR_CUDA, "xt_get_device_errors: no device flag");
  cudaStream_t s = xt::as_stream(stream);
  if (cudaMemcpyAsync(out, f, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return xt::check_launch("xt_get_device_errors");
  if (*out & XT_DEVERR_TIMEOUT)
    return xt::fail(XT_ERR_TIMEOUT, "a bounded wait on the device gave up");
  return XT_OK;
}

int xt_clear_device_errors(void* stream) {
  uint32_t* f = xt::errflag();
  if (!f) return xt::fail(XT_ERR_CUDA, "xt_clear_device_errors: no device flag");
  if (cudaMemsetAsync(f, 0, sizeof(uint32_t), xt::as_stream(stream)) != cudaSuccess)
    return xt::check_launch("xt_clear_device_errors");
  return XT_OK;
}

}  // extern "C"
