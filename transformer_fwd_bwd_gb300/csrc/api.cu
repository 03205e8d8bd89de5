// Status reporting, the device error flag, device facts, the launch counter and the
// optional per-GEMM event timing.
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

// GEMM timing: pairs of events recorded around each GEMM launch while enabled.
struct GemmRecord {
  double flops;
  cudaEvent_t start, stop;
  int shape[8];
};
std::mutex g_prof_mu;
std::vector<cudaEvent_t> g_ev_pool;
std::vector<GemmRecord> g_records;
size_t g_ev_next = 0;
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

// Inside a stream capture the event becomes an event-record node of the graph, so each
// replay records it; outside, a plain record.
static void record_event(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) == cudaSuccess && st == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

bool gemm_profile_begin(cudaStream_t s, double flops, const int* shape, void** token) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on || g_ev_next + 2 > g_ev_pool.size()) return false;
  GemmRecord r{flops, g_ev_pool[g_ev_next], g_ev_pool[g_ev_next + 1], {}};
  for (int i = 0; i < 8; ++i) r.shape[i] = shape[i];
  g_ev_next += 2;
  record_event(r.start, s);
  g_records.push_back(r);
  *token = reinterpret_cast<void*>(g_records.size());
  return true;
}

void gemm_profile_end(cudaStream_t s, void* token) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  const size_t i = reinterpret_cast<size_t>(token);
  if (i >= 1 && i <= g_records.size()) record_event(g_records[i - 1].stop, s);
}

}  // namespace xt

extern "C" {

uint64_t xt_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int xt_profile_gemm(int capacity) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_records.clear();
  g_ev_next = 0;
  g_prof_on = capacity > 0;
  while (g_ev_pool.size() < size_t(2 * capacity)) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return xt::check_launch("xt_profile_gemm");
    g_ev_pool.push_back(e);
  }
  return XT_OK;
}

int xt_profile_gemm_read(double* flops, float* ms, int* shapes, int max_records, int* n) {
  XT_REQUIRE(n != nullptr, "xt_profile_gemm_read: n is NULL");
  std::lock_guard<std::mutex> lk(g_prof_mu);
  const int cnt = int(g_records.size());
  *n = cnt;
  for (int i = 0; i < cnt && i < max_records; ++i) {
    if (cudaEventSynchronize(g_records[i].stop) != cudaSuccess) return xt::check_launch("xt_profile_gemm_read");
    float t = 0.f;
    cudaEventElapsedTime(&t, g_records[i].start, g_records[i].stop);
    if (flops) flops[i] = g_records[i].flops;
    if (ms) ms[i] = t;
    if (shapes)
      for (int j = 0; j < 8; ++j) shapes[8 * i + j] = g_records[i].shape[j];
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
