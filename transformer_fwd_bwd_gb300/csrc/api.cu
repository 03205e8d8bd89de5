// Status reporting, the device error flag and device facts.
#include <mutex>

#include "common.cuh"

namespace {
thread_local char g_msg[512] = "";
constexpr int kMaxDevices = 64;
// One flag word per device; the host reaches it through cudaGetSymbolAddress.
__device__ uint32_t g_errflag;
uint32_t* g_flag_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_mu;
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

}  // namespace xt

extern "C" {

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
