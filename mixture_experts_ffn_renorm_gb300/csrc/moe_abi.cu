// moe_abi.cu -- error reporting, device status word and launch counters of
// libmoe.so, and the introspection entry points declared in moe.h.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>

#include "moe_common.cuh"

namespace {
thread_local char g_msg[1024] = "";

// one status word and one counter array per device that loads the library
__device__ unsigned int g_status = 0;
__device__ unsigned long long g_launches[MOE_KID_COUNT];

constexpr int kMaxDevices = 64;
std::mutex g_diag_mu;
std::atomic<int> g_pdl{1};
moe::DeviceDiag g_diag[kMaxDevices];
bool g_diag_ready[kMaxDevices] = {};
}  // namespace

namespace moe {

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_msg[0] = '\0'; }

DeviceDiag device_diag() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return DeviceDiag{nullptr, nullptr};
  }
  std::lock_guard<std::mutex> lock(g_diag_mu);
  if (!g_diag_ready[dev]) {
    DeviceDiag d{nullptr, nullptr};
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status) != cudaSuccess ||
        cudaGetSymbolAddress(reinterpret_cast<void**>(&d.launches), g_launches) != cudaSuccess) {
      cudaGetLastError();
      return DeviceDiag{nullptr, nullptr};
    }
    g_diag[dev] = d;
    g_diag_ready[dev] = true;
  }
  return g_diag[dev];
}

bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }

int sm_count() {
  static std::atomic<int> cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 1;
  }
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return 1;
    }
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "%s: kernel launch failed: %s", what, cudaGetErrorString(e));
  return MOE_OK;
}

}  // namespace moe

extern "C" {

const char* moe_last_error(void) { return g_msg; }

int moe_abi_version(void) { return 8; }

int moe_set_pdl(int enable) {
  moe::clear_error();
  if (enable != 0 && enable != 1)
    return moe::set_error(MOE_ERR_ARG, "moe_set_pdl: enable must be 0 or 1, got %d", enable);
  return g_pdl.exchange(enable);
}

int moe_device_status(int* status_out, int clear) {
  moe::clear_error();
  if (status_out == nullptr) return moe::set_error(MOE_ERR_ARG, "moe_device_status: status_out is NULL");
  unsigned int v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (e == cudaSuccess && clear) {
    unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
  }
  if (e != cudaSuccess)
    return moe::set_error(MOE_ERR_CUDA, "moe_device_status: %s", cudaGetErrorString(e));
  *status_out = static_cast<int>(v);
  return MOE_OK;
}

int moe_launch_counts(unsigned long long* counts, int n) {
  moe::clear_error();
  if (counts == nullptr || n <= 0) return moe::set_error(MOE_ERR_ARG, "moe_launch_counts: bad buffer");
  unsigned long long tmp[MOE_KID_COUNT];
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(tmp, g_launches, sizeof(tmp));
  if (e != cudaSuccess)
    return moe::set_error(MOE_ERR_CUDA, "moe_launch_counts: %s", cudaGetErrorString(e));
  int m = n < MOE_KID_COUNT ? n : MOE_KID_COUNT;
  for (int i = 0; i < m; ++i) counts[i] = tmp[i];
  return m;
}

}  // extern "C"
