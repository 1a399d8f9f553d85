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

namespace {
// exp and sigmoid of the bit patterns first, first + 1, ... (mod 2^32)
__global__ void __launch_bounds__(256)
exp_sigmoid_kernel(uint32_t first, long long n, float* __restrict__ e, float* __restrict__ s,
                   unsigned long long* launches) {
  moe::count_launch(launches, MOE_KID_EXP_SIGMOID);
  moe::grid_dep_wait();
  moe::grid_dep_launch();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const float x = __uint_as_float(first + static_cast<uint32_t>(i));
    if (e) e[i] = moe::exp_f32(x);
    if (s) s[i] = moe::sigmoid_f32(x);
  }
}
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

int moe_abi_version(void) { return 10; }

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

int moe_exp_sigmoid_f32(uint32_t first_bits, long long n, float* exp_out, float* sigmoid_out,
                        void* stream) {
  moe::clear_error();
  const char* op = "moe_exp_sigmoid_f32";
  if (n < 0 || n > (1ll << 32)) return moe::set_error(MOE_ERR_ARG, "%s: n=%lld outside [0, 2^32]", op, n);
  if (!exp_out && !sigmoid_out) return moe::set_error(MOE_ERR_ARG, "%s: both outputs are NULL", op);
  if ((reinterpret_cast<uintptr_t>(exp_out) & 3u) || (reinterpret_cast<uintptr_t>(sigmoid_out) & 3u))
    return moe::set_error(MOE_ERR_ALIGN, "%s: outputs must be 4-byte aligned", op);
  if (n == 0) return MOE_OK;
  const long long blocks_needed = (n + 255) / 256;
  const long long cap = 8ll * moe::sm_count();
  const unsigned blocks = static_cast<unsigned>(blocks_needed < cap ? blocks_needed : cap);
  moe::DeviceDiag diag = moe::device_diag();
  return moe::launch_status(
      moe::launch_kernel(exp_sigmoid_kernel, dim3(blocks), dim3(256), 0,
                         static_cast<cudaStream_t>(stream), nullptr, 0, first_bits, n, exp_out,
                         sigmoid_out, diag.launches),
      op);
}

}  // extern "C"
