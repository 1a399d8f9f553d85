// moe_common.cuh -- shared pieces of libmoe.so: error reporting, device status
// and launch counters, bf16 conversion and the bit-exact binary32 exp.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe.h"

namespace moe {

// ------------------------------------------------------------------ host side
// Thread-local message behind moe_last_error(); returns `code` for chaining.
int set_error(int code, const char* fmt, ...);
void clear_error();
// Device pointers of the status word and launch counters (defined once in
// moe_abi.cu; other translation units receive them as kernel arguments).
struct DeviceDiag {
  unsigned int* status;             // MOE_STATUS_* bits
  unsigned long long* launches;     // [MOE_KID_COUNT]
};
DeviceDiag device_diag();  // resolves the symbols on first use per device
int check_launch(const char* what);  // cudaGetLastError -> MOE_ERR_CUDA
int sm_count();                      // SMs of the current device (cached per device)
// result of a cudaLaunchKernelEx -> MOE_OK or MOE_ERR_CUDA (sticky error cleared)
inline int launch_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MOE_OK;
  cudaGetLastError();
  return set_error(MOE_ERR_CUDA, "%s: kernel launch failed: %s", what, cudaGetErrorString(e));
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Programmatic dependent launch (process-wide switch, moe_set_pdl; on by default).
bool pdl_enabled();

// Every kernel of the library goes through this launch: with PDL on it carries
// the programmatic-stream-serialisation attribute, so the kernel may be
// scheduled while the previous kernel in the stream is still running; its
// CTAs then do their set-up (barrier init, TMEM allocation, descriptor
// prefetch) and block in grid_dep_wait() until the predecessor has completed.
// `extra` are further launch attributes (a cluster shape).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, const cudaLaunchAttribute* extra, int n_extra,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[4];
  int n = 0;
  for (int i = 0; i < n_extra && n < 3; ++i) attr[n++] = extra[i];
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(n);
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------ device side
// Ordering against the previous kernel in the stream under programmatic
// dependent launch.  grid_dep_wait() returns once every grid this one depends
// on has completed and its memory is visible (at once without PDL); each
// kernel calls it in every CTA before its first global read of another
// kernel's output and before its first global write, so a chain of launches
// keeps full stream order.  grid_dep_launch() then lets the next kernel in
// the stream be scheduled while this one runs.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void count_launch(unsigned long long* launches, int kid) {
  if (launches != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&
      threadIdx.x == 0)
    atomicAdd(launches + kid, 1ull);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Round to nearest even on the binary32 bit pattern; NaN stays NaN (quiet).
// Same result as the hardware cvt.rn.bf16.f32, used where the rounding must
// be visible in source.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Binary32 exp used wherever the block's results must be bit-reproducible
// (the sigmoid gate and the router weights).  It is the binary32 rounding of
// one fixed sequence of double-precision operations:
//   n = rint(x * log2(e));  r = (x - n*ln2_hi) - n*ln2_lo   (Cody & Waite, 1980)
//   p = Horner form of sum_{k=0}^{13} r^k / k!   (|r| <= ln2/2: truncation < 4e-18)
//   y = p * 2^n (exact), result = (float)y
// ln2_hi = floor(ln2 * 2^32) / 2^32 (so n*ln2_hi is exact for |n| < 2^21) and
// ln2_lo = ln2 - ln2_hi rounded to double.  Every step is an explicitly
// rounded IEEE double operation (no contraction), so any conforming machine
// that performs the same steps gets the same bits.
__device__ __forceinline__ float exp_cr(float x) {
  if (x != x) return x;
  if (x > 89.0f) return __int_as_float(0x7f800000);
  if (x < -104.0f) return 0.0f;
  const double log2e = 1.4426950408889634074;            // 1/ln2 rounded to double
  const double ln2_hi = 2977044471.0 / 4294967296.0;     // exact: 32-bit head of ln2
  const double ln2_lo = 1.9082149292705877e-10;          // ln2 - ln2_hi rounded to double
  double xd = static_cast<double>(x);
  double n = rint(__dmul_rn(xd, log2e));
  double r = __dadd_rn(xd, -__dmul_rn(n, ln2_hi));
  r = __dadd_rn(r, -__dmul_rn(n, ln2_lo));
  // 1/k! for k = 13 .. 0; each k! is an exact double, each quotient rounded once
  double p = 1.0 / 6227020800.0;
  p = __dadd_rn(__dmul_rn(p, r), 1.0 / 479001600.0);
  p = __dadd_rn(__dmul_rn(p, r), 1.0 / 39916800.0);
  p = __dadd_rn(__dmul_rn(p, r), 1.0 / 3628800.0);
  p = __dadd_rn(__dmul_rn(p, r), 1.0 / 362880.0);
  p = __dadd_rn(__dmul_rn(p, r), 1.0 / 40320.0);
  p = __dadd_rn(__dmul_rn(p, r), 1.0 / 5040.0);
  p = __dadd_rn(__dmul_rn(p, r), 1.0 / 720.0);
  p = __dadd_rn(__dmul_rn(p, r), 1.0 / 120.0);
  p = __dadd_rn(__dmul_rn(p, r), 1.0 / 24.0);
  p = __dadd_rn(__dmul_rn(p, r), 1.0 / 6.0);
  p = __dadd_rn(__dmul_rn(p, r), 0.5);
  p = __dadd_rn(__dmul_rn(p, r), 1.0);
  p = __dadd_rn(__dmul_rn(p, r), 1.0);
  // 2^n as a double bit pattern: n is in [-151, 129] here, a normal exponent
  long long ni = static_cast<long long>(n);
  double two_n = __longlong_as_double((ni + 1023ll) << 52);
  return __double2float_rn(__dmul_rn(p, two_n));
}

// sigma(g) = 1 / (1 + exp_cr(-g)), two separately rounded binary32 ops
__device__ __forceinline__ float sigmoid_cr(float g) {
  float e = exp_cr(-g);
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}

}  // namespace moe
