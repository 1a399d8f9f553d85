// moe_common.cuh -- shared pieces of libmoe.so: error reporting, device status
// and launch counters, bf16 conversion and the bit-exact binary32 exp.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
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

// Binary32 exp from binary32 arithmetic, bit-identical to exp_cr (the defined
// exp above) wherever it decides; exp_f32 below takes it and falls back to
// exp_cr elsewhere, which avoids the double-precision chain for all but a few
// inputs.
// Table-driven reduction (P. T. P. Tang, "Table-driven implementation of the
// exponential function in IEEE floating-point arithmetic", ACM TOMS 15(2), 1989):
//   N = rint(x * 64/ln2), r = x - N ln2/64 (|r| <= ln2/128 plus rounding),
//   exp(x) = 2^(N >> 6) * 2^((N & 63)/64) * exp(r),
// with r, the table values 2^(j/64) and the product carried as unevaluated
// pairs of binary32 values (Dekker's exact products by fma, Knuth's TwoSum),
// about 45 bits.  exp_cr is within a few double ulps of exp(x), so both
// round to the same binary32 value unless exp(x) lies within a tiny fraction
// of an ulp of a rounding midpoint.  The pair decides unless it lies within
// 2^-16 ulp of a midpoint; then exp_fast_f32 reports no decision and the
// caller evaluates exp_cr (about 7 inputs in a million).  Checked on the
// host against the oracle's exp on every binary32 input in [-86, 88].
// ln2/64 = c1 + c2 + c3 with a 10-bit c1, so N * c1 is exact for |N| < 2^14;
// the table and the constants were computed with 60-digit decimal arithmetic.
#ifdef __CUDA_ARCH__
#define MOE_FADD(a, b) __fadd_rn((a), (b))
#define MOE_FSUB(a, b) __fsub_rn((a), (b))
#define MOE_FMUL(a, b) __fmul_rn((a), (b))
#define MOE_FFMA(a, b, c) __fmaf_rn((a), (b), (c))
#else  // host builds must not contract a*b+c (compile with -ffp-contract=off)
#define MOE_FADD(a, b) ((a) + (b))
#define MOE_FSUB(a, b) ((a) - (b))
#define MOE_FMUL(a, b) ((a) * (b))
#define MOE_FFMA(a, b, c) fmaf((a), (b), (c))
#endif

#define MOE_EXP_TAB_VALUES \
  0x1.0000000000000p+0f, 0x0.0p+0f, \
  0x1.02c9a40000000p+0f, -0x1.887fa00000000p-28f, \
  0x1.059b0e0000000p+0f, -0x1.9d4f520000000p-25f, \
  0x1.0874520000000p+0f, -0x1.e2990e0000000p-26f, \
  0x1.0b55860000000p+0f, 0x1.9f31220000000p-25f, \
  0x1.0e3ec40000000p+0f, -0x1.a585cc0000000p-25f, \
  0x1.11301e0000000p+0f, -0x1.fdb4960000000p-25f, \
  0x1.1429aa0000000p+0f, 0x1.d525bc0000000p-25f, \
  0x1.172b840000000p+0f, -0x1.c157420000000p-27f, \
  0x1.1a35be0000000p+0f, 0x1.6df96e0000000p-25f, \
  0x1.1d48740000000p+0f, -0x1.d2e8ca0000000p-25f, \
  0x1.2063b80000000p+0f, 0x1.0c519a0000000p-25f, \
  0x1.2387a60000000p+0f, 0x1.ceac480000000p-25f, \
  0x1.26b4560000000p+0f, 0x1.789f380000000p-26f, \
  0x1.29e9e00000000p+0f, -0x1.5c04240000000p-25f, \
  0x1.2d285a0000000p+0f, 0x1.b900c20000000p-26f, \
  0x1.306fe00000000p+0f, 0x1.4636e20000000p-25f, \
  0x1.33c08c0000000p+0f, -0x1.b37d200000000p-25f, \
  0x1.371a740000000p+0f, -0x1.18aac60000000p-25f, \
  0x1.3a7db40000000p+0f, -0x1.634c020000000p-25f, \
  0x1.3dea640000000p+0f, 0x1.8246840000000p-25f, \
  0x1.4160a20000000p+0f, 0x1.f72e2a0000000p-28f, \
  0x1.44e0860000000p+0f, 0x1.8624b40000000p-30f, \
  0x1.486a2c0000000p+0f, -0x1.47d8660000000p-25f, \
  0x1.4bfdae0000000p+0f, -0x1.593abc0000000p-25f, \
  0x1.4f9b280000000p+0f, -0x1.2c5a6c0000000p-25f, \
  0x1.5342b60000000p+0f, -0x1.2c56100000000p-25f, \
  0x1.56f4740000000p+0f, -0x1.295b040000000p-25f, \
  0x1.5ab07e0000000p+0f, -0x1.5bd5ec0000000p-27f, \
  0x1.5e76f20000000p+0f, -0x1.4a5bd60000000p-25f, \
  0x1.6247ec0000000p+0f, -0x1.f8b5500000000p-25f, \
  0x1.6623880000000p+0f, 0x1.2a91120000000p-27f, \
  0x1.6a09e60000000p+0f, 0x1.9fcef40000000p-26f, \
  0x1.6dfb240000000p+0f, -0x1.cd72e80000000p-27f, \
  0x1.71f75e0000000p+0f, 0x1.1d8bee0000000p-25f, \
  0x1.75feb60000000p+0f, -0x1.37b3060000000p-25f, \
  0x1.7a11480000000p+0f, -0x1.829fd00000000p-25f, \
  0x1.7e2f340000000p+0f, -0x1.2616340000000p-25f, \
  0x1.82589a0000000p+0f, -0x1.accc7c0000000p-26f, \
  0x1.868d9a0000000p+0f, -0x1.2edb440000000p-26f, \
  0x1.8ace540000000p+0f, 0x1.15506e0000000p-27f, \
  0x1.8f1aea0000000p+0f, -0x1.baa2320000000p-26f, \
  0x1.93737c0000000p+0f, -0x1.e647440000000p-25f, \
  0x1.97d82a0000000p+0f, -0x1.0d8d840000000p-31f, \
  0x1.9c49180000000p+0f, 0x1.51f8480000000p-27f, \
  0x1.a0c6680000000p+0f, -0x1.2886a60000000p-26f, \
  0x1.a5503c0000000p+0f, -0x1.b83b540000000p-25f, \
  0x1.a9e6b60000000p+0f, -0x1.50c0480000000p-25f, \
  0x1.ae89fa0000000p+0f, -0x1.a94b140000000p-26f, \
  0x1.b33a2c0000000p+0f, -0x1.ec3a820000000p-26f, \
  0x1.b7f7700000000p+0f, -0x1.a094380000000p-25f, \
  0x1.bcc1ea0000000p+0f, -0x1.f687c60000000p-25f, \
  0x1.c199be0000000p+0f, -0x1.3d56b20000000p-27f, \
  0x1.c67f120000000p+0f, 0x1.cafa2a0000000p-25f, \
  0x1.cb720e0000000p+0f, -0x1.8837cc0000000p-27f, \
  0x1.d072d40000000p+0f, 0x1.40f1300000000p-25f, \
  0x1.d5818e0000000p+0f, -0x1.822dbc0000000p-27f, \
  0x1.da9e600000000p+0f, 0x1.ed99420000000p-27f, \
  0x1.dfc9740000000p+0f, -0x1.908c940000000p-25f, \
  0x1.e502ee0000000p+0f, 0x1.e2cffe0000000p-26f, \
  0x1.ea4afa0000000p+0f, 0x1.52486c0000000p-27f, \
  0x1.efa1be0000000p+0f, 0x1.cc2b440000000p-25f, \
  0x1.f507660000000p+0f, -0x1.246eb00000000p-26f, \
  0x1.fa7c180000000p+0f, 0x1.9e90d80000000p-28f, \


static __device__ const float kExpTabDev[128] = {MOE_EXP_TAB_VALUES};
static const float kExpTabHost[128] = {MOE_EXP_TAB_VALUES};

__host__ __device__ __forceinline__ float exp_pow2i(int n) {  // 2^n, n a normal exponent
  union { unsigned u; float f; } v;
  v.u = static_cast<unsigned>(n + 127) << 23;
  return v.f;
}

__host__ __device__ __forceinline__ unsigned f32_bits(float f) {
  union { float f; unsigned u; } v;
  v.f = f;
  return v.u;
}

// true and *y = exp(x) when the binary32 pair decides; false otherwise (NaN,
// x outside [-86, 88], or within 2^-16 ulp of a rounding midpoint)
__host__ __device__ __forceinline__ bool exp_fast_f32(float x, float* y) {
  if (!(x >= -86.0f && x <= 88.0f)) return false;
  const float inv = 0x1.715476p+6f;                       // 64/ln2
  const float c1 = 0x1.63p-7f, c2 = -0x1.bd0106p-19f, c3 = 0x1.cf79acp-46f;
  const float nf = rintf(MOE_FMUL(x, inv));
  const int N = static_cast<int>(nf);
  const int j = N & 63;
  const int n = (N - j) / 64;
  // r = x - N ln2/64 as rh + rl
  const float t1 = MOE_FFMA(-nf, c1, x);                   // exact
  const float p2 = MOE_FMUL(nf, c2);
  const float p2e = MOE_FFMA(nf, c2, -p2);                 // exact error of p2
  const float rh0 = MOE_FSUB(t1, p2);                      // TwoSum(t1, -p2)
  const float b0 = MOE_FSUB(rh0, t1);
  const float e0 = MOE_FADD(MOE_FSUB(t1, MOE_FSUB(rh0, b0)), MOE_FSUB(-p2, b0));
  const float rl0 = MOE_FSUB(MOE_FSUB(e0, p2e), MOE_FMUL(nf, c3));
  const float rh = MOE_FADD(rh0, rl0);                     // TwoSum(rh0, rl0)
  const float b1 = MOE_FSUB(rh, rh0);
  const float rl = MOE_FADD(MOE_FSUB(rh0, MOE_FSUB(rh, b1)), MOE_FSUB(rl0, b1));
  // exp(r) - 1 = r + r^2/2 + r^3/6 + r^4/24 + r^5/120 as eh + el
  const float sq = MOE_FMUL(rh, rh);
  const float sqe = MOE_FFMA(rh, rh, -sq);
  const float h2 = MOE_FMUL(sq, 0.5f);
  const float poly = MOE_FFMA(rh, MOE_FFMA(rh, 0x1.111112p-7f, 0x1.555556p-5f), 0x1.555556p-3f);
  const float tail = MOE_FMUL(MOE_FMUL(sq, rh), poly);
  const float eh = MOE_FADD(rh, h2);                       // TwoSum(rh, h2)
  const float b2 = MOE_FSUB(eh, rh);
  const float ee = MOE_FADD(MOE_FSUB(rh, MOE_FSUB(eh, b2)), MOE_FSUB(h2, b2));
  const float el =
      MOE_FADD(ee, MOE_FADD(MOE_FADD(rl, MOE_FMUL(sqe, 0.5f)), MOE_FFMA(rh, rl, tail)));
  // y = T (1 + e) with T = 2^(j/64) = th + tl
#ifdef __CUDA_ARCH__
  const float th = __ldg(kExpTabDev + 2 * j), tl = __ldg(kExpTabDev + 2 * j + 1);
#else
  const float th = kExpTabHost[2 * j], tl = kExpTabHost[2 * j + 1];
#endif
  const float mh = MOE_FMUL(th, eh);
  const float ml = MOE_FFMA(th, eh, -mh);
  const float small = MOE_FADD(MOE_FADD(tl, ml), MOE_FFMA(th, el, MOE_FMUL(tl, eh)));
  const float s = MOE_FADD(th, mh);                        // Fast2Sum, |th| >= 1 > |mh|
  const float se = MOE_FSUB(mh, MOE_FSUB(s, th));
  const float lo = MOE_FADD(se, small);
  const float yh = MOE_FADD(s, lo);                        // the pair rounded to binary32
  const float err = MOE_FSUB(lo, MOE_FSUB(yh, s));         // exact: yh + err = s + lo
  // |err| in ulps of yh (the gap below a power of two is half as wide)
  const int ex = static_cast<int>((f32_bits(yh) >> 23) & 0xFFu) - 127;
  int sc = 23 - ex;
  if ((f32_bits(yh) & 0x7FFFFFu) == 0u && err < 0.0f) sc += 1;
  const float d = MOE_FMUL(err < 0.0f ? -err : err, exp_pow2i(sc));
  if (d > 0.5f - 0x1p-16f) return false;
  *y = MOE_FMUL(yh, exp_pow2i(n));                         // exact: a normal result
  return true;
}

// The defined binary32 exp as the kernels evaluate it: the binary32 pair of
// exp_fast_f32 where it decides, otherwise the double-precision chain exp_cr.
// Both give exp_cr's bits, so this is exp_cr, with double precision only for
// NaN, inputs outside [-86, 88] and about 7 in a million others.
__device__ __forceinline__ float exp_f32(float x) {
  float y;
  if (exp_fast_f32(x, &y)) return y;
  return exp_cr(x);
}

// sigma(g) = 1 / (1 + exp(-g)), two separately rounded binary32 ops after the exp
__device__ __forceinline__ float sigmoid_f32(float g) {
  const float e = exp_f32(-g);
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}

}  // namespace moe
