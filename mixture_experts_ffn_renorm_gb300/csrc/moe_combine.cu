// moe_combine.cu -- kMoeCombine, kMoeCombineGate and kSharedExpertGate
// (vllm.cpp PR #509 "MoE combine/gate ops -- SharedExpertGate, MoeCombine,
// MoeCombineGate": "What changed" gives the formulas; the review rework makes
// them bit-exact: sequential K order, one store rounding, no contraction; the
// routed_scale rework scales the finished routed sum before the shared term).
//
// Design: a pure HBM stream.  One thread owns 8 consecutive channels of one
// token, so every expert row, shared row and output row moves as one 16-byte
// vector per thread (two for f32) and a warp touches 512 contiguous bytes per
// load.  All K expert vectors of a thread are in flight at once.  The sigmoid
// of the gate is evaluated once per token per block (about 60 binary32
// operations, and a double-precision chain for the few inputs where the
// binary32 form declines); a gate block streams several slices so that it is
// amortised and overlaps the loads.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;       // channels per thread
constexpr int kChunkK = 8;    // expert rows loaded per batch of loads
constexpr int kGateIters = 4; // slices per block in the fused-sigmoid gate kernels

enum Mode { kCombine = 0, kCombineGate = 1, kGateOnly = 2 };

// 8 consecutive channels of one row: `Raw` is what a load brings in (one
// 16-byte vector of bf16, two of f32); widening to f32 is deferred to the
// arithmetic so that loads in flight hold packed data.
template <typename T>
struct Vec8;
template <>
struct Vec8<float> {
  struct Raw { float4 a, b; };
  __device__ __forceinline__ static Raw load_raw(const void* base, size_t idx) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
    return Raw{__ldg(p), __ldg(p + 1)};
  }
  __device__ __forceinline__ static void widen(const Raw& r, float* v) {
    v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w;
    v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
  }
  __device__ __forceinline__ static void load(const void* base, size_t idx, float* v) {
    widen(load_raw(base, idx), v);
  }
  __device__ __forceinline__ static void store(void* base, size_t idx, const float* v) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + idx);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    p[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};
template <>
struct Vec8<__nv_bfloat16> {
  using Raw = uint4;
  __device__ __forceinline__ static Raw load_raw(const void* base, size_t idx) {
    return __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + idx));
  }
  __device__ __forceinline__ static void widen(const Raw& a, float* v) {
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ static void load(const void* base, size_t idx, float* v) {
    widen(load_raw(base, idx), v);
  }
  __device__ __forceinline__ static void store(void* base, size_t idx, const float* v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = static_cast<uint32_t>(f32_to_bf16_bits(v[2 * i])) |
             (static_cast<uint32_t>(f32_to_bf16_bits(v[2 * i + 1])) << 16);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + idx) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

__device__ __forceinline__ float round_through_bf16(float v) {
  return __uint_as_float(static_cast<uint32_t>(f32_to_bf16_bits(v)) << 16);
}

// The routed sum of one 8-channel item: acc = (sum_k eo[t,k,c] (* w[t,k])) * rs,
// sequential in k from +0, every operation separately rounded.  All of a
// batch's expert rows are loaded before any arithmetic: rows past K load row
// K-1 again (a cache hit) instead of being predicated off, so the compiler
// keeps every load in flight at once.
template <typename EoT, bool kHasW>
__device__ __forceinline__ void routed_sum(const void* __restrict__ eo,
                                           const float* __restrict__ w, float rs, int t, int c0,
                                           int K, int H, float (&acc)[kVec]) {
#pragma unroll
  for (int i = 0; i < kVec; ++i) acc[i] = 0.0f;
  const size_t row0 = static_cast<size_t>(t) * K;
  for (int k0 = 0; k0 < K; k0 += kChunkK) {
    typename Vec8<EoT>::Raw raw[kChunkK];
    float wk[kChunkK];
#pragma unroll
    for (int j = 0; j < kChunkK; ++j) {
      const int kk = min(k0 + j, K - 1);
      raw[j] = Vec8<EoT>::load_raw(eo, (row0 + kk) * H + c0);
      wk[j] = kHasW ? __ldg(w + row0 + kk) : 1.0f;
    }
    const int kn = min(kChunkK, K - k0);
#pragma unroll
    for (int j = 0; j < kChunkK; ++j) {
      if (j < kn) {
        float v[kVec];
        Vec8<EoT>::widen(raw[j], v);
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
          float term = kHasW ? __fmul_rn(v[i], wk[j]) : v[i];
          acc[i] = __fadd_rn(acc[i], term);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kVec; ++i) acc[i] = __fmul_rn(acc[i], rs);
}

// kMoeCombine: one 8-channel item per thread
// bf16 expert rows: <= 64 registers, 4 blocks (32 warps) per SM keep more loads in flight
template <typename EoT>
constexpr int min_blocks() { return sizeof(EoT) == 2 ? 4 : 2; }

template <int kMode, typename EoT, typename ShT, typename OutT, bool kHasW, bool kHasShared>
__global__ void __launch_bounds__(kThreads, min_blocks<EoT>())
combine_kernel(const void* __restrict__ eo, const float* __restrict__ w,
               const void* __restrict__ sh, const float* __restrict__ gl, float rs, int T, int K,
               int H, void* __restrict__ out, unsigned long long* launches, int kid) {
  (void)gl;
  count_launch(launches, kid);
  grid_dep_wait();
  grid_dep_launch();
  const int ipr = H / kVec;                         // items per token row
  const long long item = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  if (item >= static_cast<long long>(T) * ipr) return;
  const int t = static_cast<int>(item / ipr);
  const int c0 = static_cast<int>(item % ipr) * kVec;
  float shv[kVec];
  if (kHasShared) Vec8<ShT>::load(sh, static_cast<size_t>(t) * H + c0, shv);
  float acc[kVec];
  routed_sum<EoT, kHasW>(eo, w, rs, t, c0, K, H, acc);
  if (kHasShared) {
#pragma unroll
    for (int i = 0; i < kVec; ++i) acc[i] = __fadd_rn(acc[i], shv[i]);
  }
  Vec8<OutT>::store(out, static_cast<size_t>(t) * H + c0, acc);
}

// kMoeCombineGate / kSharedExpertGate: a block streams kGateIters consecutive
// slices of kThreads items, so the sigmoid of each of its tokens is evaluated
// once per block, by full warps, while the first slice's loads are in flight.
// sigma(gl[t]) for every token, one per thread, into s_out[T].  One warp per
// block, so the tokens are spread over as many SMs as possible: a warp whose
// lanes meet an input the binary32 exp declines runs the double-precision
// chain, which GB300's few FP64 units execute slowly.
constexpr int kSigThreads = 32;
__global__ void __launch_bounds__(kSigThreads)
gate_sigmoid_kernel(const float* __restrict__ gl, int T, float* __restrict__ s_out,
                    unsigned long long* launches) {
  count_launch(launches, MOE_KID_GATE_SIGMOID);
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.x * kSigThreads + threadIdx.x;
  if (t < T) s_out[t] = sigmoid_f32(__ldg(gl + t));
}

// The gate ops with the sigmoids already in `sig` (gate_sigmoid_kernel): a
// plain stream, one 8-channel item per thread, no double precision.
// This kernel is always launched right after gate_sigmoid_kernel, which waits
// for all earlier work in the stream before it lets this one start; so under
// programmatic dependent launch everything this kernel reads except `sig` is
// final from its first instruction, and every earlier reader of `out` is done.
// It streams its expert and shared rows first and waits only before it reads
// the sigmoids, which overlaps the two kernels.
template <int kMode, typename EoT, typename ShT, typename OutT, bool kHasW, bool kHasShared>
__global__ void __launch_bounds__(kThreads, min_blocks<EoT>())
gate_stream_kernel(const void* __restrict__ eo, const float* __restrict__ w,
                   const void* __restrict__ sh, const float* __restrict__ sig, float rs, int T,
                   int K, int H, void* __restrict__ out, unsigned long long* launches, int kid) {
  count_launch(launches, kid);
  const int ipr = H / kVec;
  const long long item = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  const bool live = item < static_cast<long long>(T) * ipr;
  const int t = live ? static_cast<int>(item / ipr) : 0;
  const int c0 = live ? static_cast<int>(item % ipr) * kVec : 0;
  float shv[kVec], acc[kVec];
  if (live) {
    Vec8<ShT>::load(sh, static_cast<size_t>(t) * H + c0, shv);
    if (kMode == kCombineGate) routed_sum<EoT, kHasW>(eo, w, rs, t, c0, K, H, acc);
  }
  grid_dep_wait();     // the sigmoid pass has completed
  grid_dep_launch();
  if (!live) return;
  const float sg = sig[t];
  float o[kVec];
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const float g = __fmul_rn(sg, shv[i]);
    o[i] = (kMode == kGateOnly) ? g : __fadd_rn(acc[i], round_through_bf16(g));
  }
  Vec8<OutT>::store(out, static_cast<size_t>(t) * H + c0, o);
}

template <int kMode, typename EoT, typename ShT, typename OutT, bool kHasW, bool kHasShared>
__global__ void __launch_bounds__(kThreads)
gate_kernel(const void* __restrict__ eo, const float* __restrict__ w,
            const void* __restrict__ sh, const float* __restrict__ gl, float rs, int T, int K,
            int H, void* __restrict__ out, unsigned long long* launches, int kid) {
  count_launch(launches, kid);
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float s_gate[kThreads * kGateIters + 1];
  const int ipr = H / kVec;
  const long long n_items = static_cast<long long>(T) * ipr;
  const long long base = static_cast<long long>(blockIdx.x) * kThreads * kGateIters;
  long long last = base + static_cast<long long>(kThreads) * kGateIters - 1;
  if (last >= n_items) last = n_items - 1;
  const int t_first = static_cast<int>(base / ipr);
  const int n_rows = static_cast<int>(last / ipr) - t_first + 1;

  // first slice: loads issued before the sigmoids are evaluated
  long long item = base + threadIdx.x;
  bool live = item < n_items;
  int t = live ? static_cast<int>(item / ipr) : 0;
  int c0 = live ? static_cast<int>(item % ipr) * kVec : 0;
  float shv[kVec], acc[kVec];
  if (live) {
    Vec8<ShT>::load(sh, static_cast<size_t>(t) * H + c0, shv);
    if (kMode == kCombineGate) routed_sum<EoT, kHasW>(eo, w, rs, t, c0, K, H, acc);
  }
  for (int r = threadIdx.x; r < n_rows; r += kThreads)
    s_gate[r] = sigmoid_f32(__ldg(gl + t_first + r));
  __syncthreads();
  for (int it = 0; it < kGateIters; ++it) {
    if (it > 0) {
      item = base + static_cast<long long>(it) * kThreads + threadIdx.x;
      live = item < n_items;
      if (!live) break;
      t = static_cast<int>(item / ipr);
      c0 = static_cast<int>(item % ipr) * kVec;
      Vec8<ShT>::load(sh, static_cast<size_t>(t) * H + c0, shv);
      if (kMode == kCombineGate) routed_sum<EoT, kHasW>(eo, w, rs, t, c0, K, H, acc);
    }
    if (!live) break;
    const float sg = s_gate[t - t_first];
    float o[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const float g = __fmul_rn(sg, shv[i]);
      // combine-gate: the gated shared term passes through a bf16 rounding before the add
      o[i] = (kMode == kGateOnly) ? g : __fadd_rn(acc[i], round_through_bf16(g));
    }
    Vec8<OutT>::store(out, static_cast<size_t>(t) * H + c0, o);
  }
}

using KernelFn = void (*)(const void*, const float*, const void*, const float*, float, int, int,
                          int, void*, unsigned long long*, int);

// kMode 3 / 4: kCombineGate / kGateOnly reading precomputed sigmoids
template <int kMode, typename EoT, typename ShT, typename OutT>
KernelFn pick_w_sh(bool has_w, bool has_sh) {
  if constexpr (kMode == kGateOnly) {
    return gate_kernel<kMode, EoT, ShT, OutT, false, true>;
  } else if constexpr (kMode == kCombineGate) {
    return has_w ? gate_kernel<kMode, EoT, ShT, OutT, true, true>
                 : gate_kernel<kMode, EoT, ShT, OutT, false, true>;
  } else if constexpr (kMode == kGateOnly + 2) {
    return gate_stream_kernel<kGateOnly, EoT, ShT, OutT, false, true>;
  } else if constexpr (kMode == kCombineGate + 2) {
    return has_w ? gate_stream_kernel<kCombineGate, EoT, ShT, OutT, true, true>
                 : gate_stream_kernel<kCombineGate, EoT, ShT, OutT, false, true>;
  } else {
    if (has_w) return has_sh ? combine_kernel<kMode, EoT, ShT, OutT, true, true>
                             : combine_kernel<kMode, EoT, ShT, OutT, true, false>;
    return has_sh ? combine_kernel<kMode, EoT, ShT, OutT, false, true>
                  : combine_kernel<kMode, EoT, ShT, OutT, false, false>;
  }
}

template <int kMode, typename EoT, typename ShT>
KernelFn pick_out(int out_dt, bool has_w, bool has_sh) {
  return out_dt == MOE_F32 ? pick_w_sh<kMode, EoT, ShT, float>(has_w, has_sh)
                           : pick_w_sh<kMode, EoT, ShT, __nv_bfloat16>(has_w, has_sh);
}

template <int kMode, typename EoT>
KernelFn pick_sh(int sh_dt, int out_dt, bool has_w, bool has_sh) {
  return sh_dt == MOE_F32 ? pick_out<kMode, EoT, float>(out_dt, has_w, has_sh)
                          : pick_out<kMode, EoT, __nv_bfloat16>(out_dt, has_w, has_sh);
}

template <int kMode>
KernelFn pick(int eo_dt, int sh_dt, int out_dt, bool has_w, bool has_sh) {
  return eo_dt == MOE_F32 ? pick_sh<kMode, float>(sh_dt, out_dt, has_w, has_sh)
                          : pick_sh<kMode, __nv_bfloat16>(sh_dt, out_dt, has_w, has_sh);
}

const char* dt_name(int dt) {
  switch (dt) {
    case MOE_F32: return "f32";
    case MOE_BF16: return "bf16";
    case MOE_F16: return "f16";
    default: return "unknown";
  }
}

// dtype refusal: only the f32 and bf16 arms exist; f16 is named in the message
int check_dtype(const char* op, const char* arg, int dt) {
  if (dt == MOE_F32 || dt == MOE_BF16) return MOE_OK;
  return set_error(MOE_ERR_DTYPE,
                   "%s: %s dtype %s (%d) is not implemented; only f32 and bf16 arms exist",
                   op, arg, dt_name(dt), dt);
}

int common_checks(const char* op, int T, int K, int H, bool need_k) {
  if (T < 0) return set_error(MOE_ERR_ARG, "%s: T=%d < 0", op, T);
  if (need_k && (K < 1 || K > 64)) return set_error(MOE_ERR_ARG, "%s: K=%d outside [1, 64]", op, K);
  if (H <= 0) return set_error(MOE_ERR_ARG, "%s: H=%d <= 0", op, H);
  if (H % kVec != 0) return set_error(MOE_ERR_ALIGN, "%s: H=%d is not a multiple of 8", op, H);
  return MOE_OK;
}

int launch(const char* op, KernelFn fn, const void* eo, const float* w, const void* sh,
           const float* gl, float rs, int T, int K, int H, void* out, void* stream, int kid,
           bool fused_sigmoid) {
  if (T == 0) return MOE_OK;
  DeviceDiag diag = device_diag();
  const long long items = static_cast<long long>(T) * (H / kVec);
  const long long per_block =
      fused_sigmoid ? static_cast<long long>(kThreads) * kGateIters : kThreads;
  const long long blocks = (items + per_block - 1) / per_block;
  if (blocks > 0x7fffffffLL) return set_error(MOE_ERR_ARG, "%s: T*H too large", op);
  return launch_status(launch_kernel(fn, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0,
                                     static_cast<cudaStream_t>(stream), nullptr, 0, eo, w, sh,
                                     gl, rs, T, K, H, out, diag.launches, kid),
                       op);
}

// sigmoids of all T tokens into the workspace (then the stream reads them)
int precompute_sigmoids(const char* op, const float* gl, int T, void* workspace, size_t ws_bytes,
                        void* stream, const float** sig) {
  *sig = nullptr;
  if (workspace == nullptr) return MOE_OK;  // fused path: sigmoids inside the gate kernel
  if (ws_bytes < moe_gate_workspace_size(T))
    return set_error(MOE_ERR_WORKSPACE, "%s: workspace of %zu bytes is smaller than %zu", op,
                     ws_bytes, moe_gate_workspace_size(T));
  if (reinterpret_cast<uintptr_t>(workspace) & 15u)
    return set_error(MOE_ERR_ALIGN, "%s: workspace must be 16-byte aligned", op);
  float* s_out = static_cast<float*>(workspace);
  int rc = launch_status(launch_kernel(gate_sigmoid_kernel,
                                       dim3((T + kSigThreads - 1) / kSigThreads),
                                       dim3(kSigThreads), 0, static_cast<cudaStream_t>(stream),
                                       nullptr, 0, gl, T, s_out, device_diag().launches),
                         op);
  if (rc == MOE_OK) *sig = s_out;
  return rc;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_gate_workspace_size(int T) {
  if (T <= 0) return 0;
  return ((static_cast<size_t>(T) * sizeof(float)) + 255) & ~static_cast<size_t>(255);
}

extern "C" int moe_combine(const void* expert_out, int eo_dtype, const float* w,
                           const void* shared, int sh_dtype, float routed_scale, int T, int K,
                           int H, void* out, int out_dtype, void* stream) {
  clear_error();
  const char* op = "moe_combine";
  int rc;
  if ((rc = check_dtype(op, "expert_out", eo_dtype)) != MOE_OK) return rc;
  if ((rc = check_dtype(op, "out", out_dtype)) != MOE_OK) return rc;
  if (shared && (rc = check_dtype(op, "shared", sh_dtype)) != MOE_OK) return rc;
  if ((rc = common_checks(op, T, K, H, true)) != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!expert_out || !out) return set_error(MOE_ERR_ARG, "%s: expert_out/out is NULL", op);
  if (!aligned16(expert_out) || !aligned16(out) || (shared && !aligned16(shared)) ||
      (w && (reinterpret_cast<uintptr_t>(w) & 3u)))
    return set_error(MOE_ERR_ALIGN, "%s: expert_out/shared/out must be 16-byte aligned", op);
  KernelFn fn = pick<kCombine>(eo_dtype, shared ? sh_dtype : MOE_BF16, out_dtype, w != nullptr,
                               shared != nullptr);
  return launch(op, fn, expert_out, w, shared, nullptr, routed_scale, T, K, H, out, stream,
                MOE_KID_COMBINE, false);
}

extern "C" int moe_combine_gate(const void* expert_out, int eo_dtype, const float* w,
                                const void* sd, int sd_dtype, const float* gl, float routed_scale,
                                int T, int K, int H, void* out, int out_dtype, void* workspace,
                                size_t ws_bytes, void* stream) {
  clear_error();
  const char* op = "moe_combine_gate";
  int rc;
  if ((rc = check_dtype(op, "expert_out", eo_dtype)) != MOE_OK) return rc;
  if ((rc = check_dtype(op, "sd", sd_dtype)) != MOE_OK) return rc;
  if ((rc = check_dtype(op, "out", out_dtype)) != MOE_OK) return rc;
  if ((rc = common_checks(op, T, K, H, true)) != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!expert_out || !sd || !gl || !out)
    return set_error(MOE_ERR_ARG, "%s: expert_out/sd/gl/out is NULL", op);
  if (!aligned16(expert_out) || !aligned16(out) || !aligned16(sd) ||
      (reinterpret_cast<uintptr_t>(gl) & 3u) || (w && (reinterpret_cast<uintptr_t>(w) & 3u)))
    return set_error(MOE_ERR_ALIGN, "%s: expert_out/sd/out must be 16-byte aligned", op);
  const float* sig = nullptr;
  if ((rc = precompute_sigmoids(op, gl, T, workspace, ws_bytes, stream, &sig)) != MOE_OK)
    return rc;
  if (sig) {
    KernelFn fn = pick<kCombineGate + 2>(eo_dtype, sd_dtype, out_dtype, w != nullptr, true);
    return launch(op, fn, expert_out, w, sd, sig, routed_scale, T, K, H, out, stream,
                  MOE_KID_COMBINE_GATE, false);
  }
  KernelFn fn = pick<kCombineGate>(eo_dtype, sd_dtype, out_dtype, w != nullptr, true);
  return launch(op, fn, expert_out, w, sd, gl, routed_scale, T, K, H, out, stream,
                MOE_KID_COMBINE_GATE, true);
}

extern "C" int shared_expert_gate(const void* sd, int sd_dtype, const float* gl, int T, int H,
                                  void* out, int out_dtype, void* workspace, size_t ws_bytes,
                                  void* stream) {
  clear_error();
  const char* op = "shared_expert_gate";
  int rc;
  if ((rc = check_dtype(op, "sd", sd_dtype)) != MOE_OK) return rc;
  if ((rc = check_dtype(op, "out", out_dtype)) != MOE_OK) return rc;
  if ((rc = common_checks(op, T, 1, H, false)) != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!sd || !gl || !out) return set_error(MOE_ERR_ARG, "%s: sd/gl/out is NULL", op);
  if (!aligned16(sd) || !aligned16(out) || (reinterpret_cast<uintptr_t>(gl) & 3u))
    return set_error(MOE_ERR_ALIGN, "%s: sd/out must be 16-byte aligned", op);
  const float* sig = nullptr;
  if ((rc = precompute_sigmoids(op, gl, T, workspace, ws_bytes, stream, &sig)) != MOE_OK)
    return rc;
  if (sig) {
    KernelFn fn = pick<kGateOnly + 2>(MOE_BF16, sd_dtype, out_dtype, false, true);
    return launch(op, fn, nullptr, nullptr, sd, sig, 1.0f, T, 1, H, out, stream,
                  MOE_KID_SHARED_GATE, false);
  }
  KernelFn fn = pick<kGateOnly>(MOE_BF16, sd_dtype, out_dtype, false, true);
  return launch(op, fn, nullptr, nullptr, sd, gl, 1.0f, T, 1, H, out, stream,
                MOE_KID_SHARED_GATE, true);
}
