// gemm_common.cuh -- pieces shared by the tcgen05 GEMM kernels of libmoe.so
// (moe_gemm.cu: single-CTA tiles; moe_gemm_pair.cu: CTA-pair tiles): tile
// constants, bounded mbarrier waits, bf16 packing and the host-side tensor
// map and device queries.
#pragma once

#include <stdint.h>

#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace gemm {

constexpr int BM = 128;           // rows per tile on one SM (MMA M of one CTA)
constexpr int BK = 64;            // bf16 per 128-byte swizzled row: K per stage
constexpr int UMMA_K = 16;        // K per tcgen05.mma (kind::f16)
constexpr int kMaxGroups = 1024;
// groups a CTA-pair launch takes (its schedule tables in shared memory); calls
// with more take single-CTA tiles
constexpr int kMaxPairGroups = 512;
// Limit of the waits that drain a CTA's own copies and MMAs before it exits
// (always this long, whatever the pipeline limit is set to).
constexpr unsigned long long kDrainLimitNs = 1000000000ull;

// Bounded mbarrier wait of a pipeline role.  Returns false when this CTA is
// aborting: another role gave up, or this wait ran past `limit_ns` of device
// time, in which case it raises MOE_STATUS_TIMEOUT and the CTA's abort flag.
// Each probe may suspend the thread until the phase completes, for about the
// limit (the probe's suspend-time hint, which the hardware may stretch), and
// the clock and the abort flag are checked after every probe that comes back
// empty, so a wait gives up one to a few limits after it began.  The first
// probe suspends at once: a non-blocking probe in front of it, on every wait
// of the MMA issuer, cost both prefill GEMMs 2 to 4 % of their time.
// kCluster: acquire at cluster scope (the barrier is arrived on by the peer CTA).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* status, unsigned long long limit_ns) {
  const uint32_t hint = static_cast<uint32_t>(limit_ns < 0xFFFFFFFFull ? limit_ns : 0xFFFFFFFFull);
  auto probe = [&]() {
    if (!kCluster) return ptx::mbar_try_wait_hint(bar, parity, hint);
    if (!ptx::mbar_try_wait_cluster(bar, parity, hint)) return false;
    ptx::fence_acquire_cluster();
    return true;
  };
  if (probe()) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (probe()) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      if (status) atomicOr(status, static_cast<unsigned int>(MOE_STATUS_TIMEOUT));
      *abort_flag = 1;
      return false;
    }
  }
}

// The same bounded wait by spinning on the non-blocking probe, for a thread
// whose reaction time is on the critical path (a TMA producer feeding a
// latency-bound stage ring wakes sooner than from a suspending probe); the
// abort flag and the clock are checked every 64 probes.
__device__ __forceinline__ bool wait_bar_spin(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, unsigned int* status,
                                              unsigned long long limit_ns) {
  if (ptx::mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ptx::mbar_test_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      if (status) atomicOr(status, static_cast<unsigned int>(MOE_STATUS_TIMEOUT));
      *abort_flag = 1;
      return false;
    }
  }
}

// Drain wait: polls until the phase completes or kDrainLimitNs passes.
__device__ __forceinline__ void spin_bounded(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer_ns() - t0 < kDrainLimitNs) {
  }
}

// two values rounded to bf16 (nearest even) in one conversion, lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// ------------------------------------------------------------------ host side
// rows x cols bf16 matrix (row-major, cols contiguous) as a TMA map with a box
// of 64 columns x box_rows rows and the 128-byte swizzle
int make_tmap(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows,
              const char* op, const char* what);
// the same for one-byte elements (FP8 codes), unswizzled
int make_tmap_u8(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows,
                 const char* op, const char* what);
int num_sms();
// limit of the pipeline waits in nanoseconds (moe_set_wait_limit_ns)
unsigned long long pipeline_wait_ns();

// the CTA-pair kernels (moe_gemm_pair.cu): arguments already checked by the
// entry points of moe_gemm.cu
// (a_row_gather non-null: routed row r is row a_row_gather[r] / gather_div of
// a_bf16 [a_rows, H], copied by gatherer warps)
int launch_pair_gateup(const char* op, const void* a_bf16, int a_rows,
                       const int32_t* a_row_gather, int gather_div, const void* w13_bf16,
                       const int32_t* group_offsets, int P, int H, int I, int G, void* act_bf16,
                       cudaStream_t stream);
// (staged rows: the launch writes x_perm[r] = x[sorted_pair[r] / K] itself,
// chunk by chunk, and its tiles read x_perm behind per-chunk ready flags)
int launch_pair_gateup_staged(const char* op, const void* x_bf16, int T,
                              const int32_t* sorted_pair, int K, void* x_perm_bf16,
                              const void* w13_bf16, const int32_t* group_offsets, int P, int H,
                              int I, int G, void* act_bf16, int32_t* stage_flags,
                              unsigned int* stage_ctl, cudaStream_t stream);
int launch_pair_down(const char* op, const void* act_bf16, const void* w2_bf16,
                     const int32_t* group_offsets, const float* pair_weight,
                     const int32_t* row_to_pair, int P, int I, int H, int G, void* out_bf16,
                     cudaStream_t stream);

}  // namespace gemm
}  // namespace moe
