// moe_route.cu -- the ungrouped softmax router with top-k and renormalisation
// (vllm.cpp PR #509, "Honest gaps": only the ungrouped softmax router is in
// scope there; grouped, bias-corrected (noaux_tc) and sigmoid forms are refused).
//
// Two kernels: the logits GEMM on tcgen05 tensor cores (moe_gemm.cu, f32
// epilogue with the optional per-expert bias) and a warp-per-token selection
// kernel.  When T x E makes few GEMM tiles, the GEMM splits K into up to 16
// ranges that store partial sums in the workspace, and the selection kernel
// adds them in range order (then the bias) before it selects.  Batches of at
// most kSmallRouterT tokens (decode) take a CUDA-core logits kernel instead,
// one warp per expert and two tokens, which stores finished logits.
// Selection runs on the f32 logits themselves (softmax is monotone), so the
// chosen ids do not depend on exp; the weights use the bit-exact binary32 exp
// and are summed in rank order, so they are bit-identical to the sequential
// definition for the same logits.
#include <math.h>

#include "moe_common.cuh"

namespace moe {

int router_splits(int T, int H, int E);
int launch_router_logits(const void* x, const void* w_router, const float* bias, int T, int H,
                         int E, float* logits, int ksplit, cudaStream_t stream);

namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxGroups = 64;   // n_group limit of the grouped router

// The router forms beyond ungrouped softmax (selection bias, sigmoid scores,
// expert groups); all off: the plain router.
struct RouteEx {
  const float* select_bias;  // [E] or null: added to the scores for the choice only
  int scoring;               // 0 softmax (choice on the logits), 1 sigmoid
  int n_group;               // contiguous expert groups (1: none)
  int topk_group;            // groups that stay eligible
  int group_score;           // 0: a group's best key; 1: its two best keys added
};

// Order-preserving 32-bit key of a logit for the selection: larger key = ranks
// higher.  -0 and +0 share a key (they compare equal), every NaN gets key 0
// (below -inf, whose key is 0x007FFFFF), and equal keys go to the lower expert
// id -- the order "descending value, ties to the lower id, NaN last".
__device__ __forceinline__ uint32_t rank_key(float v) {
  if (v != v) return 0u;
  uint32_t u = __float_as_uint(v);
  if ((u & 0x7FFFFFFFu) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// shared-expert gate logit of token t: a plain f32 dot product of x[t] and wsg
// (one warp; the result from lane 0)
__device__ __forceinline__ void shared_gate_logit(const uint16_t* __restrict__ x,
                                                  const uint16_t* __restrict__ wsg, int H, int t,
                                                  int lane, float* __restrict__ gl_out) {
  const uint16_t* xr = x + static_cast<size_t>(t) * H;
  float acc = 0.0f;
  for (int h = lane * 8; h < H; h += 256) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(xr + h));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(wsg + h));
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc += __uint_as_float(aw[q] << 16) * __uint_as_float(bw[q] << 16);
      acc += __uint_as_float(aw[q] & 0xFFFF0000u) * __uint_as_float(bw[q] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) gl_out[t] = acc;
}

// Router logits of small batches (T <= kSmallRouterT) on CUDA cores: warp w
// owns expert w % E and the kTokWarp tokens kTokWarp (w / E), ...  Lane l owns
// the 8-element chunks l, l + 32, ... of H.  For each block of kChunks chunks
// the lane loads the expert's weights and the tokens' inputs all at once (one
// memory round trip), and adds each token's products into its f32 sum by fused
// multiply-adds in index order.  The warp adds its 32 lane sums by a
// butterfly, and lane 0 adds the bias and stores the logits.  At these sizes
// the tensor-core GEMM is a latency chain (a 128-row token tile, a K split
// whose partial sums the selection adds back); here the E x T/kTokWarp warps
// each wait for one round trip per 2048 elements of H, the router weights come
// from L2 after their first read, and x stays in L2.
constexpr int kSmallRouterT = 64;
constexpr int kLogitWarps = 8;
constexpr int kChunks = 8;     // 16-byte chunks per lane and block: 2048 of H
constexpr int kTokWarp = 2;    // tokens per warp

__global__ void __launch_bounds__(kLogitWarps * 32)
router_logits_small(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr,
                    const float* __restrict__ bias, int T, int H, int E,
                    float* __restrict__ logits, unsigned long long* launches) {
  count_launch(launches, MOE_KID_ROUTE_LOGITS);
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * kLogitWarps + static_cast<int>(threadIdx.x >> 5);
  const int e = w % E;
  const int t0 = (w / E) * kTokWarp;
  if (t0 >= T) return;
  const int nt = min(kTokWarp, T - t0);
  const uint16_t* wrow = wr + static_cast<size_t>(e) * H;
  float sum[kTokWarp];
#pragma unroll
  for (int u = 0; u < kTokWarp; ++u) sum[u] = 0.0f;
  for (int hb = 0; hb < H; hb += 256 * kChunks) {
    uint4 w4[kChunks];
    uint4 x4[kTokWarp][kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const int h = hb + 256 * c + 8 * lane;
      w4[c] = h < H ? __ldg(reinterpret_cast<const uint4*>(wrow + h)) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < kTokWarp; ++u)
        x4[u][c] = (h < H && u < nt)
                       ? __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + u) * H + h))
                       : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kTokWarp; ++u)
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const uint32_t xw[4] = {x4[u][c].x, x4[u][c].y, x4[u][c].z, x4[u][c].w};
        const uint32_t ww[4] = {w4[c].x, w4[c].y, w4[c].z, w4[c].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          sum[u] = __fmaf_rn(__uint_as_float(xw[q] << 16), __uint_as_float(ww[q] << 16), sum[u]);
          sum[u] = __fmaf_rn(__uint_as_float(xw[q] & 0xFFFF0000u),
                             __uint_as_float(ww[q] & 0xFFFF0000u), sum[u]);
        }
      }
  }
  const float b = bias ? __ldg(bias + e) : 0.0f;
#pragma unroll
  for (int u = 0; u < kTokWarp; ++u) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum[u] += __shfl_xor_sync(0xffffffffu, sum[u], o);
    if (lane == 0 && u < nt)
      logits[static_cast<size_t>(t0 + u) * E + e] = bias ? __fadd_rn(sum[u], b) : sum[u];
  }
}

// Does key a (expert ia) rank above key b (expert ib): larger first, ties to
// the lower index, NaN last (the order of rank_key).
__device__ __forceinline__ bool ranks_above(float a, int ia, float b, int ib) {
  const uint32_t ka = rank_key(a), kb = rank_key(b);
  return ka > kb || (ka == kb && ia < ib);
}

// The warp's top-K of one token for the plain router (at most 8 entries a lane):
// lane j < K receives the j-th pick, its id and the value it reports.  Each
// lane sorts its entries once by the selection order (key descending, ties to
// the lower id); every pick then compares only the lanes' heads, and the
// winning lane shifts its list.  Entries past E get key 0 and an id >= E, so
// they rank below every expert (a NaN expert, also key 0, wins the tie on its
// lower id) and are never reached, since K <= E.
template <int kPerLane>
__device__ __forceinline__ void select_sorted_heads(const uint32_t (&key)[kPerLane],
                                                    const float (&sc)[kPerLane], int E, int K,
                                                    int lane, float& my_sel, int& my_id) {
  uint32_t hk[kPerLane];
  uint32_t hid[kPerLane];
  float hv[kPerLane];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int e = lane + 32 * i;
    hk[i] = e < E ? key[i] : 0u;
    hid[i] = static_cast<uint32_t>(e);
    hv[i] = sc[i];
  }
  // odd-even transposition sort: kPerLane rounds of neighbour exchanges
#pragma unroll
  for (int r = 0; r < kPerLane; ++r)
#pragma unroll
    for (int i = r & 1; i + 1 < kPerLane; i += 2) {
      const bool sw = hk[i + 1] > hk[i] || (hk[i + 1] == hk[i] && hid[i + 1] < hid[i]);
      const uint32_t k0 = hk[i], i0 = hid[i];
      const float v0 = hv[i];
      hk[i] = sw ? hk[i + 1] : k0;
      hid[i] = sw ? hid[i + 1] : i0;
      hv[i] = sw ? hv[i + 1] : v0;
      hk[i + 1] = sw ? k0 : hk[i + 1];
      hid[i + 1] = sw ? i0 : hid[i + 1];
      hv[i + 1] = sw ? v0 : hv[i + 1];
    }
  for (int j = 0; j < K; ++j) {
    const uint32_t top = __reduce_max_sync(0xffffffffu, hk[0]);
    const uint32_t win = __reduce_min_sync(0xffffffffu, hk[0] == top ? hid[0] : 0xFFFFFFFFu);
    const int owner = static_cast<int>(win & 31u);
    const float wv = __shfl_sync(0xffffffffu, hv[0], owner);
    if (owner == lane) {
#pragma unroll
      for (int i = 0; i + 1 < kPerLane; ++i) {
        hk[i] = hk[i + 1];
        hid[i] = hid[i + 1];
        hv[i] = hv[i + 1];
      }
      hk[kPerLane - 1] = 0u;
      hid[kPerLane - 1] = 0xFFFFFFFFu;
    }
    if (lane == j) {
      my_sel = wv;
      my_id = static_cast<int>(win);
    }
  }
}

// One warp selects the top-K of one token.  The weights' exps are then
// evaluated by the whole block, one (token, rank) pair per thread, so that
// they run on full warps (a warp instruction costs the same with 8 or 32
// lanes active).
// kEx: the extended forms of RouteEx.  Each lane turns its logits into scores
// (sigmoid_f32 for sigmoid scoring) and keys (score + selection bias); the keys
// go to shared memory, where lane g scores expert group g; the warp picks the
// topk_group best groups, and the expert choice skips experts of the others.
template <int kPerLane, bool kEx>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
topk_kernel(const float* __restrict__ logits, int n_part, const float* __restrict__ bias,
            float* __restrict__ logits_out, int T, int E, int K, int renormalize,
            const uint16_t* __restrict__ x, const uint16_t* __restrict__ wsg, int H,
            int32_t* __restrict__ ids, float* __restrict__ w, float* __restrict__ gl_out,
            unsigned long long* launches, RouteEx rx) {
  count_launch(launches, MOE_KID_ROUTE_TOPK);
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float s_sel[kWarpsPerBlock][32];
  __shared__ float s_ex[kWarpsPerBlock][32];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int t = blockIdx.x * kWarpsPerBlock + wib;
  const bool live = t < T;
  float v[kPerLane];
  float my_sel = 0.0f;
  int my_id = 0;
  if (live) {
    // n_part K-range partial sums of each logit, added in range order, then the
    // bias.  The loads of kQ ranges (at most 16, the largest split) are issued
    // before their additions, so that a K split costs a few memory round trips
    // rather than one per range.
    constexpr int kLoads = kEx ? 16 : 32;  // loads in flight per lane
    constexpr int kQ = kPerLane >= kLoads ? 1 : (kLoads / kPerLane > 16 ? 16 : kLoads / kPerLane);
    const float* row = logits + static_cast<size_t>(t) * E;
    const size_t slab = static_cast<size_t>(T) * E;
    if (n_part == 1) {
      // no K split (prefill-sized batches): one load per logit
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldg(row + e) : 0.0f;
      }
    } else {
      for (int q0 = 0; q0 < n_part; q0 += kQ) {
        float part[kQ][kPerLane];
#pragma unroll
        for (int j = 0; j < kQ; ++j)
#pragma unroll
          for (int i = 0; i < kPerLane; ++i) {
            const int e = lane + 32 * i;
            part[j][i] = (q0 + j < n_part && e < E) ? __ldg(row + (q0 + j) * slab + e) : 0.0f;
          }
#pragma unroll
        for (int j = 0; j < kQ; ++j)
          if (q0 + j < n_part)
#pragma unroll
            for (int i = 0; i < kPerLane; ++i)
              v[i] = q0 + j == 0 ? part[j][i] : __fadd_rn(v[i], part[j][i]);
      }
    }
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        if (bias) v[i] = __fadd_rn(v[i], __ldg(bias + e));
        if (logits_out) logits_out[static_cast<size_t>(t) * E + e] = v[i];
      } else {
        v[i] = 0.0f;
      }
    }
    uint32_t key[kPerLane];
    float sc[kPerLane];      // what a chosen expert reports: its logit, or its sigmoid score
    uint32_t taken = 0;
    if (!kEx) {
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        key[i] = rank_key(v[i]);
        sc[i] = v[i];
      }
    } else {
      extern __shared__ float s_dyn[];
      float* s_key = s_dyn + static_cast<size_t>(wib) * E;
      float* s_gsc = s_dyn + static_cast<size_t>(kWarpsPerBlock) * E + wib * kMaxGroups;
      unsigned char* s_gok = reinterpret_cast<unsigned char*>(
                                 s_dyn + static_cast<size_t>(kWarpsPerBlock) * (E + kMaxGroups)) +
                             wib * kMaxGroups;
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        sc[i] = 0.0f;
        float kv = 0.0f;
        if (e < E) {
          sc[i] = rx.scoring == 1 ? sigmoid_f32(v[i]) : v[i];
          kv = rx.select_bias ? __fadd_rn(sc[i], __ldg(rx.select_bias + e)) : sc[i];
          s_key[e] = kv;
        }
        key[i] = rank_key(kv);
      }
      __syncwarp();
      // group scores: lane g scans group g in expert order
      const int gs = E / rx.n_group;
      for (int g = lane; g < rx.n_group; g += 32) {
        int b0 = -1, b1 = -1;
        for (int e = g * gs; e < g * gs + gs; ++e) {
          if (b0 < 0 || ranks_above(s_key[e], e, s_key[b0], b0)) {
            b1 = b0;
            b0 = e;
          } else if (b1 < 0 || ranks_above(s_key[e], e, s_key[b1], b1)) {
            b1 = e;
          }
        }
        s_gsc[g] = rx.group_score == 0 ? s_key[b0] : __fadd_rn(s_key[b0], s_key[b1]);
        s_gok[g] = 0;
      }
      __syncwarp();
      // the topk_group best groups (descending score, ties to the lower group)
      constexpr int kGroupsPerLane = kMaxGroups / 32;
      uint32_t gtaken = 0;
      for (int j = 0; j < rx.topk_group; ++j) {
        uint32_t bk = 0u, bid = 0xFFFFFFFFu;
#pragma unroll
        for (int q = 0; q < kGroupsPerLane; ++q) {
          const int g = lane + 32 * q;
          if (g < rx.n_group && !((gtaken >> q) & 1u)) {
            const uint32_t k = rank_key(s_gsc[g]);
            if (bid == 0xFFFFFFFFu || k > bk) {
              bk = k;
              bid = static_cast<uint32_t>(g);
            }
          }
        }
        const uint32_t top = __reduce_max_sync(0xffffffffu, bid == 0xFFFFFFFFu ? 0u : bk);
        const uint32_t cand = (bid != 0xFFFFFFFFu && bk == top) ? bid : 0xFFFFFFFFu;
        const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
        if (win != 0xFFFFFFFFu && static_cast<int>(win & 31u) == lane) {
          gtaken |= 1u << (win >> 5);
          s_gok[win] = 1;
        }
        __syncwarp();
      }
      // experts of the other groups are never chosen
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !s_gok[e / gs]) taken |= 1u << i;
      }
    }
    if (!kEx && kPerLane <= 8) {
      select_sorted_heads<kPerLane>(key, sc, E, K, lane, my_sel, my_id);
    } else {
    for (int j = 0; j < K; ++j) {
      // this lane's best untaken entry (ascending id, so ties keep the lower id)
      uint32_t bk = 0u, bid = 0xFFFFFFFFu;
      float bv = 0.0f;
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (bid == 0xFFFFFFFFu || key[i] > bk)) {
          bk = key[i];
          bid = static_cast<uint32_t>(e);
          bv = sc[i];
        }
      }
      // the warp's best: highest key, then lowest id among the lanes holding it
      const uint32_t top = __reduce_max_sync(0xffffffffu, bid == 0xFFFFFFFFu ? 0u : bk);
      const uint32_t cand = (bid != 0xFFFFFFFFu && bk == top) ? bid : 0xFFFFFFFFu;
      const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
      const int owner = static_cast<int>(win & 31u);
      const float wv = __shfl_sync(0xffffffffu, bv, owner);
      if (owner == lane) taken |= 1u << (win >> 5);
      if (lane == j) {
        my_sel = wv;
        my_id = static_cast<int>(win);
      }
    }
    }
    s_sel[wib][lane] = my_sel;
  }
  __syncthreads();
  if (kEx && rx.scoring == 1) {
    // sigmoid scores: w_j = s_j / ((s_0 + s_1) + ...) or s_j
    if (!live) return;
    float den = 0.0f;
    for (int j = 0; j < K; ++j) den = __fadd_rn(den, s_sel[wib][j]);
    if (lane < K) {
      ids[static_cast<size_t>(t) * K + lane] = my_id;
      w[static_cast<size_t>(t) * K + lane] = renormalize ? __fdiv_rn(my_sel, den) : my_sel;
    }
    if (wsg != nullptr) shared_gate_logit(x, wsg, H, t, lane, gl_out);
    return;
  }
  // e_j = exp(l_j - l_0) for every (token, rank) pair of the block
  const int n_live = min(kWarpsPerBlock, T - static_cast<int>(blockIdx.x) * kWarpsPerBlock);
  for (int q = threadIdx.x; q < n_live * K; q += blockDim.x) {
    const int tt = q / K, j = q - tt * K;
    const float d = __fsub_rn(s_sel[tt][j], s_sel[tt][0]);
    // rank 0: d is +0 for a finite top logit and exp(+0) is exactly 1
    s_ex[tt][j] = (j == 0 && d == 0.0f) ? 1.0f : exp_f32(d);
  }
  __syncthreads();
  if (!live) return;
  const float m = s_sel[wib][0];
  float S = 0.0f;
  float ex = 0.0f;
  if (renormalize) {
    for (int j = 0; j < K; ++j) S = __fadd_rn(S, s_ex[wib][j]);
    if (lane < K) ex = s_ex[wib][lane];
  } else {
    float ev[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) ev[i] = exp_f32(__fsub_rn(v[i], m));
#pragma unroll
    for (int i = 0; i < kPerLane; ++i)
      for (int l = 0; l < 32; ++l) {
        const float term = __shfl_sync(0xffffffffu, ev[i], l);
        if (l + 32 * i < E) S = __fadd_rn(S, term);
      }
    if (lane < K) ex = s_ex[wib][lane];
  }
  if (lane < K) {
    ids[static_cast<size_t>(t) * K + lane] = my_id;
    w[static_cast<size_t>(t) * K + lane] = __fdiv_rn(ex, S);
  }
  if (wsg != nullptr) shared_gate_logit(x, wsg, H, t, lane, gl_out);
}

using TopkFn = void (*)(const float*, int, const float*, float*, int, int, int, int,
                        const uint16_t*, const uint16_t*, int, int32_t*, float*, float*,
                        unsigned long long*, RouteEx);

template <bool kEx>
TopkFn pick_topk(int E) {
  if (E <= 32) return topk_kernel<1, kEx>;
  if (E <= 64) return topk_kernel<2, kEx>;
  if (E <= 128) return topk_kernel<4, kEx>;
  if (E <= 256) return topk_kernel<8, kEx>;
  if (E <= 512) return topk_kernel<16, kEx>;
  return topk_kernel<32, kEx>;
}

size_t logits_bytes(int T, int E) {
  return ((static_cast<size_t>(T) * E * sizeof(float)) + 255) & ~static_cast<size_t>(255);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_route_topk_workspace_size(int T, int E, int K) {
  (void)K;
  if (T <= 0 || E <= 0) return 0;
  // the largest K split any H allows (the split never exceeds H / 64 ranges)
  return logits_bytes(T, E) * static_cast<size_t>(router_splits(T, 1 << 20, E));
}

namespace moe {
namespace {

int route_impl(const char* op, const void* x_bf16, const void* w_router_bf16,
               const float* logit_bias, const void* w_shared_gate_bf16, const float* logits_in,
               int T, int H, int E, int K, int renormalize, const RouteEx& ex,
               int32_t* topk_ids, float* topk_w, float* logits_out, float* gate_logit_out,
               void* workspace, size_t ws_bytes, void* stream) {
  if (T < 0) return set_error(MOE_ERR_ARG, "%s: T=%d < 0", op, T);
  if (E < 1 || E > 1024) return set_error(MOE_ERR_ARG, "%s: E=%d outside [1, 1024]", op, E);
  if (K < 1 || K > E || K > 32)
    return set_error(MOE_ERR_ARG, "%s: K=%d outside [1, min(E, 32)]", op, K);
  if (renormalize != 0 && renormalize != 1)
    return set_error(MOE_ERR_ARG, "%s: renormalize must be 0 or 1", op);
  const bool need_x = logits_in == nullptr || w_shared_gate_bf16 != nullptr;
  if (need_x && (H <= 0 || H % 8 != 0))
    return set_error(MOE_ERR_ALIGN, "%s: H=%d must be a positive multiple of 8", op, H);
  if (T == 0) return MOE_OK;
  if (!topk_ids || !topk_w) return set_error(MOE_ERR_ARG, "%s: topk_ids/topk_w is NULL", op);
  if (!logits_in && (!x_bf16 || !w_router_bf16))
    return set_error(MOE_ERR_ARG, "%s: x/w_router is NULL and no logits_in given", op);
  if (w_shared_gate_bf16 && (!x_bf16 || !gate_logit_out))
    return set_error(MOE_ERR_ARG, "%s: w_shared_gate needs x and gate_logit_out", op);
  if ((x_bf16 && !aligned16(x_bf16)) || (w_router_bf16 && !aligned16(w_router_bf16)) ||
      (w_shared_gate_bf16 && !aligned16(w_shared_gate_bf16)))
    return set_error(MOE_ERR_ALIGN, "%s: x/w_router/w_shared_gate must be 16-byte aligned", op);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float* logits = logits_in;
  int n_part = 1;
  const float* part_bias = nullptr;   // added by the selection kernel after a K split
  float* sel_logits_out = nullptr;    // written by the selection kernel after a K split
  if (!logits) {
    if (workspace && !aligned16(workspace))
      return set_error(MOE_ERR_ALIGN, "%s: workspace must be 16-byte aligned", op);
    // K split into ranges of partial sums in the workspace, as many as it holds
    const size_t slab = static_cast<size_t>(T) * E * sizeof(float);
    // small batches: finished logits from the CUDA-core kernel, no K split
    const bool small = T <= kSmallRouterT;
    int splits = small ? 1 : router_splits(T, H, E);
    const size_t fit = workspace ? ws_bytes / slab : 0;
    if (static_cast<size_t>(splits) > fit) splits = static_cast<int>(fit);
    float* dst = logits_out;
    if (splits > 1) {
      dst = static_cast<float*>(workspace);
      n_part = splits;
      part_bias = logit_bias;
      sel_logits_out = logits_out;
    } else if (!dst) {
      if (!workspace || ws_bytes < logits_bytes(T, E))
        return set_error(MOE_ERR_WORKSPACE,
                         "%s: workspace of %zu bytes is smaller than the %zu bytes of logits", op,
                         ws_bytes, logits_bytes(T, E));
      dst = static_cast<float*>(workspace);
    }
    int rc;
    if (small) {
      rc = launch_status(
          launch_kernel(router_logits_small,
                        dim3((E * ((T + kTokWarp - 1) / kTokWarp) + kLogitWarps - 1) / kLogitWarps),
                        dim3(kLogitWarps * 32), 0, s, nullptr, 0,
                        static_cast<const uint16_t*>(x_bf16),
                        static_cast<const uint16_t*>(w_router_bf16), logit_bias, T, H, E, dst,
                        device_diag().launches),
          op);
    } else {
      rc = launch_router_logits(x_bf16, w_router_bf16, logit_bias, T, H, E, dst, n_part, s);
    }
    if (rc != MOE_OK) return rc;
    logits = dst;
  } else if (logits_out && logits_out != logits_in) {
    if (cudaMemcpyAsync(logits_out, logits_in, static_cast<size_t>(T) * E * sizeof(float),
                        cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "%s: copy of logits failed: %s", op,
                       cudaGetErrorString(cudaGetLastError()));
  }
  DeviceDiag diag = device_diag();
  const int blocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const bool extended = ex.scoring != 0 || ex.n_group != 1 || ex.select_bias != nullptr;
  const size_t smem = extended ? static_cast<size_t>(kWarpsPerBlock) *
                                     ((E + kMaxGroups) * sizeof(float) + kMaxGroups)
                               : 0;
  return launch_status(
      launch_kernel(extended ? pick_topk<true>(E) : pick_topk<false>(E), dim3(blocks),
                    dim3(kWarpsPerBlock * 32), smem, s, nullptr, 0, logits, n_part, part_bias,
                    sel_logits_out, T, E, K, renormalize, static_cast<const uint16_t*>(x_bf16),
                    static_cast<const uint16_t*>(w_shared_gate_bf16), H, topk_ids, topk_w,
                    gate_logit_out, diag.launches, ex),
      op);
}

}  // namespace
}  // namespace moe

extern "C" int moe_route_topk(const void* x_bf16, const void* w_router_bf16,
                              const float* logit_bias, const void* w_shared_gate_bf16,
                              const float* logits_in, int T, int H, int E, int K, int renormalize,
                              int scoring, int n_group, int32_t* topk_ids, float* topk_w,
                              float* logits_out, float* gate_logit_out, void* workspace,
                              size_t ws_bytes, void* stream) {
  clear_error();
  const char* op = "moe_route_topk";
  if (scoring != 0)
    return set_error(MOE_ERR_UNSUPPORTED,
                     "%s: scoring=%d is not implemented here; only ungrouped softmax (0) is "
                     "(sigmoid scores: moe_route_topk_ex)", op, scoring);
  if (n_group != 1)
    return set_error(MOE_ERR_UNSUPPORTED,
                     "%s: grouped routing (n_group=%d) is not implemented here; only n_group=1 "
                     "is (expert groups: moe_route_topk_ex)", op, n_group);
  const RouteEx ex{nullptr, 0, 1, 1, 0};
  return route_impl(op, x_bf16, w_router_bf16, logit_bias, w_shared_gate_bf16, logits_in, T, H,
                    E, K, renormalize, ex, topk_ids, topk_w, logits_out, gate_logit_out,
                    workspace, ws_bytes, stream);
}

extern "C" int moe_route_topk_ex(const void* x_bf16, const void* w_router_bf16,
                                 const float* logit_bias, const float* select_bias,
                                 const void* w_shared_gate_bf16, const float* logits_in, int T,
                                 int H, int E, int K, int renormalize, int scoring, int n_group,
                                 int topk_group, int group_score, int32_t* topk_ids,
                                 float* topk_w, float* logits_out, float* gate_logit_out,
                                 void* workspace, size_t ws_bytes, void* stream) {
  clear_error();
  const char* op = "moe_route_topk_ex";
  if (scoring != 0 && scoring != 1)
    return set_error(MOE_ERR_UNSUPPORTED, "%s: scoring=%d is not 0 (softmax) or 1 (sigmoid)", op,
                     scoring);
  if (select_bias && scoring != 1)
    return set_error(MOE_ERR_UNSUPPORTED,
                     "%s: a selection bias is implemented for sigmoid scores only", op);
  if (E < 1 || E > 1024) return set_error(MOE_ERR_ARG, "%s: E=%d outside [1, 1024]", op, E);
  if (n_group < 1 || n_group > kMaxGroups || E % n_group != 0)
    return set_error(MOE_ERR_ARG, "%s: n_group=%d must divide E=%d and be at most %d", op,
                     n_group, E, kMaxGroups);
  if (topk_group < 1 || topk_group > n_group)
    return set_error(MOE_ERR_ARG, "%s: topk_group=%d outside [1, n_group=%d]", op, topk_group,
                     n_group);
  if (group_score != 0 && group_score != 1)
    return set_error(MOE_ERR_ARG, "%s: group_score=%d is not 0 (best) or 1 (two best)", op,
                     group_score);
  if (group_score == 1 && E / n_group < 2)
    return set_error(MOE_ERR_ARG, "%s: two-best group scores need groups of two experts", op);
  if (K > topk_group * (E / n_group))
    return set_error(MOE_ERR_ARG, "%s: K=%d exceeds the %d experts of the eligible groups", op,
                     K, topk_group * (E / n_group));
  if (select_bias && (reinterpret_cast<uintptr_t>(select_bias) & 3u))
    return set_error(MOE_ERR_ALIGN, "%s: select_bias must be 4-byte aligned", op);
  const RouteEx ex{select_bias, scoring, n_group, topk_group, group_score};
  return route_impl(op, x_bf16, w_router_bf16, logit_bias, w_shared_gate_bf16, logits_in, T, H,
                    E, K, renormalize, ex, topk_ids, topk_w, logits_out, gate_logit_out,
                    workspace, ws_bytes, stream);
}
