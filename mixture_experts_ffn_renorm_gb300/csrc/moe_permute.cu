// moe_permute.cu -- tokens into expert-contiguous order: a deterministic,
// stable counting sort of the P = T*K (token, slot) pairs by expert.  The
// expert path keeps one bf16 row per routed pair, P rows of H (vllm.cpp PR #509
// review, finding 2), and the expert GEMM is grouped over expert ids (PR #523,
// "What changed").
//
//   count   one warp per chunk of 512 pairs: per-chunk expert histogram in
//           shared memory (bad ids raise MOE_STATUS_BAD_ID and are skipped)
//   scan    one block: per expert (one warp each), exclusive scan of the chunk
//           counts in chunk order (up to 128 experts and 128 chunks: a warp's
//           four experts loaded at once and scanned interleaved); then the
//           exclusive scan over experts -> expert_offsets
//   place   one warp per chunk again, 32 pairs at a time in pair order: the
//           rank of a pair among equal experts of its step comes from one
//           ballot per id bit, so rows inside an expert ascend with p
//   gather  (optional) x_perm[row] = x[sorted_pair[row] / K], 16 bytes a thread
//           (zeros for a row outside x)
// Up to kSmallChunks chunks whose histograms fit in 48 KB of shared memory
// (decode batches; the large layer's 16384 pairs over 256 experts) count, scan
// and place run in one block (permute_small): the same steps, one launch
// instead of three.
// Everything is a function of the ids alone: no atomics decide an order.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kChunk = 512;  // pairs per warp
constexpr int kWarps = 2;    // warps (chunks) per block: many small blocks spread the sort
constexpr int kIdsPerLane = kChunk / 32;

// A chunk's ids into registers, lane-strided (pair p0 + lane + 32 k in slot k),
// every load in flight at once; pairs at or past p1 read as -1.
__device__ __forceinline__ void load_chunk_ids(const int32_t* __restrict__ ids, int p0, int p1,
                                               int lane, int (&v)[kIdsPerLane]) {
#pragma unroll
  for (int k = 0; k < kIdsPerLane; ++k) {
    const int p = p0 + lane + 32 * k;
    v[k] = p < p1 ? __ldg(ids + p) : -1;
  }
}

// Histogram of a chunk's ids into the warp's shared counts; out-of-range ids
// are skipped and reported through the status word.
__device__ __forceinline__ void count_chunk_ids(const int (&v)[kIdsPerLane], int p0, int p1,
                                                int E, int lane, int32_t* h,
                                                unsigned int* status) {
  bool bad = false;
#pragma unroll
  for (int k = 0; k < kIdsPerLane; ++k) {
    const int e = v[k];
    if (p0 + lane + 32 * k >= p1) continue;
    if (e >= 0 && e < E) atomicAdd(h + e, 1);
    else bad = true;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0 && status)
    atomicOr(status, static_cast<unsigned int>(MOE_STATUS_BAD_ID));
}

// The lanes of the warp holding the same expert id as this lane (among the
// valid ones): one ballot per bit of the id, each narrowing the set to the
// lanes that agree on that bit.  A fixed ceil(log2 E) ballots, where
// __match_any_sync slows down with the number of distinct ids in the warp.
__device__ __forceinline__ uint32_t same_expert_lanes(int e, bool valid, int id_bits) {
  uint32_t peers = __ballot_sync(0xffffffffu, valid);
  for (int b = 0; b < id_bits; ++b) {
    const bool bit = (e >> b) & 1;
    const uint32_t m = __ballot_sync(0xffffffffu, bit);
    peers &= bit ? m : ~m;
  }
  return peers;
}

// Stable placement of a chunk: cnt[e] holds the first row of expert e still
// free for this chunk; 32 pairs at a time in pair order, the rank of a pair
// among equal experts of its step from the lanes that share its id.
__device__ __forceinline__ void place_chunk_ids(const int (&v)[kIdsPerLane], int p0, int p1,
                                                int E, int lane, int32_t* cnt,
                                                int32_t* __restrict__ sorted_pair,
                                                int32_t* __restrict__ pair_to_row) {
  const int id_bits = E > 1 ? 32 - __clz(E - 1) : 0;
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int k = 0; k < kIdsPerLane; ++k) {
    if (p0 + 32 * k >= p1) break;                // uniform across the warp
    const int p = p0 + lane + 32 * k;
    const int e = v[k];
    const bool valid = p < p1 && e >= 0 && e < E;
    const uint32_t peers = same_expert_lanes(e, valid, id_bits);
    int row = 0;
    if (valid) row = cnt[e] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid && (peers & lt_mask) == 0) cnt[e] += __popc(peers);  // lowest lane of the group
    __syncwarp();
    if (valid) {
      sorted_pair[row] = p;
      pair_to_row[p] = row;
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32)
permute_count(const int32_t* __restrict__ ids, int P, int E, int n_chunks,
              int32_t* __restrict__ hist, unsigned int* status, unsigned long long* launches) {
  count_launch(launches, MOE_KID_PERMUTE_COUNT);
  grid_dep_wait();
  grid_dep_launch();
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kWarps + warp;
  int32_t* h = sh + warp * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  if (c < n_chunks) {
    const int p0 = c * kChunk, p1 = min(P, p0 + kChunk);
    int v[kIdsPerLane];
    load_chunk_ids(ids, p0, p1, lane, v);
    count_chunk_ids(v, p0, p1, E, lane, h, status);
    __syncwarp();
    for (int e = lane; e < E; e += 32) hist[static_cast<size_t>(e) * n_chunks + c] = h[e];
  }
}

// hist is laid out [E][n_chunks]: one warp scans one expert's chunk counts
// (coalesced, all loads of a batch in flight), then the block scans the
// per-expert totals into expert_offsets.
__global__ void __launch_bounds__(1024)
permute_scan(int32_t* __restrict__ hist, int E, int n_chunks, int32_t* __restrict__ offsets,
             unsigned long long* launches) {
  count_launch(launches, MOE_KID_PERMUTE_SCAN);
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int32_t tot[1024];
  __shared__ int32_t warp_sum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kBatch = 8;
  const int epw = (E + 31) >> 5;           // experts per warp
  const int nb = (n_chunks + 31) >> 5;     // 32-chunk batches per expert
  if (epw <= 4 && nb <= 4) {
    // Up to 128 experts and 128 chunks (the prefill batch): all of a warp's
    // counts are loaded at once, one round trip, and its experts' scans run
    // interleaved, four independent shuffle chains.
    int v[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int e = warp + 32 * a, c = 32 * b + lane;
        v[a][b] = (a < epw && e < E && b < nb && c < n_chunks)
                      ? hist[static_cast<size_t>(e) * n_chunks + c] : 0;
      }
    int carry[4] = {0, 0, 0, 0};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      int incl[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) incl[a] = v[a][b];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1)
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const int u = __shfl_up_sync(0xffffffffu, incl[a], o);
          if (lane >= o) incl[a] += u;
        }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int e = warp + 32 * a, c = 32 * b + lane;
        if (a < epw && e < E && b < nb && c < n_chunks)
          hist[static_cast<size_t>(e) * n_chunks + c] = carry[a] + incl[a] - v[a][b];
        carry[a] += __shfl_sync(0xffffffffu, incl[a], 31);
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int e = warp + 32 * a;
      if (lane == 0 && a < epw && e < E) tot[e] = carry[a];
    }
  } else {
  for (int e = warp; e < E; e += 32) {
    int32_t* row = hist + static_cast<size_t>(e) * n_chunks;
    int carry = 0;
    for (int c0 = 0; c0 < n_chunks; c0 += 32 * kBatch) {
      int v[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int c = c0 + b * 32 + lane;
        v[b] = c < n_chunks ? row[c] : 0;
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        int incl = v[b];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += u;
        }
        const int c = c0 + b * 32 + lane;
        if (c < n_chunks) row[c] = carry + incl - v[b];
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (lane == 0) tot[e] = carry;
  }
  }
  __syncthreads();
  // block-wide exclusive scan of the per-expert totals (E <= 1024)
  const int run = tid < E ? tot[tid] : 0;
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int ws = warp_sum[lane];
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    warp_sum[lane] = wi - ws;
  }
  __syncthreads();
  const int excl = warp_sum[warp] + incl - run;
  if (tid < E) offsets[tid] = excl;
  if (tid == E - 1) offsets[E] = excl + run;
}

__global__ void __launch_bounds__(kWarps * 32)
permute_place(const int32_t* __restrict__ ids, int P, int E, int n_chunks,
              const int32_t* __restrict__ hist, const int32_t* __restrict__ offsets,
              int32_t* __restrict__ sorted_pair, int32_t* __restrict__ pair_to_row,
              unsigned long long* launches) {
  count_launch(launches, MOE_KID_PERMUTE_PLACE);
  grid_dep_wait();
  grid_dep_launch();
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kWarps + warp;
  if (c >= n_chunks) return;
  const int p0 = c * kChunk, p1 = min(P, p0 + kChunk);
  int v[kIdsPerLane];
  load_chunk_ids(ids, p0, p1, lane, v);          // in flight while the counts load
  int32_t* cnt = sh + warp * E;
  for (int e = lane; e < E; e += 32)
    cnt[e] = hist[static_cast<size_t>(e) * n_chunks + c] + __ldg(offsets + e);
  __syncwarp();
  place_chunk_ids(v, p0, p1, E, lane, cnt, sorted_pair, pair_to_row);
}

// One warp per permuted row; each lane keeps up to 8 16-byte vectors of the
// row in flight before it stores any of them.  The x_perm rows are written with
// the streaming (evict-first) policy: the gate/up GEMM reads them back from DRAM
// anyway (268 MB at prefill size), while x (34 MB) is read K times and stays in
// L2 only if the stream of x_perm writes does not push it out (with plain
// stores x was read from DRAM about 2.8 times).
__global__ void __launch_bounds__(256)
permute_gather(const uint16_t* __restrict__ x, int x_rows, const int32_t* __restrict__ sorted_pair,
               int P, int K, int H, uint16_t* __restrict__ x_perm, unsigned long long* launches) {
  count_launch(launches, MOE_KID_PERMUTE_GATHER);
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const int vpr = H / 8;
  for (long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       row < P; row += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
    const int src = __ldg(sorted_pair + row) / K;
    const bool in = src >= 0 && src < x_rows;      // a row outside x is written as zeros
    const uint4* s = reinterpret_cast<const uint4*>(x + static_cast<size_t>(in ? src : 0) * H);
    uint4* d = reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(row) * H);
    for (int v0 = 0; v0 < vpr; v0 += 32 * 8) {
      uint4 buf[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int v = v0 + i * 32 + lane;
        if (v < vpr) buf[i] = in ? __ldg(s + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int v = v0 + i * 32 + lane;
        if (v < vpr) __stcs(d + v, buf[i]);
      }
    }
  }
}

// Count, scan and place for n_chunks <= kSmallChunks in one block: warp c owns
// chunk c as in permute_count / permute_place; the chunk histograms and the
// expert offsets stay in shared memory ([n_chunks][E] + [E] ints).
constexpr int kSmallChunks = 32;
__global__ void __launch_bounds__(kSmallChunks * 32)
permute_small(const int32_t* __restrict__ ids, int P, int E, int n_chunks,
              int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_pair,
              int32_t* __restrict__ pair_to_row, unsigned int* status,
              unsigned long long* launches) {
  count_launch(launches, MOE_KID_PERMUTE_SMALL);
  grid_dep_wait();
  grid_dep_launch();
  extern __shared__ int32_t sh[];
  __shared__ int32_t warp_sum[kSmallChunks];   // one per warp
  int32_t* hist = sh;                         // [n_chunks][E]
  int32_t* base = sh + n_chunks * E;          // [E]: first row of each expert
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int kT = kSmallChunks * 32;
  // 1. per-chunk histograms; the chunk's ids stay in registers for step 4
  int32_t* h = hist + warp * E;
  const int p0 = warp * kChunk, p1 = min(P, p0 + kChunk);
  int v[kIdsPerLane];
  if (warp < n_chunks) {
    load_chunk_ids(ids, p0, p1, lane, v);
    for (int e = lane; e < E; e += 32) h[e] = 0;
    __syncwarp();
    count_chunk_ids(v, p0, p1, E, lane, h, status);
  }
  __syncthreads();
  // 2. per expert: exclusive prefix over the chunks (in chunk order), total in base[e]
  for (int e = tid; e < E; e += kT) {
    int run = 0;
    for (int c = 0; c < n_chunks; ++c) {
      const int v = hist[c * E + e];
      hist[c * E + e] = run;
      run += v;
    }
    base[e] = run;
  }
  __syncthreads();
  // 3. exclusive scan of the totals over experts: thread tid owns experts
  //    [tid * per, tid * per + per), a warp scan, then a scan of the warp sums
  const int per = (E + kT - 1) / kT;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int local = 0;
  for (int e = e0; e < e1; ++e) local += base[e];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kSmallChunks; ++w) {
    const int v = warp_sum[w];
    if (w < warp) before += v;
    total += v;
  }
  int run = before + incl - local;
  for (int e = e0; e < e1; ++e) {
    const int v = base[e];
    base[e] = run;
    offsets[e] = run;
    run += v;
  }
  if (tid == 0) offsets[E] = total;
  __syncthreads();
  // 4. place chunk `warp`, 32 pairs at a time in pair order
  if (warp >= n_chunks) return;
  for (int e = lane; e < E; e += 32) h[e] += base[e];
  __syncwarp();
  place_chunk_ids(v, p0, p1, E, lane, h, sorted_pair, pair_to_row);
}

int n_chunks_of(long long P) { return static_cast<int>((P + kChunk - 1) / kChunk); }

}  // namespace
}  // namespace moe

namespace moe {
namespace {

// the optional x_perm gather after the sort
int gather(const char* op, const void* x_bf16, int x_rows, void* x_perm_bf16,
           const int32_t* sorted_pair, long long P, int K, int H, cudaStream_t s,
           const DeviceDiag& diag) {
  if (!x_perm_bf16) return MOE_OK;
  long long g = (P + 7) / 8;  // 8 rows (warps) per block, at most 32 blocks per SM
  const long long cap = 32LL * sm_count();
  if (g > cap) g = cap;
  return launch_status(
      launch_kernel(permute_gather, dim3(static_cast<unsigned>(g)), dim3(256), 0, s, nullptr, 0,
                    static_cast<const uint16_t*>(x_bf16), x_rows, sorted_pair, static_cast<int>(P), K, H,
                    static_cast<uint16_t*>(x_perm_bf16), diag.launches),
      op);
}

}  // namespace
}  // namespace moe

namespace moe {
// x_perm[r] = x[sorted_pair[r] / K] for r < P on its own (the gate/up entry
// with staged rows uses it for batches that take single-CTA tiles)
int launch_row_gather(const char* op, const void* x_bf16, int x_rows, void* x_perm_bf16,
                      const int32_t* sorted_pair, long long P, int K, int H, cudaStream_t s) {
  return gather(op, x_bf16, x_rows, x_perm_bf16, sorted_pair, P, K, H, s, device_diag());
}
}  // namespace moe

using namespace moe;

extern "C" size_t moe_permute_workspace_size(int T, int K, int E) {
  if (T <= 0 || K <= 0 || E <= 0) return 0;
  const long long P = static_cast<long long>(T) * K;
  return ((static_cast<size_t>(n_chunks_of(P)) * E * sizeof(int32_t)) + 255) &
         ~static_cast<size_t>(255);
}

extern "C" int moe_permute(const int32_t* topk_ids, const void* x_bf16, int T, int K, int E,
                           int H, int32_t* expert_offsets, int32_t* sorted_pair,
                           int32_t* pair_to_row, void* x_perm_bf16, void* workspace,
                           size_t ws_bytes, void* stream) {
  clear_error();
  const char* op = "moe_permute";
  if (T < 0) return set_error(MOE_ERR_ARG, "%s: T=%d < 0", op, T);
  if (K < 1 || K > 32) return set_error(MOE_ERR_ARG, "%s: K=%d outside [1, 32]", op, K);
  if (E < 1 || E > 1024) return set_error(MOE_ERR_ARG, "%s: E=%d outside [1, 1024]", op, E);
  if (!expert_offsets) return set_error(MOE_ERR_ARG, "%s: expert_offsets is NULL", op);
  if (x_perm_bf16 && (!x_bf16 || H <= 0))
    return set_error(MOE_ERR_ARG, "%s: x_perm needs x and H > 0", op);
  if (x_perm_bf16 && (H % 8 != 0 || !aligned16(x_bf16) || !aligned16(x_perm_bf16)))
    return set_error(MOE_ERR_ALIGN, "%s: x/x_perm need 16-byte alignment and H %% 8 == 0", op);
  const long long P = static_cast<long long>(T) * K;
  if (P > 0x7fffffffLL) return set_error(MOE_ERR_ARG, "%s: T*K too large", op);
  if (P > 0 && (!topk_ids || !sorted_pair || !pair_to_row))
    return set_error(MOE_ERR_ARG, "%s: ids/sorted_pair/pair_to_row is NULL", op);
  const size_t need = moe_permute_workspace_size(T, K, E);
  if (need > 0 && (!workspace || ws_bytes < need))
    return set_error(MOE_ERR_WORKSPACE, "%s: workspace of %zu bytes is smaller than %zu", op,
                     ws_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceDiag diag = device_diag();
  const int n_chunks = n_chunks_of(P);
  int32_t* hist = static_cast<int32_t*>(workspace);
  const int blocks = (n_chunks + kWarps - 1) / kWarps;
  const size_t smem = static_cast<size_t>(kWarps) * E * sizeof(int32_t);
  const size_t smem_small = static_cast<size_t>(n_chunks + 1) * E * sizeof(int32_t);
  if (n_chunks > 0 && n_chunks <= kSmallChunks && smem_small <= 48 * 1024) {
    int rc = launch_status(launch_kernel(permute_small, dim3(1), dim3(kSmallChunks * 32),
                                         smem_small, s, nullptr, 0, topk_ids,
                                         static_cast<int>(P), E, n_chunks, expert_offsets,
                                         sorted_pair, pair_to_row, diag.status, diag.launches),
                           op);
    if (rc != MOE_OK) return rc;
    return gather(op, x_bf16, T, x_perm_bf16, sorted_pair, P, K, H, s, diag);
  }
  if (n_chunks > 0) {
    int rc = launch_status(launch_kernel(permute_count, dim3(blocks), dim3(kWarps * 32), smem, s,
                                         nullptr, 0, topk_ids, static_cast<int>(P), E, n_chunks,
                                         hist, diag.status, diag.launches),
                           op);
    if (rc != MOE_OK) return rc;
  }
  int rc = launch_status(launch_kernel(permute_scan, dim3(1), dim3(1024), 0, s, nullptr, 0, hist,
                                       E, n_chunks, expert_offsets, diag.launches),
                         op);
  if (rc != MOE_OK || n_chunks == 0) return rc;
  rc = launch_status(launch_kernel(permute_place, dim3(blocks), dim3(kWarps * 32), smem, s,
                                   nullptr, 0, topk_ids, static_cast<int>(P), E, n_chunks, hist,
                                   expert_offsets, sorted_pair, pair_to_row, diag.launches),
                     op);
  if (rc != MOE_OK) return rc;
  return gather(op, x_bf16, T, x_perm_bf16, sorted_pair, P, K, H, s, diag);
}
