// moe_gemm.cu -- grouped BF16 GEMMs of the MoE expert block on tcgen05 tensor
// cores: kMoeGroupedGemmBf16GateUpSilu and kMoeGroupedGemmBf16 (vllm.cpp issue
// #3094 "Row: BACKEND-ROCM-BF16-MOE", which also fixes their numeric contract:
// BF16 narrowing of the gate/up result before activation, routing weight
// applied before the down result is stored), plus the router-logit GEMM.
// This file holds the single-CTA tiles (one SM per 128-row x N tile); the
// CTA-pair tiles of large batches are in moe_gemm_pair.cu.
//
// One persistent, warp-specialised kernel template:
//   warp 0      TMA producer: A tile [128 x 64] and B tile [kN x 64] bf16 per
//               stage, 128-byte swizzle, into a kStages-deep shared-memory ring
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer
//               (M = 128, N = kN, K = 16 per instruction, f32 accumulators in
//               TMEM, double-buffered so the epilogue overlaps the next tile)
//   warps 2-5   epilogue: tcgen05.ld of one accumulator row per thread, the
//               fused op (bf16 narrowing + SiLU-mul, or routing weight +
//               scatter, or bias + f32 store) and 16-byte stores
//   warps 6-9   (gathered A only) cp.async copies of the routed rows of x into
//               the swizzled A stage, so no permuted copy of x is needed
// The tile schedule is built on the device from the group offsets (the
// routing histogram): every CTA scans ceil(rows_g / 128) * n_tiles over the
// groups in shared memory and walks tiles blockIdx.x, blockIdx.x + gridDim.x,
// ...  All tiles cost the same, so the static stride balances any skew of the
// expert load to within one tile per CTA.  No host round trip, no scratch.
//
// Every wait on an mbarrier is bounded (one second of device time by
// default, moe_set_wait_limit_ns); on expiry the kernel raises
// MOE_STATUS_TIMEOUT in the library's status word, every role stops, and
// before the CTA exits its in-flight copies and MMAs are drained (waits of
// their own, always one second) and its TMEM is freed.
#include <stdio.h>

#include <atomic>
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "gemm_common.cuh"

namespace moe {
namespace gemm {

constexpr int kThreads = 192;        // producer, MMA, 4 epilogue warps
// with gathered A rows, one more thread per A row of a tile gathers it:
// 4 more warps for 128-row tiles, 1 for 32-row tiles
constexpr int kConverters = 256;     // FP8 weights: 8 warps that dequantise B
constexpr int kThreadsFp8 = kThreads + kConverters;
constexpr int A_BYTES = BM * BK * 2;
// bytes of the 227 KB per-block shared memory left for the stage ring after the
// barriers, the schedule tables (2 x 4 KB), the epilogue staging buffers
// (4 x 4 KB) and the 1 KB alignment slack
constexpr int kSmemBudget = 227 * 1024 - 11 * 1024 - 16 * 1024;
constexpr int kStgBytes = 32 * 128;  // epilogue staging: 32 rows x 64 bf16 per warp
constexpr int kNarrowRows = 32;      // rows per tile when experts hold few rows

enum Epi { EPI_GATEUP = 0, EPI_DOWN = 1, EPI_F32 = 2 };

struct Params {
  const int32_t* group_offsets;  // [G+1] device, or null: one group [0, P)
  int P;                         // rows of the product
  int Kdim;                      // contraction length
  int N;                         // output columns
  int G;                         // groups
  int b_rows_per_group;          // rows of the 2-D view of B per group
  int half_off;                  // gate/up: row offset of the up half inside a group
  const uint16_t* a;             // gathered A: row-major [a_rows, Kdim] bf16
  int a_rows;
  const int32_t* row_gather;     // gathered A: product row r reads row row_gather[r] / gather_div
  int gather_div;
  void* out;
  const float* pair_weight;      // down: [P] by destination row, or null
  const int32_t* row_to_pair;    // down: destination row, or null
  const float* bias;             // f32 epilogue: per output column, or null
  // A second, dense problem in the same launch: rows [0, P2) of the A matrix
  // behind the second A tensor map times the one weight matrix behind the
  // second B map, into out2 [P2, N2] (no weight, no scatter).  Its tiles come
  // after the grouped ones in the schedule.  P2 == 0: none.
  int P2;
  int N2;
  int Kdim2;
  int half_off2;                 // gate/up: row offset of the up half in its weight
  void* out2;
  // FP8 weights (kFp8B): E4M3 codes behind the B tensor map, one f32 scale per
  // 128 x 128 block of each group's weight matrix, b_scale[g][row/128][col/128]
  // with scale_rb = ceil(b_rows_per_group / 128) and scale_cb = ceil(Kdim / 128)
  const float* b_scale;
  int scale_rb;
  int scale_cb;
  // f32 epilogue only: split K into ksplit ranges of ceil(nk / ksplit) k-blocks;
  // each (tile, range) is a unit of its own and stores its partial sum, without
  // the bias, at out + range * P * N.  ksplit == 1: the whole K, bias added.
  int ksplit;
  unsigned long long wait_ns;    // limit of every pipeline wait
  unsigned int* status;
  unsigned long long* launches;
  int kid;
};

// Stage ring depth: as many stages of `stage_bytes` as fit the budget, at most 12.
__host__ __device__ constexpr int stages_for_bytes_with(int stage_bytes, int budget) {
  return budget / stage_bytes > 12 ? 12 : budget / stage_bytes;
}
__host__ __device__ constexpr int stages_for_bytes(int stage_bytes) {
  return stages_for_bytes_with(stage_bytes, kSmemBudget);
}

// kConv > 0 (FP8 weights): the stage ring holds A and the raw weight codes
// (kRawBytes a stage); the bf16 B tiles the MMA reads live in a second ring of
// kConv stages, written by the converter warps.
template <int kStages, int kBBytes, int kABytes = A_BYTES, int kConv = 0, int kRawBytes = 0,
          int kEpiBytes = 4 * kStgBytes>
struct Smem {
  static_assert(kStages >= 2, "stage ring too shallow");
  static constexpr int B_BYTES = kBBytes;
  static constexpr int RAW_BYTES = kRawBytes;
  static constexpr int STAGE_A = 0;
  static constexpr int STAGE_RAW = kStages * kABytes;
  static constexpr int STAGE_B = STAGE_RAW + kStages * kRawBytes;
  static constexpr int STAGE_EPI = STAGE_B + (kConv ? kConv : kStages) * B_BYTES;  // staging buffers
  static constexpr int BARS = STAGE_EPI + kEpiBytes;
  // full[kStages], empty[kStages], conv_full[kConv], conv_empty[kConv], tfull[2], tempty[2],
  // drain
  static constexpr int NBARS = 2 * kStages + 2 * kConv + 5;
  static constexpr int MISC = BARS + NBARS * 8;           // tmem slot, abort flag, scan scratch
  static constexpr int TILE_START = MISC + 64;            // int[kMaxGroups + 1]
  static constexpr int GOFF = TILE_START + (kMaxGroups + 1) * 4;
  static constexpr int BYTES = GOFF + (kMaxGroups + 1) * 4;
  static constexpr int ALLOC = BYTES + 1024;              // slack to align the base to 1024
};

// Compile-time shape of one kernel instantiation.
//   kN      MMA N (accumulator columns per tile)
//   kARows  rows per tile and per A box: 128, or 32 when experts hold few
//           rows.  The MMA is still M = 128; with 32-row tiles it reads the 96
//           rows after the stage's A box from whatever shared memory follows
//           (a later stage), and those accumulator rows are never stored.  A
//           stage then holds 4 KB of A instead of 16, so the same shared memory
//           keeps about twice as many weight bytes in flight.
//   kFp8B   B holds FP8 E4M3 weight codes with block scales: TMA brings A and the
//           codes into the stage ring, eight converter warps write the scaled
//           bf16 B tiles into a second ring, and the MMA reads A and that
template <int kN, int kEpi, bool kGatherA, int kARows = BM, bool kFp8B = false>
struct Cfg {
  static_assert(kARows == BM || (kARows % 8 == 0 && (!kGatherA || kARows == 32)),
                "short A tiles: 32 rows when gathered");
  static_assert(!kFp8B || !kGatherA, "FP8 weights: TMA A tiles");
  static constexpr int kTileM = kARows;                           // product rows per tile
  static constexpr int kABytes = kARows * BK * 2;                 // A bytes per stage
  static constexpr int kBBytes = kN * BK * 2;
  static constexpr int kRawBytes = kFp8B ? kN * BK : 0;           // FP8 codes per stage
  static constexpr int kConv = kFp8B ? (kBBytes >= 32 * 1024 ? 2 : 4) : 0;
  static constexpr int kStages =
      kFp8B ? stages_for_bytes_with(kABytes + kRawBytes, kSmemBudget - kConv * kBBytes)
            : stages_for_bytes(kABytes + kBBytes);
  // B boxes: gate/up loads its gate and up halves separately
  static constexpr int kBoxB = (kEpi == EPI_GATEUP) ? kN / 2 : (kN < 128 ? kN : 128);
  static constexpr int kBnOut = (kEpi == EPI_GATEUP) ? kN / 2 : kN;  // output columns per tile
  static constexpr int kThreadsT = kFp8B ? kThreadsFp8 : (kGatherA ? kThreads + kARows : kThreads);
  static constexpr int kEpiCols = 64;                             // columns staged per pass
  static constexpr int kStgWarp = 32 * kEpiCols * 2;
  using S = Smem<kStages, kBBytes, kABytes, kConv, kRawBytes, 4 * kStgWarp>;
};

struct Tile {
  int g, row0, row_end, n0;
  int pb;    // 0: the grouped problem, 1: the second (dense) problem
  int ks;    // K range of a split-K unit (0 without split)
};

// M tiles of a group of `rows` rows
__device__ __forceinline__ int group_m_tiles(int rows, int tile_m) {
  return rows <= 0 ? 0 : (rows + tile_m - 1) / tile_m;
}

__device__ __forceinline__ Tile decode_tile(int tile, const int* tile_start, const int* goff,
                                            int G, int n_tiles, int bn_out, int tile_m) {
  int lo = 0, hi = G;  // tile_start[lo] <= tile < tile_start[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid;
  }
  const int local = tile - tile_start[lo];
  const int m = local / n_tiles, n = local - m * n_tiles;
  Tile t;
  t.g = lo;
  t.row0 = goff[lo] + m * tile_m;
  t.row_end = min(goff[lo + 1], t.row0 + tile_m);
  t.n0 = n * bn_out;
  t.pb = 0;
  t.ks = 0;
  return t;
}

// Placement of the second problem's `extra` tiles: after the `routed` grouped
// tiles (schedule indices routed .. routed + extra - 1).  The persistent CTAs
// take tiles round-robin, so the second problem's tiles fill the ragged last
// round of the grouped ones.  On the large layer (all routed tiles streaming
// weights from HBM, shared-expert tiles bound by the tensor pipe) this beats
// interleaving them evenly, which leaves the CTAs that drew one late on their
// share of the HBM stream (gate/up 683 us at the end, 720 us interleaved, 711 us
// as two launches).
struct Sched2 {
  int routed, extra, n2_tiles, P2;
};

__device__ __forceinline__ Tile locate_tile(int i, const int* tile_start, const int* goff, int G,
                                            int n_tiles, int bn_out, int tile_m,
                                            const Sched2& s2) {
  if (s2.extra > 0 && i >= s2.routed) {
    const int q = i - s2.routed;
    const int m = q / s2.n2_tiles;
    Tile t;
    t.g = 0;
    t.row0 = m * tile_m;
    t.row_end = min(s2.P2, t.row0 + tile_m);
    t.n0 = (q - m * s2.n2_tiles) * bn_out;
    t.pb = 1;
    t.ks = 0;
    return t;
  }
  return decode_tile(i, tile_start, goff, G, n_tiles, bn_out, tile_m);
}

// split-K units (f32 epilogue): schedule index i is K range i % ksplit of tile i / ksplit
__device__ __forceinline__ Tile locate_unit(int i, int ksplit, const int* tile_start,
                                            const int* goff, int G, int n_tiles, int bn_out,
                                            int tile_m, const Sched2& s2) {
  if (ksplit <= 1) return locate_tile(i, tile_start, goff, G, n_tiles, bn_out, tile_m, s2);
  const int q = i / ksplit;
  Tile t = locate_tile(q, tile_start, goff, G, n_tiles, bn_out, tile_m, s2);
  t.ks = i - q * ksplit;
  return t;
}

template <int kN, int kEpi, bool kGatherA, int kARows, bool kFp8B>
__global__ void __launch_bounds__(Cfg<kN, kEpi, kGatherA, kARows, kFp8B>::kThreadsT, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmA2,
                    const __grid_constant__ CUtensorMap tmB2, const Params p) {
  using C = Cfg<kN, kEpi, kGatherA, kARows, kFp8B>;
  using S = typename C::S;
  constexpr int kABytes = C::kABytes;
  constexpr int kConv = C::kConv;
  constexpr int kStages = C::kStages;
  constexpr int kNThreads = C::kThreadsT;
  constexpr int kTileM = C::kTileM;
  constexpr int kBnOut = C::kBnOut;
  constexpr int kBoxB = C::kBoxB;
  constexpr int kBoxBytes = kBoxB * BK * (kFp8B ? 1 : 2);   // one B box as loaded
  // gathered A: each row-thread keeps kDepth stages of copies in flight before
  // it must retire the oldest one (kDepth < kStages keeps the ring deadlock-free)
  constexpr int kDepth = kStages - 1;
  constexpr int kTmemCols = 2 * kN;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(BM, kN);
  constexpr uint32_t kStageTx = (kGatherA ? 0 : kABytes) + (kFp8B ? S::RAW_BYTES : S::B_BYTES);
  constexpr int kEpiCols = C::kEpiCols;
  constexpr int kStgWarp = C::kStgWarp;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::MISC + 4);
  int* scan_tmp = reinterpret_cast<int*>(smem + S::MISC + 8);   // 10 ints
  int* tile_start = reinterpret_cast<int*>(smem + S::TILE_START);
  int* goff = reinterpret_cast<int*>(smem + S::GOFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int unit = static_cast<int>(blockIdx.x);
  const int n_units = static_cast<int>(gridDim.x);
  const unsigned long long wait_ns = p.wait_ns;
  auto bar_full = [&](int s) { return ptx::smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return ptx::smem_u32(bars + kStages + s); };
  auto bar_cfull = [&](int s) { return ptx::smem_u32(bars + 2 * kStages + s); };
  auto bar_cempty = [&](int s) { return ptx::smem_u32(bars + 2 * kStages + kConv + s); };
  auto bar_tfull = [&](int a) { return ptx::smem_u32(bars + 2 * kStages + 2 * kConv + a); };
  auto bar_tempty = [&](int a) { return ptx::smem_u32(bars + 2 * kStages + 2 * kConv + 2 + a); };
  const uint32_t bar_drain = ptx::smem_u32(bars + 2 * kStages + 2 * kConv + 4);

  count_launch(p.launches, p.kid);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar_full(s), kGatherA ? 1 + kARows : 1);
      // FP8 weights: a stage is free once the MMA and every converter are done with it
      ptx::mbar_init(bar_empty(s), kFp8B ? 1 + kConverters : 1);
    }
    for (int s = 0; s < kConv; ++s) {
      ptx::mbar_init(bar_cfull(s), kConverters);
      ptx::mbar_init(bar_cempty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(bar_tfull(a), 1);
      ptx::mbar_init(bar_tempty(a), BM);
    }
    ptx::mbar_init(bar_drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    if (p.P2 > 0) {
      ptx::tma_prefetch_desc(&tmA2);
      ptx::tma_prefetch_desc(&tmB2);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }

  // the set-up above touches no global data; from here on this kernel reads
  // what the previous kernel in the stream wrote (group offsets, A rows)
  grid_dep_wait();
  grid_dep_launch();

  // ---- device-side tile schedule from the group offsets
  const int G = p.G;
  for (int g = threadIdx.x; g <= G; g += kNThreads)
    goff[g] = p.group_offsets ? __ldg(p.group_offsets + g) : (g == 0 ? 0 : p.P);
  __syncthreads();
  const int n_tiles = (p.N + kBnOut - 1) / kBnOut;
  const int chunk = (G + kNThreads - 1) / kNThreads;
  const int g_lo = min(G, static_cast<int>(threadIdx.x) * chunk);
  const int g_hi = min(G, g_lo + chunk);
  int local = 0;
  for (int g = g_lo; g < g_hi; ++g) local += group_m_tiles(goff[g + 1] - goff[g], kTileM) * n_tiles;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scan_tmp[warp] = incl;
  __syncthreads();
  int warp_base = 0, total = 0;
  for (int w = 0; w < kNThreads / 32; ++w) {
    int v = scan_tmp[w];
    if (w < warp) warp_base += v;
    total += v;
  }
  int run = warp_base + incl - local;
  for (int g = g_lo; g < g_hi; ++g) {
    tile_start[g] = run;
    run += group_m_tiles(goff[g + 1] - goff[g], kTileM) * n_tiles;
  }
  if (threadIdx.x == 0) tile_start[G] = total;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int nk = (p.Kdim + BK - 1) / BK;
  constexpr bool kCan2 = !kGatherA;
  const int ksplit = (kEpi == EPI_F32 && p.ksplit > 1) ? p.ksplit : 1;
  const int nk_split = (nk + ksplit - 1) / ksplit;   // k-blocks per K range
  Sched2 s2{total, 0, 1, 0};
  if (kCan2 && p.P2 > 0) {
    s2.n2_tiles = (p.N2 + kBnOut - 1) / kBnOut;
    s2.extra = ((p.P2 + kTileM - 1) / kTileM) * s2.n2_tiles;
    s2.P2 = p.P2;
    total += s2.extra;
  }
  total *= ksplit;
  const int nk2 = (p.Kdim2 + BK - 1) / BK;

  // state the exit drain needs: the producer's ring position and copy count,
  // whether the MMA issuer issued anything
  int prod_stage = 0;
  uint32_t prod_phase = 0;
  int prod_issued = 0;
  bool mma_any = false;

  if (kGatherA && warp >= 6) {
    // ------------------------------------------------------------ A-row gatherers
    // Thread i owns row i of this CTA's A tile (128 or 32 rows): row_gather[row] / gather_div
    // picks the source row, and each stage copies its 64 columns (8 x 16 B)
    // with cp.async into the 128-byte-swizzled layout a TMA SWIZZLE_128B box
    // would produce (16-byte chunk c of row i lands at chunk c ^ (i % 8)).
    // Indices outside [0, a_rows) read zeros, like a TMA out-of-bounds box, and
    // so do the rows past the tile's group, which are never stored: at decode
    // a tile holds one or two routed rows, and its other rows, copied from the
    // next groups' tokens, sent every CTA's requests to the same few lines of x.
    const int i = static_cast<int>(threadIdx.x) - kThreads;
    int stage = 0;
    uint32_t phase = 0;
    int pending = 0;
    bool ok = true;
    for (int tile = unit; ok && tile < total; tile += n_units) {
      const Tile t = decode_tile(tile, tile_start, goff, G, n_tiles, kBnOut, kTileM);
      const int srow = t.row0 + i < t.row_end ? __ldg(p.row_gather + t.row0 + i) / p.gather_div : -1;
      const bool in = srow >= 0 && srow < p.a_rows;
      const uint16_t* src = p.a + static_cast<size_t>(in ? srow : 0) * p.Kdim;
      for (int kb = 0; kb < nk; ++kb) {
        if (!wait_bar(bar_empty(stage), phase ^ 1u, abort_flag, p.status, wait_ns)) {
          ok = false;
          break;
        }
        const uint32_t dst = sbase + S::STAGE_A + stage * kABytes + i * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int col = kb * BK + c * 8;
          const bool live = in && col < p.Kdim;    // Kdim % 8 == 0: a chunk is all in or out
          ptx::cp_async_16(dst + ((c ^ (i & 7)) << 4), src + (live ? col : 0), live ? 16u : 0u);
        }
        ptx::cp_async_commit();
        if (++pending == kDepth) {
          ptx::cp_async_wait<kDepth - 1>();
          ptx::fence_proxy_async_smem();
          int old = stage - (kDepth - 1);
          if (old < 0) old += kStages;
          ptx::mbar_arrive(bar_full(old));
          --pending;
        }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    ptx::cp_async_wait<0>();
    if (ok) {
      ptx::fence_proxy_async_smem();
      for (int q = pending; q > 0; --q) {
        int old = stage - q;
        if (old < 0) old += kStages;
        ptx::mbar_arrive(bar_full(old));
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // A box (unless gathered) and B boxes, completion on the stage's barrier
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = unit; ok && tile < total; tile += n_units) {
        const Tile t = locate_unit(tile, ksplit, tile_start, goff, G, n_tiles, kBnOut, kTileM, s2);
        const bool second = kCan2 && t.pb == 1;
        const CUtensorMap* mA = second ? &tmA2 : &tmA;
        const CUtensorMap* mB = second ? &tmB2 : &tmB;
        const int kb_lo = t.ks * nk_split;
        const int nk_t = second ? nk2 : min(nk, kb_lo + nk_split);
        // B rows of the tile (gate/up: the gate half, then the up half)
        int brow0, brow1;
        if (second) {
          brow0 = t.n0;
          brow1 = brow0 + p.half_off2;
        } else {
          brow0 = t.g * p.b_rows_per_group + t.n0;
          brow1 = brow0 + p.half_off;
        }
        for (int kb = second ? 0 : kb_lo; kb < nk_t; ++kb) {
          // spinning: the producer's reaction time is part of the ring's round trip
          if (!wait_bar_spin(bar_empty(stage), phase ^ 1u, abort_flag, p.status, wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t sa = sbase + S::STAGE_A + stage * kABytes;
          const uint32_t sb = kFp8B ? sbase + S::STAGE_RAW + stage * S::RAW_BYTES
                                    : sbase + S::STAGE_B + stage * S::B_BYTES;
          const uint32_t fb = bar_full(stage);
          ptx::mbar_arrive_expect_tx(fb, kStageTx);
          if (!kGatherA) ptx::tma_load_2d(sa, mA, kb * BK, t.row0, fb);
          if (kEpi == EPI_GATEUP) {
            ptx::tma_load_2d(sb, mB, kb * BK, brow0, fb);
            ptx::tma_load_2d(sb + kBoxBytes, mB, kb * BK, brow1, fb);
          } else {
#pragma unroll
            for (int h = 0; h < kN / kBoxB; ++h)
              ptx::tma_load_2d(sb + h * kBoxBytes, mB, kb * BK, brow0 + h * kBoxB, fb);
          }
          ++prod_issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      prod_stage = stage;
      prod_phase = phase;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int cst = 0;             // FP8 weights: stage of the converted ring
      uint32_t cphase = 0;
      uint32_t uses0 = 0, uses1 = 0;  // accumulator slot uses: the barrier phases
      int acc = 0;
      bool ok = true;
      for (int tile = unit; ok && tile < total; tile += n_units) {
        if (!wait_bar(bar_tempty(acc), ((acc ? uses1 : uses0) & 1u) ^ 1u, abort_flag, p.status,
                      wait_ns)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kN);
        int nk_t = nk;
        if (ksplit > 1) {
          const int kb_lo = (tile % ksplit) * nk_split;
          nk_t = min(nk, kb_lo + nk_split) - kb_lo;
        } else if (kCan2 && s2.extra > 0 &&
                   locate_tile(tile, tile_start, goff, G, n_tiles, kBnOut, kTileM, s2).pb) {
          nk_t = nk2;
        }
        for (int kb = 0; kb < nk_t; ++kb) {
          if (!wait_bar(bar_full(stage), phase, abort_flag, p.status, wait_ns)) {
            ok = false;
            break;
          }
          if (kFp8B && !wait_bar(bar_cfull(cst), cphase, abort_flag, p.status, wait_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t da = ptx::desc_kmajor_sw128(sbase + S::STAGE_A + stage * kABytes);
          const uint64_t db = ptx::desc_kmajor_sw128(sbase + S::STAGE_B +
                                                     (kFp8B ? cst : stage) * S::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            // +32 bytes along K inside the 128-byte swizzle atom: +2 in the address field
            ptx::mma_bf16(d, da + 2ull * k, db + 2ull * k, kIdesc, (kb | k) != 0 ? 1u : 0u);
          mma_any = true;
          ptx::mma_commit(bar_empty(stage));
          if (kFp8B) {
            ptx::mma_commit(bar_cempty(cst));
            if (++cst == kConv) { cst = 0; cphase ^= 1u; }
          }
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit(bar_tfull(acc));
        if (acc) ++uses1;
        else ++uses0;
        acc ^= 1;
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int r_in_tile = q * 32 + lane;
    uint32_t uses0 = 0, uses1 = 0;          // completions seen on each full barrier
    int acc = 0;
    for (int tile = unit; tile < total; tile += n_units) {
      const Tile t = locate_unit(tile, ksplit, tile_start, goff, G, n_tiles, kBnOut, kTileM, s2);
      const bool second = kCan2 && t.pb == 1;
      const int n_out = second ? p.N2 : p.N;
      const uint32_t aphase = (acc ? uses1 : uses0) & 1u;
      // every lane polls with its own clock: the warp goes on only if all of
      // them saw the accumulator, since the TMEM loads below need the whole warp
      const bool landed = wait_bar(bar_tfull(acc), aphase, abort_flag, p.status, wait_ns);
      if (!__all_sync(0xffffffffu, landed)) {
        *abort_flag = 1;
        break;
      }
      ptx::tc_fence_after();
      const int row = t.row0 + r_in_tile;
      const bool valid = row < t.row_end;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * kN);
      if (kEpi == EPI_GATEUP || kEpi == EPI_DOWN) {
        // bf16 outputs go out through a per-warp staging buffer: the warp's 32
        // rows x 64 columns (128 B a row) are written to shared memory by row
        // (16-byte pieces XOR-swizzled by row to spread the banks), then read
        // back so that eight lanes store one row's 128 contiguous bytes: full
        // 128-byte lines instead of 32 scattered 16-byte pieces per store.
        uint16_t* out = static_cast<uint16_t*>(second ? p.out2 : p.out);
        const uint32_t stg = sbase + S::STAGE_EPI + static_cast<uint32_t>(warp - 2) * kStgWarp;
        constexpr int kH = kEpiCols / 32;        // 32-column TMEM loads per pass
        constexpr int kPieces = kEpiCols / 8;    // 16-byte pieces of a staged row
        constexpr int kRowsPer = 32 / kPieces;   // rows one store instruction covers
        int dst_row = row;
        float wgt = 1.0f;
        if (kEpi == EPI_DOWN && valid && !second) {
          if (p.row_to_pair) dst_row = __ldg(p.row_to_pair + row);
          if (p.pair_weight) wgt = __ldg(p.pair_weight + dst_row);
        }
#pragma unroll 1
        for (int c = 0; c < kBnOut / kEpiCols; ++c) {
          uint32_t packed[kEpiCols / 2];
#pragma unroll
          for (int h = 0; h < kH; ++h) {
            uint32_t g[32];
            ptx::tmem_ld_32x32b_x32(taddr + c * kEpiCols + h * 32, g);
            if (kEpi == EPI_GATEUP) {
              uint32_t u[32];
              ptx::tmem_ld_32x32b_x32(taddr + kBnOut + c * kEpiCols + h * 32, u);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                float a2[2];
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                  // narrowing before the activation: gate and up are rounded to bf16 first
                  const uint32_t gu =
                      pack_bf16x2(__uint_as_float(g[j + q2]), __uint_as_float(u[j + q2]));
                  const float gz = __uint_as_float(gu << 16);
                  const float uz = __uint_as_float(gu & 0xFFFF0000u);
                  // SiLU is tolerance-checked, so the fast reciprocal division serves
                  // (it gives the IEEE quotient's 0 where 1 + exp(-g) overflows)
                  const float sl = __fdividef(gz, 1.0f + __expf(-gz));
                  a2[q2] = sl * uz;
                }
                packed[h * 16 + j / 2] = pack_bf16x2(a2[0], a2[1]);
              }
            } else {
              ptx::tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                // the routing weight: one f32 multiply, then the one bf16 rounding
                const bool wt = p.pair_weight && !second;
                const float a = wt ? __fmul_rn(__uint_as_float(g[j]), wgt) : __uint_as_float(g[j]);
                const float b = wt ? __fmul_rn(__uint_as_float(g[j + 1]), wgt)
                                   : __uint_as_float(g[j + 1]);
                packed[h * 16 + j / 2] = pack_bf16x2(a, b);
              }
            }
          }
          if (c == kBnOut / kEpiCols - 1) {  // the accumulator is in registers: free it now
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_tempty(acc));
          }
          // row `lane` of the staging buffer, piece k at slot k ^ (lane % kPieces)
#pragma unroll
          for (int k = 0; k < kPieces; ++k)
            ptx::st_shared_v4(stg + lane * (2 * kEpiCols) + ((k ^ (lane & (kPieces - 1))) << 4),
                              packed[4 * k], packed[4 * k + 1], packed[4 * k + 2],
                              packed[4 * k + 3]);
          __syncwarp();
          const int col0 = t.n0 + c * kEpiCols;
#pragma unroll
          for (int i = 0; i < kPieces; ++i) {       // kRowsPer rows per store instruction
            const int r = i * kRowsPer + lane / kPieces;  // row of the warp this lane stores
            const int k = lane % kPieces;                 // its 16-byte piece of that row
            const int drow = __shfl_sync(0xffffffffu, dst_row, r);
            const int rvalid = __shfl_sync(0xffffffffu, valid ? 1 : 0, r);
            const uint4 v = ptx::ld_shared_v4(stg + r * (2 * kEpiCols) +
                                              ((k ^ (r & (kPieces - 1))) << 4));
            const int col = col0 + k * 8;
            if (rvalid && col < n_out)
              *reinterpret_cast<uint4*>(out + static_cast<size_t>(drow) * n_out + col) = v;
          }
          __syncwarp();
        }
      } else {
        // a split-K unit stores its partial sum, without the bias, in its own slab
        float* out = static_cast<float*>(p.out) +
                     static_cast<size_t>(t.ks) * static_cast<size_t>(p.P) * p.N;
        const float* bias = ksplit > 1 ? nullptr : p.bias;
#pragma unroll 1
        for (int c = 0; c < kBnOut / 32; ++c) {
          uint32_t y[32];
          ptx::tmem_ld_32x32b_x32(taddr + c * 32, y);
          ptx::tmem_ld_wait();
          const int col = t.n0 + c * 32;
          if (valid && col < p.N) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              v[j] = __uint_as_float(y[j]);
              if (bias && col + j < p.N) v[j] = __fadd_rn(v[j], __ldg(bias + col + j));
            }
            float* dst = out + static_cast<size_t>(row) * p.N + col;
            if ((p.N & 3) == 0) {
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4)
                if (col + 4 * q4 < p.N)
                  reinterpret_cast<float4*>(dst)[q4] =
                      make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col + j < p.N) dst[j] = v[j];
            }
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_tempty(acc));
      }
      if (acc) ++uses1;
      else ++uses0;
      acc ^= 1;
    }
  } else if (kFp8B) {
    // ------------------------------------------------------------ FP8 converters
    // Thread ct of warps 6-13 handles 16-byte pieces q = ct + 256 j of the B tile:
    // row q / 8, codes 8 (q % 8) .. 8 (q % 8) + 7 of the stage's 64 columns.  Each
    // weight becomes bf16(f32(code) * scale) with the scale of its 128 x 128
    // block, written where a TMA SWIZZLE_128B box would put it (16-byte piece c
    // of row r at piece c ^ (r % 8)), so the MMA reads it like any bf16 B tile.
    const int ct = static_cast<int>(threadIdx.x) - kThreads;
    int stage = 0, cst = 0;
    uint32_t phase = 0, cphase = 0;
    bool ok = true;
    for (int tile = unit; ok && tile < total; tile += n_units) {
      const Tile t = locate_unit(tile, ksplit, tile_start, goff, G, n_tiles, kBnOut, kTileM, s2);
      // weight rows (within the group) of tile rows [0, kN/2) and [kN/2, kN)
      const int wrow0 = t.n0;
      const int wrow1 = (kEpi == EPI_GATEUP) ? t.n0 + p.half_off : t.n0 + kN / 2;
      const float* scale_g =
          p.b_scale + static_cast<size_t>(t.g) * static_cast<size_t>(p.scale_rb) * p.scale_cb;
      const int kb_lo = t.ks * nk_split;
      const int kb_hi = min(nk, kb_lo + nk_split);
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (!wait_bar(bar_full(stage), phase, abort_flag, p.status, wait_ns)) {
          ok = false;
          break;
        }
        if (!wait_bar(bar_cempty(cst), cphase ^ 1u, abort_flag, p.status, wait_ns)) {
          ok = false;
          break;
        }
        const uint8_t* raw = smem + S::STAGE_RAW + stage * S::RAW_BYTES;
        const uint32_t dst = sbase + S::STAGE_B + cst * S::B_BYTES;
        const int cblk = (kb * BK) / 128;
        // the scale of a row's block is reloaded only when the block changes
        int sc_blk = -1;
        float sc = 0.0f;
#pragma unroll 4
        for (int j = 0; j < kN * 8 / kConverters; ++j) {
          const int q = ct + kConverters * j;
          const int r = q >> 3, c = q & 7;
          const int wr = r < kN / 2 ? wrow0 + r : wrow1 + (r - kN / 2);
          // rows past the group's own (a ragged last N tile) are never stored
          const int rblk = min(wr / 128, p.scale_rb - 1);
          if (rblk != sc_blk) {
            sc = __ldg(scale_g + static_cast<size_t>(rblk) * p.scale_cb + cblk);
            sc_blk = rblk;
          }
          const uint2 codes = *reinterpret_cast<const uint2*>(raw + r * BK + c * 8);
          const uint32_t cw[2] = {codes.x, codes.y};
          uint32_t packed[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const __nv_fp8x2_storage_t two =
                static_cast<__nv_fp8x2_storage_t>((cw[h >> 1] >> ((h & 1) * 16)) & 0xFFFFu);
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);  // exact
            const float lo = __fmul_rn(__half2float(__ushort_as_half(hr.x)), sc);
            const float hi = __fmul_rn(__half2float(__ushort_as_half(hr.y)), sc);
            packed[h] = pack_bf16x2(lo, hi);
          }
          ptx::st_shared_v4(dst + r * 128 + ((c ^ (r & 7)) << 4), packed[0], packed[1], packed[2],
                            packed[3]);
        }
        ptx::fence_proxy_async_smem();     // the tensor core reads these through the async proxy
        ptx::mbar_arrive(bar_cfull(cst));
        ptx::mbar_arrive(bar_empty(stage));
        if (++cst == kConv) { cst = 0; cphase ^= 1u; }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // A role gave up.  Copies and MMAs issued before that may still be in
    // flight whichever role stopped first, so wait for them (bounded) before
    // the shared memory and the TMEM they target are released.
    if (warp == 0 && lane == 0) {
      int s = prod_stage;
      uint32_t ph = prod_phase;
      for (int i = 0; i < min(prod_issued, kStages); ++i) {
        if (--s < 0) { s = kStages - 1; ph ^= 1u; }
        spin_bounded(bar_full(s), ph);
      }
    }
    if (warp == 1 && lane == 0 && mma_any) {
      ptx::mma_commit(bar_drain);
      spin_bounded(bar_drain, 0);
    }
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

// rows x cols bf16 matrix (row-major, cols contiguous), box of 64 cols x box_rows rows
int make_tmap(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows,
              const char* op, const char* what) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(MOE_ERR_CUDA, "%s: cuTensorMapEncodeTiled is unavailable", op);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(MOE_ERR_CUDA, "%s: tensor map for %s rejected (CUresult %d)", op, what,
                     static_cast<int>(r));
  return MOE_OK;
}

// rows x cols FP8 codes (one byte each, cols contiguous), box of 64 cols x box_rows
// rows, unswizzled (the converter warps read it as plain rows of 64 bytes)
int make_tmap_u8(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows,
                 const char* op, const char* what) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(MOE_ERR_CUDA, "%s: cuTensorMapEncodeTiled is unavailable", op);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(MOE_ERR_CUDA, "%s: tensor map for %s rejected (CUresult %d)", op, what,
                     static_cast<int>(r));
  return MOE_OK;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 148;
  }
  return n;
}

// limit of the pipeline waits (process-wide; see moe_set_wait_limit_ns)
std::atomic<unsigned long long> g_wait_ns{kDrainLimitNs};
unsigned long long pipeline_wait_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

// tile_bound: an upper bound on the number of tiles (of C::kTileM rows); the
// grid is that many CTAs, capped at the SM count
template <int kN, int kEpi, bool kGatherA = false, int kARows = BM, bool kFp8B = false>
int launch(const char* op, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ta2,
           const CUtensorMap& tb2, Params p, long long tile_bound, cudaStream_t stream) {
  using C = Cfg<kN, kEpi, kGatherA, kARows, kFp8B>;
  auto kern = grouped_gemm_kernel<kN, kEpi, kGatherA, kARows, kFp8B>;
  const int smem = C::S::ALLOC;
  // per instantiation and device, set once (racing threads set the same value)
  static std::atomic<int> configured_dev[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  if (dev < 0 || dev >= 64 || !configured_dev[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return set_error(MOE_ERR_CUDA, "%s: cannot reserve %d bytes of shared memory: %s", op, smem,
                       cudaGetErrorString(cudaGetLastError()));
    if (dev >= 0 && dev < 64) configured_dev[dev].store(1, std::memory_order_release);
  }
  // persistent grid: at most one CTA per SM
  long long units = tile_bound;
  const long long max_units = num_sms();
  if (units > max_units) units = max_units;
  if (units < 1) units = 1;
  DeviceDiag diag = device_diag();
  p.status = diag.status;
  p.launches = diag.launches;
  p.wait_ns = pipeline_wait_ns();
  return launch_status(launch_kernel(kern, dim3(static_cast<unsigned>(units), 1, 1),
                                     dim3(C::kThreadsT, 1, 1), smem, stream, nullptr, 0, ta, tb,
                                     ta2, tb2, p),
                       op);
}

// one grouped problem (the second-problem maps are unused copies)
template <int kN, int kEpi, bool kGatherA = false, int kARows = BM, bool kFp8B = false>
int launch(const char* op, const CUtensorMap& ta, const CUtensorMap& tb, Params p,
           long long tile_bound, cudaStream_t stream) {
  return launch<kN, kEpi, kGatherA, kARows, kFp8B>(op, ta, tb, ta, tb, p, tile_bound, stream);
}

int check_common(const char* op, int P, int Kdim, int N, int G, const void* a, const void* b,
                 const void* out) {
  if (P < 0) return set_error(MOE_ERR_ARG, "%s: P=%d < 0", op, P);
  if (Kdim <= 0 || N <= 0) return set_error(MOE_ERR_ARG, "%s: dimensions must be positive", op);
  if (G < 1 || G > kMaxGroups)
    return set_error(MOE_ERR_ARG, "%s: G=%d outside [1, %d]", op, G, kMaxGroups);
  if (Kdim % 8 != 0 || N % 8 != 0)
    return set_error(MOE_ERR_ALIGN, "%s: H and I must be multiples of 8", op);
  if (P > 0 && (!a || !b || !out)) return set_error(MOE_ERR_ARG, "%s: NULL operand", op);
  if (!aligned16(a) || !aligned16(b) || !aligned16(out))
    return set_error(MOE_ERR_ALIGN, "%s: operands must be 16-byte aligned", op);
  return MOE_OK;
}

long long tile_bound(int P, int G, int N, int bn_out, int tile_m = BM) {
  long long mt = (P + tile_m - 1) / tile_m + (G < P ? G : P);
  return mt * ((N + bn_out - 1) / bn_out);
}

// tiling of the grouped GEMMs (process-wide; see moe_set_gemm_pairing)
std::atomic<int> g_pairing{MOE_GEMM_AUTO};

// CTA-pair tiles (moe_gemm_pair.cu) for a bf16 grouped GEMM over x_perm-style
// rows: forced by MOE_GEMM_PAIR; with MOE_GEMM_AUTO when the groups average at
// least 32 rows and the call has at least 1024 (prefill-sized batches, where the
// tensor cores bind and the pair tiles' smaller padding and shared-memory fill
// pay); never for MOE_GEMM_SINGLE.
bool use_pair_tiles(int P, int G) {
  if (G > kMaxPairGroups) return false;
  const int mode = g_pairing.load(std::memory_order_relaxed);
  if (mode == MOE_GEMM_PAIR) return true;
  return mode == MOE_GEMM_AUTO && P >= 1024 && static_cast<long long>(P) >= 32LL * G;
}

}  // namespace gemm

// router logits l[t, e] = x[t,:] . w_router[e,:] (+ bias[e]) in f32 (used by moe_route.cu)
// K ranges for the router logits GEMM: enough (tile, range) units to give every
// SM one when T x E alone makes few tiles (decode), at most 16, every range
// non-empty.  ranges * T * E floats of partial sums.
int launch_row_gather(const char* op, const void* x_bf16, int x_rows, void* x_perm_bf16,
                      const int32_t* sorted_pair, long long P, int K, int H, cudaStream_t s);

int router_splits(int T, int H, int E) {
  using namespace gemm;
  const long long tiles = static_cast<long long>((T + BM - 1) / BM) * ((E + 63) / 64);
  long long want = tiles > 0 ? num_sms() / tiles : 1;
  if (want > 16) want = 16;
  if (want < 1) want = 1;
  const int nk = (H + BK - 1) / BK;
  if (want > nk) want = nk;
  const int per = static_cast<int>((nk + want - 1) / want);
  return (nk + per - 1) / per;
}

int launch_router_logits(const void* x, const void* w_router, const float* bias, int T, int H,
                         int E, float* logits, int ksplit, cudaStream_t stream) {
  using namespace gemm;
  const char* op = "moe_route_topk";
  if (T == 0) return MOE_OK;
  CUtensorMap ta, tb;
  int rc;
  // 128 x 64 tiles: twice the CTAs of a full-width tile, so more SMs stream x
  if ((rc = make_tmap(&ta, x, T, H, BM, op, "x")) != MOE_OK) return rc;
  if ((rc = make_tmap(&tb, w_router, E, H, 64, op, "w_router")) != MOE_OK) return rc;
  Params p{};
  p.group_offsets = nullptr;
  p.P = T;
  p.Kdim = H;
  p.N = E;
  p.G = 1;
  p.b_rows_per_group = E;
  p.half_off = 0;
  p.out = logits;
  p.bias = bias;
  p.ksplit = ksplit < 1 ? 1 : ksplit;
  p.kid = MOE_KID_ROUTE_LOGITS;
  return launch<64, EPI_F32>(op, ta, tb, p, tile_bound(T, 1, E, 64) * p.ksplit, stream);
}

}  // namespace moe

using namespace moe;
using namespace moe::gemm;

extern "C" size_t moe_grouped_gemm_workspace_size(int, int, int, int) { return 0; }

extern "C" int moe_set_gemm_pairing(int mode) {
  clear_error();
  if (mode == 3 || mode == 4)
    return set_error(MOE_ERR_UNSUPPORTED,
                     "moe_set_gemm_pairing: mode %d is not built (AUTO, SINGLE or PAIR)", mode);
  if (mode != MOE_GEMM_AUTO && mode != MOE_GEMM_SINGLE && mode != MOE_GEMM_PAIR)
    return set_error(MOE_ERR_ARG, "moe_set_gemm_pairing: mode %d is not 0, 1 or 2", mode);
  return g_pairing.exchange(mode);
}

extern "C" int moe_set_wait_limit_ns(unsigned long long ns) {
  clear_error();
  if (ns < 1000ull || ns > kDrainLimitNs)
    return set_error(MOE_ERR_ARG, "moe_set_wait_limit_ns: %llu ns is outside [1000, %llu]", ns,
                     kDrainLimitNs);
  g_wait_ns.store(ns, std::memory_order_relaxed);
  return MOE_OK;
}

extern "C" int moe_grouped_gemm_gateup_silu_bf16(const void* a_bf16, int a_rows,
                                                 const int32_t* a_row_gather, int gather_div,
                                                 const void* w13_bf16,
                                                 const int32_t* group_offsets, int P, int H,
                                                 int I, int G, void* act_bf16, void* workspace,
                                                 size_t ws_bytes, void* stream) {
  (void)workspace;
  (void)ws_bytes;
  clear_error();
  const char* op = "moe_grouped_gemm_gateup_silu_bf16";
  int rc;
  if ((rc = check_common(op, P, H, I, G, a_bf16, w13_bf16, act_bf16)) != MOE_OK) return rc;
  if (!group_offsets && G != 1)
    return set_error(MOE_ERR_ARG, "%s: group_offsets is NULL with G=%d", op, G);
  if (a_row_gather && (a_rows < 1 || gather_div < 1))
    return set_error(MOE_ERR_ARG, "%s: gathering needs a_rows >= 1 and gather_div >= 1", op);
  if (P == 0) return MOE_OK;
  if (use_pair_tiles(P, G))
    return launch_pair_gateup(op, a_bf16, a_rows, a_row_gather, gather_div, w13_bf16,
                              group_offsets, P, H, I, G, act_bf16,
                              static_cast<cudaStream_t>(stream));
  // Few rows per expert (decode): each tile streams its weight rows from HBM
  // and the tile count decides the balance; 128-wide tiles (64 gate + 64 up
  // rows) double it, which cuts the idle tail of the last round (decode layer,
  // 82 of 128 experts touched: 127 -> 115 us).  32-row tiles load 4 KB of A per
  // stage instead of 16 (a TMA box of x_perm, or one gatherer warp's copies of
  // routed rows of x), so the ring keeps more weight bytes in flight.
  // Tensor-bound loads keep 128 x 256.
  const bool narrow = static_cast<long long>(P) <= 16LL * G;
  CUtensorMap ta, tb;
  if ((rc = make_tmap(&tb, w13_bf16, static_cast<long long>(G) * 2 * I, H, narrow ? 64 : 128, op,
                      "w13")) != MOE_OK)
    return rc;
  if (a_row_gather) {
    ta = tb;  // unused: the gatherer warps read A rows directly
  } else if ((rc = make_tmap(&ta, a_bf16, P, H, narrow ? kNarrowRows : BM, op, "a")) !=
             MOE_OK) {
    return rc;
  }
  Params p{};
  p.group_offsets = group_offsets;
  p.P = P;
  p.Kdim = H;
  p.N = I;
  p.G = G;
  p.b_rows_per_group = 2 * I;
  p.half_off = I;
  p.a = static_cast<const uint16_t*>(a_bf16);
  p.a_rows = a_rows;
  p.row_gather = a_row_gather;
  p.gather_div = gather_div;
  p.out = act_bf16;
  p.kid = MOE_KID_GEMM_GATEUP;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a_row_gather && narrow)
    return launch<128, EPI_GATEUP, true, kNarrowRows>(op, ta, tb, p,
                                                      tile_bound(P, G, I, 64, kNarrowRows), s);
  if (a_row_gather)
    return launch<256, EPI_GATEUP, true>(op, ta, tb, p, tile_bound(P, G, I, 128), s);
  if (narrow)
    return launch<128, EPI_GATEUP, false, kNarrowRows>(op, ta, tb, p,
                                                       tile_bound(P, G, I, 64, kNarrowRows), s);
  return launch<256, EPI_GATEUP>(op, ta, tb, p, tile_bound(P, G, I, 128), s);
}

// staged rows: a 256-byte control block (the last launch's flag value, a
// count of finished CTAs), then one flag per 16 routed rows
extern "C" size_t moe_gateup_staged_workspace_size(int P) {
  if (P <= 0) return 0;
  const size_t flags = static_cast<size_t>((P + 15) / 16) * sizeof(int32_t);
  return 256 + ((flags + 255) & ~static_cast<size_t>(255));
}

extern "C" int moe_grouped_gemm_gateup_silu_bf16_staged(
    const void* x_bf16, int T, const int32_t* sorted_pair, int K, void* x_perm_bf16,
    const void* w13_bf16, const int32_t* group_offsets, int P, int H, int I, int G,
    void* act_bf16, void* workspace, size_t ws_bytes, void* stream) {
  clear_error();
  const char* op = "moe_grouped_gemm_gateup_silu_bf16_staged";
  int rc;
  if ((rc = check_common(op, P, H, I, G, x_bf16, w13_bf16, act_bf16)) != MOE_OK) return rc;
  if (!group_offsets && G != 1)
    return set_error(MOE_ERR_ARG, "%s: group_offsets is NULL with G=%d", op, G);
  if (P == 0) return MOE_OK;
  if (T < 1 || K < 1) return set_error(MOE_ERR_ARG, "%s: T=%d and K=%d must be >= 1", op, T, K);
  if (!sorted_pair || !x_perm_bf16)
    return set_error(MOE_ERR_ARG, "%s: sorted_pair or x_perm is NULL", op);
  if (!aligned16(x_perm_bf16))
    return set_error(MOE_ERR_ALIGN, "%s: x_perm must be 16-byte aligned", op);
  const size_t need = moe_gateup_staged_workspace_size(P);
  if (!workspace || ws_bytes < need || !aligned16(workspace))
    return set_error(MOE_ERR_WORKSPACE, "%s: workspace of %zu bytes is smaller than %zu", op,
                     ws_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (use_pair_tiles(P, G)) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    return launch_pair_gateup_staged(op, x_bf16, T, sorted_pair, K, x_perm_bf16, w13_bf16,
                                     group_offsets, P, H, I, G, act_bf16,
                                     reinterpret_cast<int32_t*>(ws + 256),
                                     reinterpret_cast<unsigned int*>(ws), s);
  }
  // single-CTA tiles: the row gather, then the tiles over x_perm
  if ((rc = launch_row_gather(op, x_bf16, T, x_perm_bf16, sorted_pair, P, K, H, s)) != MOE_OK)
    return rc;
  return moe_grouped_gemm_gateup_silu_bf16(x_perm_bf16, P, nullptr, 1, w13_bf16, group_offsets, P,
                                           H, I, G, act_bf16, nullptr, 0, stream);
}

extern "C" int moe_grouped_gemm_down_bf16(const void* act_bf16, const void* w2_bf16,
                                          const int32_t* group_offsets, const float* pair_weight,
                                          const int32_t* row_to_pair, int P, int I, int H, int G,
                                          void* out_bf16, void* workspace, size_t ws_bytes,
                                          void* stream) {
  (void)workspace;
  (void)ws_bytes;
  clear_error();
  const char* op = "moe_grouped_gemm_down_bf16";
  int rc;
  if ((rc = check_common(op, P, I, H, G, act_bf16, w2_bf16, out_bf16)) != MOE_OK) return rc;
  if (!group_offsets && G != 1)
    return set_error(MOE_ERR_ARG, "%s: group_offsets is NULL with G=%d", op, G);
  if (P == 0) return MOE_OK;
  if (use_pair_tiles(P, G))
    return launch_pair_down(op, act_bf16, w2_bf16, group_offsets, pair_weight, row_to_pair, P, I,
                            H, G, out_bf16, static_cast<cudaStream_t>(stream));
  // few rows per expert: 32-row tiles, as in the gate/up GEMM
  const bool narrow = static_cast<long long>(P) <= 16LL * G;
  CUtensorMap ta, tb;
  if ((rc = make_tmap(&ta, act_bf16, P, I, narrow ? kNarrowRows : BM, op, "act")) != MOE_OK)
    return rc;
  if ((rc = make_tmap(&tb, w2_bf16, static_cast<long long>(G) * H, I, 128, op, "w2")) != MOE_OK)
    return rc;
  Params p{};
  p.group_offsets = group_offsets;
  p.P = P;
  p.Kdim = I;
  p.N = H;
  p.G = G;
  p.b_rows_per_group = H;
  p.half_off = 0;
  p.out = out_bf16;
  p.pair_weight = pair_weight;
  p.row_to_pair = row_to_pair;
  p.kid = MOE_KID_GEMM_DOWN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (narrow)
    return launch<256, EPI_DOWN, false, kNarrowRows>(op, ta, tb, p,
                                                     tile_bound(P, G, H, 256, kNarrowRows), s);
  return launch<256, EPI_DOWN>(op, ta, tb, p, tile_bound(P, G, H, 256), s);
}

namespace {

// arguments of the shared expert's half of a fused launch
int check_shared(const char* op, int Ts, int Kdim2, int N2, const void* a2, const void* b2,
                 const void* out2) {
  if (Ts < 0) return set_error(MOE_ERR_ARG, "%s: Ts=%d < 0", op, Ts);
  if (Kdim2 <= 0 || N2 <= 0)
    return set_error(MOE_ERR_ARG, "%s: shared-expert dimensions must be positive", op);
  if (Kdim2 % 8 != 0 || N2 % 8 != 0)
    return set_error(MOE_ERR_ALIGN, "%s: H and I_shared must be multiples of 8", op);
  if (Ts > 0 && (!a2 || !b2 || !out2))
    return set_error(MOE_ERR_ARG, "%s: NULL shared-expert operand", op);
  if (!aligned16(a2) || !aligned16(b2) || !aligned16(out2))
    return set_error(MOE_ERR_ALIGN, "%s: shared-expert operands must be 16-byte aligned", op);
  return MOE_OK;
}

}  // namespace

extern "C" int moe_grouped_gemm_gateup_silu_bf16_shared(
    const void* a_bf16, const void* w13_bf16, const int32_t* group_offsets, int P, int H, int I,
    int G, void* act_bf16, const void* xs_bf16, int Ts, const void* w13s_bf16, int Is,
    void* acts_bf16, void* workspace, size_t ws_bytes, void* stream) {
  clear_error();
  const char* op = "moe_grouped_gemm_gateup_silu_bf16_shared";
  int rc;
  if ((rc = check_common(op, P, H, I, G, a_bf16, w13_bf16, act_bf16)) != MOE_OK) return rc;
  if (!group_offsets && G != 1)
    return set_error(MOE_ERR_ARG, "%s: group_offsets is NULL with G=%d", op, G);
  if ((rc = check_shared(op, Ts, H, Is, xs_bf16, w13s_bf16, acts_bf16)) != MOE_OK) return rc;
  // one side empty: the plain single-problem launches (the same tiles either way)
  if (Ts == 0)
    return moe_grouped_gemm_gateup_silu_bf16(a_bf16, P, nullptr, 1, w13_bf16, group_offsets, P, H,
                                             I, G, act_bf16, workspace, ws_bytes, stream);
  if (P == 0)
    return moe_grouped_gemm_gateup_silu_bf16(xs_bf16, Ts, nullptr, 1, w13s_bf16, nullptr, Ts, H,
                                             Is, 1, acts_bf16, workspace, ws_bytes, stream);
  clear_error();
  CUtensorMap ta, tb, ta2, tb2;
  if ((rc = make_tmap(&ta, a_bf16, P, H, BM, op, "a")) != MOE_OK ||
      (rc = make_tmap(&tb, w13_bf16, static_cast<long long>(G) * 2 * I, H, 128, op, "w13")) !=
          MOE_OK ||
      (rc = make_tmap(&ta2, xs_bf16, Ts, H, BM, op, "xs")) != MOE_OK ||
      (rc = make_tmap(&tb2, w13s_bf16, 2LL * Is, H, 128, op, "w13s")) != MOE_OK)
    return rc;
  Params p{};
  p.group_offsets = group_offsets;
  p.P = P;
  p.Kdim = H;
  p.N = I;
  p.G = G;
  p.b_rows_per_group = 2 * I;
  p.half_off = I;
  p.out = act_bf16;
  p.P2 = Ts;
  p.N2 = Is;
  p.Kdim2 = H;
  p.half_off2 = Is;
  p.out2 = acts_bf16;
  p.kid = MOE_KID_GEMM_GATEUP;
  const long long extra = ((Ts + BM - 1) / BM) * static_cast<long long>((Is + 127) / 128);
  return launch<256, EPI_GATEUP>(op, ta, tb, ta2, tb2, p, tile_bound(P, G, I, 128) + extra,
                                 static_cast<cudaStream_t>(stream));
}

extern "C" int moe_grouped_gemm_down_bf16_shared(
    const void* act_bf16, const void* w2_bf16, const int32_t* group_offsets,
    const float* pair_weight, const int32_t* row_to_pair, int P, int I, int H, int G,
    void* out_bf16, const void* acts_bf16, int Ts, const void* w2s_bf16, int Is, void* sd_bf16,
    void* workspace, size_t ws_bytes, void* stream) {
  clear_error();
  const char* op = "moe_grouped_gemm_down_bf16_shared";
  int rc;
  if ((rc = check_common(op, P, I, H, G, act_bf16, w2_bf16, out_bf16)) != MOE_OK) return rc;
  if (!group_offsets && G != 1)
    return set_error(MOE_ERR_ARG, "%s: group_offsets is NULL with G=%d", op, G);
  if ((rc = check_shared(op, Ts, Is, H, acts_bf16, w2s_bf16, sd_bf16)) != MOE_OK) return rc;
  if (Ts == 0)
    return moe_grouped_gemm_down_bf16(act_bf16, w2_bf16, group_offsets, pair_weight, row_to_pair,
                                      P, I, H, G, out_bf16, workspace, ws_bytes, stream);
  if (P == 0)
    return moe_grouped_gemm_down_bf16(acts_bf16, w2s_bf16, nullptr, nullptr, nullptr, Ts, Is, H,
                                      1, sd_bf16, workspace, ws_bytes, stream);
  clear_error();
  CUtensorMap ta, tb, ta2, tb2;
  if ((rc = make_tmap(&ta, act_bf16, P, I, BM, op, "act")) != MOE_OK ||
      (rc = make_tmap(&tb, w2_bf16, static_cast<long long>(G) * H, I, 128, op, "w2")) !=
          MOE_OK ||
      (rc = make_tmap(&ta2, acts_bf16, Ts, Is, BM, op, "acts")) != MOE_OK ||
      (rc = make_tmap(&tb2, w2s_bf16, H, Is, 128, op, "w2s")) != MOE_OK)
    return rc;
  Params p{};
  p.group_offsets = group_offsets;
  p.P = P;
  p.Kdim = I;
  p.N = H;
  p.G = G;
  p.b_rows_per_group = H;
  p.half_off = 0;
  p.out = out_bf16;
  p.pair_weight = pair_weight;
  p.row_to_pair = row_to_pair;
  p.P2 = Ts;
  p.N2 = H;
  p.Kdim2 = Is;
  p.half_off2 = 0;
  p.out2 = sd_bf16;
  p.kid = MOE_KID_GEMM_DOWN;
  const long long extra = ((Ts + BM - 1) / BM) * static_cast<long long>((H + 255) / 256);
  return launch<256, EPI_DOWN>(op, ta, tb, ta2, tb2, p, tile_bound(P, G, H, 256) + extra,
                               static_cast<cudaStream_t>(stream));
}

namespace {

// FP8 weights: codes and scales present and aligned, dimensions whole 16-byte rows
int check_fp8(const char* op, int rows_per_group, int Kdim, const void* q, const float* scale) {
  if (!q || !scale) return set_error(MOE_ERR_ARG, "%s: FP8 weight codes or scales are NULL", op);
  if (Kdim % 16 != 0)
    return set_error(MOE_ERR_ALIGN, "%s: K=%d of the FP8 weights must be a multiple of 16", op,
                     Kdim);
  if (!aligned16(q) || (reinterpret_cast<uintptr_t>(scale) & 3u))
    return set_error(MOE_ERR_ALIGN, "%s: FP8 codes must be 16-byte, scales 4-byte aligned", op);
  (void)rows_per_group;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_grouped_gemm_gateup_silu_fp8w(const void* a_bf16, const uint8_t* w13_e4m3,
                                                 const float* w13_scale,
                                                 const int32_t* group_offsets, int P, int H,
                                                 int I, int G, void* act_bf16, void* workspace,
                                                 size_t ws_bytes, void* stream) {
  (void)workspace;
  (void)ws_bytes;
  clear_error();
  const char* op = "moe_grouped_gemm_gateup_silu_fp8w";
  int rc;
  if ((rc = check_common(op, P, H, I, G, a_bf16, w13_e4m3, act_bf16)) != MOE_OK) return rc;
  if (!group_offsets && G != 1)
    return set_error(MOE_ERR_ARG, "%s: group_offsets is NULL with G=%d", op, G);
  if (P == 0) return MOE_OK;
  if ((rc = check_fp8(op, 2 * I, H, w13_e4m3, w13_scale)) != MOE_OK) return rc;
  const bool narrow = static_cast<long long>(P) <= 16LL * G;
  CUtensorMap ta, tb;
  if ((rc = make_tmap(&ta, a_bf16, P, H, narrow ? kNarrowRows : BM, op, "a")) != MOE_OK ||
      (rc = make_tmap_u8(&tb, w13_e4m3, static_cast<long long>(G) * 2 * I, H, narrow ? 64 : 128,
                         op, "w13")) != MOE_OK)
    return rc;
  Params p{};
  p.group_offsets = group_offsets;
  p.P = P;
  p.Kdim = H;
  p.N = I;
  p.G = G;
  p.b_rows_per_group = 2 * I;
  p.half_off = I;
  p.out = act_bf16;
  p.b_scale = w13_scale;
  p.scale_rb = (2 * I + 127) / 128;
  p.scale_cb = (H + 127) / 128;
  p.kid = MOE_KID_GEMM_GATEUP;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (narrow)
    return launch<128, EPI_GATEUP, false, kNarrowRows, true>(
        op, ta, tb, p, tile_bound(P, G, I, 64, kNarrowRows), s);
  return launch<256, EPI_GATEUP, false, BM, true>(op, ta, tb, p, tile_bound(P, G, I, 128), s);
}

extern "C" int moe_grouped_gemm_down_fp8w(const void* act_bf16, const uint8_t* w2_e4m3,
                                          const float* w2_scale, const int32_t* group_offsets,
                                          const float* pair_weight, const int32_t* row_to_pair,
                                          int P, int I, int H, int G, void* out_bf16,
                                          void* workspace, size_t ws_bytes, void* stream) {
  (void)workspace;
  (void)ws_bytes;
  clear_error();
  const char* op = "moe_grouped_gemm_down_fp8w";
  int rc;
  if ((rc = check_common(op, P, I, H, G, act_bf16, w2_e4m3, out_bf16)) != MOE_OK) return rc;
  if (!group_offsets && G != 1)
    return set_error(MOE_ERR_ARG, "%s: group_offsets is NULL with G=%d", op, G);
  if (P == 0) return MOE_OK;
  if ((rc = check_fp8(op, H, I, w2_e4m3, w2_scale)) != MOE_OK) return rc;
  const bool narrow = static_cast<long long>(P) <= 16LL * G;
  CUtensorMap ta, tb;
  if ((rc = make_tmap(&ta, act_bf16, P, I, narrow ? kNarrowRows : BM, op, "act")) != MOE_OK ||
      (rc = make_tmap_u8(&tb, w2_e4m3, static_cast<long long>(G) * H, I, 128, op, "w2")) !=
          MOE_OK)
    return rc;
  Params p{};
  p.group_offsets = group_offsets;
  p.P = P;
  p.Kdim = I;
  p.N = H;
  p.G = G;
  p.b_rows_per_group = H;
  p.half_off = 0;
  p.out = out_bf16;
  p.pair_weight = pair_weight;
  p.row_to_pair = row_to_pair;
  p.b_scale = w2_scale;
  p.scale_rb = (H + 127) / 128;
  p.scale_cb = (I + 127) / 128;
  p.kid = MOE_KID_GEMM_DOWN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (narrow)
    return launch<256, EPI_DOWN, false, kNarrowRows, true>(
        op, ta, tb, p, tile_bound(P, G, H, 256, kNarrowRows), s);
  return launch<256, EPI_DOWN, false, BM, true>(op, ta, tb, p, tile_bound(P, G, H, 256), s);
}
