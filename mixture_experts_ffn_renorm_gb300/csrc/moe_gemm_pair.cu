// moe_gemm_pair.cu -- the grouped BF16 GEMMs of the MoE expert block on CTA
// pairs, for batches with many rows per expert (prefill).  Same two ops and
// the same numeric contract as the single-CTA tiles of moe_gemm.cu (vllm.cpp
// issue #3094 "Row: BACKEND-ROCM-BF16-MOE": gate and up narrowed to bf16
// before the activation; the routing weight applied once, before the down
// result is stored).
//
// A tile puts weight rows (output features) on the MMA's M side and routed
// tokens on its N side.  One tcgen05.mma.cta_group::2 with M = 256 spans the
// two SMs of a cluster: each SM holds 128 weight rows (its half of A) and half
// of the tile's tokens (its half of B), and its tensor memory receives its 128
// weight rows x all N tokens.  A tile covers up to 256 consecutive rows of one
// group, with N their count rounded up to 16, so a group is padded to 16 rows
// rather than to a multiple of the 128 or 256 rows of a token-major tile.  Per
// SM and 64-wide K step a stage holds 16 KB of weights and at most 16 KB of
// tokens, against 48 KB for a 128 x 256 single-CTA tile doing the same MMA
// work, so the shared-memory fill per MMA drops by a third.
//
//   warp 0      TMA producer, in both CTAs: each loads its own half of every
//               stage, and the bytes of both halves are counted on the even
//               CTA's stage barrier
//   warp 1      TMEM allocation in both CTAs; in the even CTA, the one thread
//               that issues the pair's MMAs
//   warps 2-9   epilogue, in both CTAs: two groups of four warps take a tile's
//               32-token chunks in turn; tcgen05.ld of 32 tokens of one weight
//               row per thread, the fused op, and a transpose through shared
//               memory into token-major output rows stored as 16-byte vectors
//
//   warps 10-11 (gate/up with gathered rows only) cp.async copies of the CTA's
//               token rows straight from x: routed row r is row
//               row_gather[r] / gather_div of x, so no permuted copy of x is
//               needed.  The copies land in the 128-byte-swizzled layout of the
//               TMA token box and report on an mbarrier as they complete: in the
//               even CTA the stage's full barrier itself; in the odd CTA a
//               barrier of its own, which warp 1 relays to the even CTA's full
//               barrier after a proxy fence.
//   warps 10-12 (gate/up with staged rows only) warps 10-11 of every CTA write
//               x_perm rows from x, 16-row chunks in row order spread over the
//               grid, each chunk released through a flag in global memory;
//               warp 12 watches the flags of the chunks this CTA's tiles read and
//               counts the ready tiles in shared memory, and the producer reads
//               that count once per tile before it loads the tile's token boxes
//               from x_perm.  The flags carry a value one past the last launch's
//               (kept in the caller's workspace), so no reset is needed between
//               calls.
//
// gate/up: a CTA's 128 weight rows are the up rows of 64 output features
// followed by the gate rows of the same 64, so TMEM lanes 0-63 hold up and
// lanes 64-127 gate.  The warps that read up lanes narrow them to bf16 and pass
// them through shared memory to the warps that read the matching gate lanes,
// which do the SiLU-mul.  Warp w issues on the SM's sub-partition w % 4 and
// may read only TMEM lane quarter w % 4, so this order puts the SiLU work on
// sub-partitions 2 and 3 and keeps 0 and 1, where the producer and the MMA
// issuer run, for the light narrowing warps: the ring is latency-bound, and
// every issue slot the producer waits for lengthens its round trip.
//
// The tile schedule is built on the device from the group offsets, as in
// moe_gemm.cu: groups in order, each group's token blocks of 256, each block's
// feature blocks; pair u takes tiles u, u + pairs, ...  Waits are bounded like
// moe_gemm.cu's; a CTA that gives up tells its peer, the MMAs are drained, and
// both CTAs let their in-flight copies land before they free tensor memory.
#include <atomic>

#include "gemm_common.cuh"

namespace moe {
namespace gemm {
namespace {

constexpr int kPairThreads = 320;     // producer, MMA, two groups of four epilogue warps
constexpr int kGatherThreads = 64;    // + two warps that gather token rows (on sub-partitions 2, 3)
// staged rows: + two stager warps (sub-partitions 2, 3) and one watcher warp
constexpr int kStagedThreads = 96;
constexpr int kStageRows = 16;        // routed rows per staging chunk (one ready flag each)

// Where a gate/up launch takes its token rows from: TMA boxes of a permuted
// matrix the caller wrote (x_perm); 16-byte cp.async copies from x by gatherer
// warps; or TMA boxes of x_perm that stager warps of the same launch write from
// x, chunk by chunk, ahead of the tiles that read them.
enum PairSrc { SRC_TMA = 0, SRC_GATHER = 1, SRC_STAGED = 2 };

__host__ __device__ constexpr int pair_threads(int src) {
  return kPairThreads + (src == SRC_GATHER ? kGatherThreads : src == SRC_STAGED ? kStagedThreads : 0);
}
constexpr int kTokBlock = 256;        // tokens per tile at most (MMA N)
// token rows per TMA box: three tensor maps over the token rows, with boxes of
// 32, 64 and 128 rows; a stage takes the smallest that covers its N / 2 rows
constexpr int kTokBoxMin = 32;
// gate/up: the last token block of a group with at most kShortTok rows is a
// short block; its tiles take two feature blocks each (the weights of the
// second fill the stage's token slot, its token rows a 2 KB side slot), so a
// short block costs half the tiles and twice the weight rows per stage
constexpr int kShortTok = 32;
constexpr int kSideBytes = 16 * BK * 2;   // one CTA's token rows of a short tile's stage
constexpr int kPStages = 6;
constexpr int kWBytes = 128 * BK * 2; // one CTA's weight rows per stage: 16 KB
constexpr int kTBytes = 128 * BK * 2; // one CTA's token rows per stage, at most: 16 KB
// after a CTA gives up: how long it lets its TMA copies land before the pair
// frees its shared and tensor memory (copies are counted on the even CTA's
// barriers, so the odd CTA cannot wait for its own copies directly)
constexpr unsigned long long kCopyGraceNs = 100000ull;

enum PairEpi { PEPI_GATEUP = 0, PEPI_DOWN = 1 };

struct PairParams {
  const int32_t* group_offsets;  // [G+1], or null: one group [0, P)
  int P;                         // routed rows (tokens of the product)
  int Kdim;                      // contraction length
  int N;                         // output columns (I for gate/up, H for down)
  int G;
  int w_rows_per_group;          // rows of the weight matrix per group (2I or H)
  int half_off;                  // gate/up: offset of the up rows inside a group (I)
  void* out;                     // bf16 [P, N] (down: rows by dst)
  const float* pair_weight;      // down: [P] by destination row, or null
  const int32_t* row_to_pair;    // down: destination row of each product row, or null
  const uint16_t* a;             // gathered rows: x [a_rows, Kdim] bf16
  int a_rows;
  const int32_t* row_gather;     // gathered rows: routed row r is x row row_gather[r] / gather_div
  int gather_div;
  uint16_t* stage_out;           // staged rows: x_perm [P, Kdim], written by the stagers
  int32_t* stage_flags;          // staged rows: [ceil(P / kStageRows)] chunk flags
  unsigned int* stage_ctl;       // staged rows: [0] epoch of the last launch, [1] CTAs done
  unsigned long long wait_ns;
  unsigned int* status;
  unsigned long long* launches;
  int kid;
};

struct PSmem {
  static constexpr int STAGE_W = 0;                                  // kPStages x 16 KB
  static constexpr int STAGE_T = STAGE_W + kPStages * kWBytes;       // kPStages x 16 KB
  static constexpr int EPI = STAGE_T + kPStages * kTBytes;           // 2 groups x 8 KB
  static constexpr int META_DST = EPI + 2 * 8192;                    // down: int[2][256]
  static constexpr int META_W = META_DST + 2 * kTokBlock * 4;        // down: float[2][256]
  // gate/up short tiles: kPStages side slots of token rows (over the down's META)
  static constexpr int SIDE = EPI + 2 * 8192;
  // full[kPStages], empty[kPStages], tfull[2], tempty[2], drain, gathered[kPStages]
  static constexpr int BARS = SIDE + kPStages * kSideBytes;
  static constexpr int NBARS = 3 * kPStages + 5;
  // tmem slot, abort flag, scan (one int per warp), staged rows: ready tiles, epoch
  static constexpr int MISC = BARS + NBARS * 8;
  static constexpr int TILE_START = MISC + 128;
  static constexpr int GOFF = TILE_START + (kMaxPairGroups + 1) * 4;
  static constexpr int BYTES = GOFF + (kMaxPairGroups + 1) * 4;
  static constexpr int ALLOC = BYTES + 1024;
};
static_assert(PSmem::META_W + 2 * kTokBlock * 4 <= PSmem::BARS, "down's META inside SIDE");
static_assert(PSmem::SIDE % 1024 == 0, "side slots on the 128-byte swizzle's 1 KB atoms");
static_assert(PSmem::ALLOC <= 227 * 1024, "pair GEMM shared memory");

struct PTile {
  int g, r0, n_tok, n0;
  int nblk;   // feature blocks of the tile: 1, or 2 for a short block's tile
};

// tiles of a group of `rows` rows: its token blocks times n_fb feature blocks,
// the short last block (shorts) taking its feature blocks two at a time
__device__ __forceinline__ int pair_group_tiles(int rows, int n_fb, bool shorts) {
  if (rows <= 0) return 0;
  const int m = (rows + kTokBlock - 1) / kTokBlock;
  const int last = rows - (m - 1) * kTokBlock;
  return (m - 1) * n_fb + (shorts && last <= kShortTok ? (n_fb + 1) / 2 : n_fb);
}

__device__ __forceinline__ PTile pair_tile(int tile, const int* tile_start, const int* goff, int G,
                                           int n_fb, int fb_cols, bool shorts) {
  int lo = 0, hi = G;  // tile_start[lo] <= tile < tile_start[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid;
  }
  const int local = tile - tile_start[lo];
  const int rows = goff[lo + 1] - goff[lo];
  const int m_last = (rows - 1) / kTokBlock;          // the group's last token block
  const int last = rows - m_last * kTokBlock;
  PTile t;
  t.g = lo;
  if (shorts && last <= kShortTok && local >= m_last * n_fb) {
    const int j = local - m_last * n_fb;               // two feature blocks: 2j, 2j + 1
    t.r0 = goff[lo] + m_last * kTokBlock;
    t.n_tok = last;
    t.n0 = 2 * j * fb_cols;
    t.nblk = min(2, n_fb - 2 * j);
    return t;
  }
  const int m = local / n_fb;
  t.r0 = goff[lo] + m * kTokBlock;
  t.n_tok = min(goff[lo + 1], t.r0 + kTokBlock) - t.r0;
  t.n0 = (local - m * n_fb) * fb_cols;
  t.nblk = 1;
  return t;
}

// staged rows: bounded wait of the producer until the watcher has published
// more than `n` ready tiles (a shared-memory counter; acquire at CTA scope)
__device__ __forceinline__ bool wait_ready(uint32_t s_ready, uint32_t n, volatile int* abort_flag,
                                           unsigned int* status, unsigned long long limit_ns) {
  if (ptx::ld_acquire_cta_shared_u32(s_ready) > n) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (ptx::ld_acquire_cta_shared_u32(s_ready) > n) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      if (status) atomicOr(status, static_cast<unsigned int>(MOE_STATUS_TIMEOUT));
      *abort_flag = 1;
      return false;
    }
  }
}

// staged rows: bounded wait of the watcher until a chunk's flag holds this
// launch's value (set by a stager of any CTA; acquire at GPU scope)
__device__ __forceinline__ bool wait_flag(const int32_t* flag, uint32_t want,
                                          volatile int* abort_flag, unsigned int* status,
                                          unsigned long long limit_ns) {
  if (ptx::ld_acquire_gpu_u32(flag) == want) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    __nanosleep(64);
    if (ptx::ld_acquire_gpu_u32(flag) == want) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      if (status) atomicOr(status, static_cast<unsigned int>(MOE_STATUS_TIMEOUT));
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

// kEpi: PEPI_GATEUP (weights W13 [G, 2I, K], fb_cols = 128 output features per
// tile, 64 per CTA) or PEPI_DOWN (weights W2 [G, H, K], 256 per tile, 128 per CTA).
// kSrc (PairSrc): where the token rows come from; gathered and staged rows are
// gate/up only.
template <int kEpi, int kSrc>
__global__ void __launch_bounds__(pair_threads(kSrc), 1)
pair_gemm_kernel(const __grid_constant__ CUtensorMap tmT16,
                 const __grid_constant__ CUtensorMap tmT32,
                 const __grid_constant__ CUtensorMap tmT64,
                 const __grid_constant__ CUtensorMap tmT128,
                 const __grid_constant__ CUtensorMap tmW, const PairParams p) {
  constexpr bool kGU = kEpi == PEPI_GATEUP;
  constexpr bool kGather = kSrc == SRC_GATHER;
  constexpr bool kStaged = kSrc == SRC_STAGED;
  // short blocks' tiles take two feature blocks (gate/up with TMA token boxes)
  constexpr bool kShorts = kGU && !kGather;
  static_assert(kGU || kSrc == SRC_TMA, "gathered or staged token rows: gate/up only");
  constexpr int kNT = pair_threads(kSrc);
  constexpr int kFbCols = kGU ? 128 : 256;   // output features per tile (both CTAs)
  constexpr int kWBox = kGU ? 64 : 128;      // weight rows per TMA box
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PSmem::BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + PSmem::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + PSmem::MISC + 4);
  int* scan_tmp = reinterpret_cast<int*>(smem + PSmem::MISC + 8);   // one int per warp
  // staged rows: how many of this CTA's tiles have their rows staged (watcher ->
  // producer), and this launch's flag value
  const uint32_t s_ready = ptx::smem_u32(smem + PSmem::MISC + 64);
  volatile uint32_t* s_epoch = reinterpret_cast<volatile uint32_t*>(smem + PSmem::MISC + 68);
  int* tile_start = reinterpret_cast<int*>(smem + PSmem::TILE_START);
  int* goff = reinterpret_cast<int*>(smem + PSmem::GOFF);
  int* s_dst = reinterpret_cast<int*>(smem + PSmem::META_DST);
  float* s_w = reinterpret_cast<float*>(smem + PSmem::META_W);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int unit = static_cast<int>(blockIdx.x >> 1);
  const int n_units = static_cast<int>(gridDim.x >> 1);
  const unsigned long long wait_ns = p.wait_ns;
  auto bar_full = [&](int s) { return ptx::smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return ptx::smem_u32(bars + kPStages + s); };
  auto bar_tfull = [&](int a) { return ptx::smem_u32(bars + 2 * kPStages + a); };
  auto bar_tempty = [&](int a) { return ptx::smem_u32(bars + 2 * kPStages + 2 + a); };
  const uint32_t bar_drain = ptx::smem_u32(bars + 2 * kPStages + 4);
  auto bar_gath = [&](int s) { return ptx::smem_u32(bars + 2 * kPStages + 5 + s); };

  count_launch(p.launches, p.kid);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      // the even CTA's expect-tx arrive; with gathered rows also one arrive per
      // gatherer of the even CTA and the odd CTA's relay
      ptx::mbar_init(bar_full(s), kGather && leader ? 2 + kGatherThreads : 1);
      ptx::mbar_init(bar_empty(s), 1);   // the pair's MMA commit
      if (kGather) ptx::mbar_init(bar_gath(s), kGatherThreads);  // this CTA's gatherers
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(bar_tfull(a), 1);
      ptx::mbar_init(bar_tempty(a), 16);  // one arrive per epilogue warp of both CTAs
    }
    ptx::mbar_init(bar_drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (kShorts) ptx::tma_prefetch_desc(&tmT16);
    ptx::tma_prefetch_desc(&tmT32);
    ptx::tma_prefetch_desc(&tmT64);
    ptx::tma_prefetch_desc(&tmT128);
    ptx::tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    ptx::tmem_alloc2(ptx::smem_u32(tmem_slot), 2 * kTokBlock);
    ptx::tmem_relinquish2();
  }

  grid_dep_wait();
  grid_dep_launch();
  // staged rows: the flag value of this launch is one past the last launch's;
  // the last CTA of this launch records it at exit (every CTA reads it first,
  // after the previous grid has completed)
  if (kStaged && threadIdx.x == 0) {
    *s_epoch = *reinterpret_cast<volatile uint32_t*>(p.stage_ctl) + 1u;
    ptx::st_release_cta_shared_u32(s_ready, 0u);
  }

  // ---- device-side tile schedule (every CTA computes the same one)
  const int G = p.G;
  for (int g = threadIdx.x; g <= G; g += kNT)
    goff[g] = p.group_offsets ? __ldg(p.group_offsets + g) : (g == 0 ? 0 : p.P);
  __syncthreads();
  const int n_fb = (p.N + kFbCols - 1) / kFbCols;
  const int chunk = (G + kNT - 1) / kNT;
  const int g_lo = min(G, static_cast<int>(threadIdx.x) * chunk);
  const int g_hi = min(G, g_lo + chunk);
  int local = 0;
  for (int g = g_lo; g < g_hi; ++g) local += pair_group_tiles(goff[g + 1] - goff[g], n_fb, kShorts);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scan_tmp[warp] = incl;
  __syncthreads();
  int warp_base = 0, total = 0;
  for (int w = 0; w < kNT / 32; ++w) {
    const int v = scan_tmp[w];
    if (w < warp) warp_base += v;
    total += v;
  }
  int run = warp_base + incl - local;
  for (int g = g_lo; g < g_hi; ++g) {
    tile_start[g] = run;
    run += pair_group_tiles(goff[g + 1] - goff[g], n_fb, kShorts);
  }
  if (threadIdx.x == 0) tile_start[G] = total;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the peer's barriers exist before any remote arrive or copy
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int nk = (p.Kdim + BK - 1) / BK;

  bool mma_any = false;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Lane 0 waits for the stage and arms the even CTA's barrier; then the
    // stage's boxes (weight rows in one or two boxes, token rows in one unless
    // the gatherers copy them; a short tile's second feature block in two more)
    // are issued by lanes 0-4 as a single warp instruction.
    int stage = 0;
    uint32_t phase = 0;
    uint32_t n_tile = 0;
    bool ok = true;
    for (int tile = unit; ok && tile < total; tile += n_units, ++n_tile) {
      if (kStaged) {
        // the tile's rows of x_perm are staged (the watcher has seen their flags)
        bool rdy = true;
        if (lane == 0) rdy = wait_ready(s_ready, n_tile, abort_flag, p.status, wait_ns);
        if (!__shfl_sync(0xffffffffu, rdy ? 1 : 0, 0)) {
          ok = false;
          break;
        }
      }
      const PTile t = pair_tile(tile, tile_start, goff, G, n_fb, kFbCols, kShorts);
      const bool sh = kShorts && t.n_tok <= kShortTok;   // a short block's tile
      const int half = ((t.n_tok + 15) & ~15) >> 1;      // tokens this CTA holds
      const int tbox = sh ? 16 : (half <= 32 ? 32 : (half <= 64 ? 64 : 128));
      const CUtensorMap* mt =
          sh ? &tmT16 : (tbox == 32 ? &tmT32 : (tbox == 64 ? &tmT64 : &tmT128));
      const uint32_t bytes = (sh ? t.nblk : 1) * kWBytes + (kGather ? 0 : tbox * (BK * 2));
      const int trow = t.r0 + static_cast<int>(rank) * half;
      // this CTA's 128 weight rows: gate/up, the 64 up rows of its features
      // then their 64 gate rows; down, 128 consecutive output rows
      const int wrow_g = t.g * p.w_rows_per_group + t.n0 + static_cast<int>(rank) * (kFbCols / 2);
      // this lane's box: lane 0 the first weight box (up rows, or the down rows),
      // lane 1 the gate box, lane 2 the tokens (a short tile's into its side
      // slot); lanes 3 and 4 the up and gate boxes of a short tile's second
      // feature block, into the stage's token slot
      const bool issues = lane == 0 || (!kGather && lane == 2) || (kGU && lane == 1) ||
                          (sh && t.nblk == 2 && (lane == 3 || lane == 4));
      const int wl = lane >= 3 ? lane - 3 : lane;        // box within its feature block
      const int wrow_l = wrow_g + (lane >= 3 ? kFbCols : 0);
      const CUtensorMap* mbox = lane == 2 ? mt : &tmW;
      const int ybox = lane == 2 ? trow : (kGU && wl == 0 ? wrow_l + p.half_off : wrow_l);
      const uint32_t dbox = lane == 2 ? (sh ? PSmem::SIDE : PSmem::STAGE_T)
                                      : (lane >= 3 ? PSmem::STAGE_T : PSmem::STAGE_W) +
                                            wl * (kWBox * 128);
      const uint32_t dstep = lane == 2 ? (sh ? kSideBytes : kTBytes) : (lane >= 3 ? kTBytes : kWBytes);
      for (int kb = 0; kb < nk; ++kb) {
        bool got = true;
        if (lane == 0) {
          // spinning: the producer's reaction time is part of the ring's round trip
          got = wait_bar_spin(bar_empty(stage), phase ^ 1u, abort_flag, p.status, wait_ns);
          if (got && leader) ptx::mbar_arrive_expect_tx(bar_full(stage), 2 * bytes);
        }
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (issues)
          ptx::tma_load_2d_pair(sbase + dbox + stage * dstep, mbox, kb * BK, ybox,
                                ptx::mapa_shared(bar_full(stage), 0));
        if (++stage == kPStages) { stage = 0; phase ^= 1u; }
      }
    }
    (void)n_tile;
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t uses0 = 0, uses1 = 0;
      int acc = 0;
      bool ok = true;
      for (int tile = unit; ok && tile < total; tile += n_units) {
        const PTile t = pair_tile(tile, tile_start, goff, G, n_fb, kFbCols, kShorts);
        const bool sh = kShorts && t.n_tok <= kShortTok;
        const bool two = sh && t.nblk == 2;
        const int N = (t.n_tok + 15) & ~15;
        const uint32_t idesc = ptx::idesc_bf16_f32(256, N);
        if (!wait_bar<true>(bar_tempty(acc), ((acc ? uses1 : uses0) & 1u) ^ 1u, abort_flag,
                            p.status, wait_ns)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kTokBlock);
        for (int kb = 0; kb < nk; ++kb) {
          if (!wait_bar(bar_full(stage), phase, abort_flag, p.status, wait_ns)) {
            ok = false;
            break;
          }
          // gathered rows: the even CTA's cp.async writes, observed through the
          // barrier, ordered before the tensor core's reads
          if (kGather) ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          const uint64_t dw = ptx::desc_kmajor_sw128(sbase + PSmem::STAGE_W + stage * kWBytes);
          // a short tile's tokens sit in the side slot, its second feature
          // block's weights in the token slot (accumulated 128 columns on)
          const uint64_t dt = ptx::desc_kmajor_sw128(
              sbase + (sh ? PSmem::SIDE + stage * kSideBytes : PSmem::STAGE_T + stage * kTBytes));
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            ptx::mma_bf16_pair(d, dw + 2ull * k, dt + 2ull * k, idesc, (kb | k) != 0 ? 1u : 0u);
          if (two) {
            const uint64_t dw2 = ptx::desc_kmajor_sw128(sbase + PSmem::STAGE_T + stage * kTBytes);
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k)
              ptx::mma_bf16_pair(d + 128u, dw2 + 2ull * k, dt + 2ull * k, idesc,
                                 (kb | k) != 0 ? 1u : 0u);
          }
          mma_any = true;
          ptx::mma_commit_pair(bar_empty(stage), 3);   // frees the stage in both CTAs
          if (++stage == kPStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit_pair(bar_tfull(acc), 3);       // the accumulator is ready in both
        if (acc) ++uses1;
        else ++uses0;
        acc ^= 1;
      }
    } else if (kGather && lane == 0 && !leader) {
      // ---------------------------------------------------------- relay (odd CTA)
      // Once this CTA's gatherers have landed a stage (observed through the
      // barrier), fence their writes for the tensor core and arrive on the even
      // CTA's full barrier of the stage.  The arrive is relaxed: the copies are
      // already performed and fenced when it is made, and a release at cluster
      // scope on every stage measured 2.6 times slower for the whole GEMM.
      const uint32_t full_leader = ptx::mapa_shared(bar_full(0), 0);  // + 8 * stage
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = unit; ok && tile < total; tile += n_units) {
        for (int kb = 0; kb < nk; ++kb) {
          if (!wait_bar_spin(bar_gath(stage), phase, abort_flag, p.status, wait_ns)) {
            ok = false;
            break;
          }
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive_remote_relaxed(full_leader + 8u * stage);
          if (++stage == kPStages) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (kStaged && warp >= kPairThreads / 32 && warp < kPairThreads / 32 + 2) {
    // ------------------------------------------------------------ stagers
    // Warps 10 and 11 of every CTA copy routed rows of x into x_perm, one
    // chunk of kStageRows rows at a time: stager s of the grid takes chunks
    // s, s + stagers, ... (in row order, so the chunks the first tiles of every
    // pair read come first).  A row is 16-byte vectors, lanes striding over it,
    // two rows' loads in flight before their stores.  When its chunk is written
    // each lane fences its stores for the async proxy (TMA reads them) and for
    // the GPU, and lane 0 releases the chunk's flag with this launch's value.
    const int gs = static_cast<int>(blockIdx.x) * 2 + (warp - kPairThreads / 32);
    const int n_stagers = static_cast<int>(gridDim.x) * 2;
    const int n_chunks = (p.P + kStageRows - 1) / kStageRows;
    const int vpr = p.Kdim / 8;                   // 16-byte vectors per row
    const uint32_t epoch = *s_epoch;
    const uint4* x = reinterpret_cast<const uint4*>(p.a);
    uint4* xp = reinterpret_cast<uint4*>(p.stage_out);
    for (int c = gs; c < n_chunks && !*abort_flag; c += n_stagers) {
      const int r0 = c * kStageRows, nr = min(kStageRows, p.P - r0);
      int my_src = -1;                            // lane i: source row of row r0 + i
      if (lane < nr) {
        const int sr = __ldg(p.row_gather + r0 + lane) / p.gather_div;
        my_src = sr >= 0 && sr < p.a_rows ? sr : -1;
      }
      for (int i = 0; i < nr; i += 2) {
        const int s0 = __shfl_sync(0xffffffffu, my_src, i);
        const int s1 = __shfl_sync(0xffffffffu, my_src, (i + 1) & 31);
        const bool two = i + 1 < nr;
        for (int v0 = lane; v0 < vpr; v0 += 32 * 8) {
          uint4 a[8], b[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int v = v0 + 32 * q;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            a[q] = (v < vpr && s0 >= 0) ? __ldg(x + static_cast<size_t>(s0) * vpr + v) : z;
            b[q] = (v < vpr && two && s1 >= 0) ? __ldg(x + static_cast<size_t>(s1) * vpr + v) : z;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int v = v0 + 32 * q;
            if (v < vpr) {
              xp[static_cast<size_t>(r0 + i) * vpr + v] = a[q];
              if (two) xp[static_cast<size_t>(r0 + i + 1) * vpr + v] = b[q];
            }
          }
        }
      }
      ptx::fence_proxy_async_global();
      __threadfence();
      __syncwarp();
      if (lane == 0) ptx::st_release_gpu_u32(p.stage_flags + c, epoch);
    }
  } else if (kStaged && warp == kPairThreads / 32 + 2) {
    // ------------------------------------------------------------ watcher
    // Lane 0 walks this CTA's tiles ahead of the producer: once every chunk
    // holding the CTA's rows of a tile carries this launch's flag value, it
    // fences for the async proxy and publishes the count of ready tiles.
    if (lane == 0) {
      const uint32_t epoch = *s_epoch;
      uint32_t n_ready = 0;
      bool ok = true;
      for (int tile = unit; ok && tile < total; tile += n_units) {
        const PTile t = pair_tile(tile, tile_start, goff, G, n_fb, kFbCols, kShorts);
        const int half = ((t.n_tok + 15) & ~15) >> 1;
        const int lo = t.r0 + static_cast<int>(rank) * half;        // this CTA's rows
        const int cnt = min(half, t.n_tok - static_cast<int>(rank) * half);  // real ones
        if (cnt > 0) {
          for (int c = lo / kStageRows; ok && c <= (lo + cnt - 1) / kStageRows; ++c)
            ok = wait_flag(p.stage_flags + c, epoch, abort_flag, p.status, wait_ns);
          if (!ok) break;
          ptx::fence_proxy_async_global();
        }
        ptx::st_release_cta_shared_u32(s_ready, ++n_ready);
      }
    }
  } else if (kGather && warp >= kPairThreads / 32) {
    // ------------------------------------------------------------ token-row gatherers
    // Warp gw copies rows [64 gw, 64 gw + 64) of this CTA's half of the tile's
    // tokens: each warp instruction moves four rows, lane l the 16-byte chunk
    // l % 8 of row l / 8 (128 contiguous bytes per row), into the slot chunk
    // c ^ (row % 8) that the 128-byte swizzle gives it.  Tokens past the tile's
    // end, and rows outside [0, a_rows), are written as zeros.  The copies go
    // through the SM's load/store path, which moves about two thirds of the
    // token bytes a stage ring fed by TMA boxes of a permuted matrix takes in
    // the same time; the gatherers spin on the stage barrier, since their
    // reaction time adds to every stage's round trip.
    const int gw = warp - kPairThreads / 32;
    const int c = lane & 7;
    const int rsub = lane >> 3;
    const uint16_t* a = p.a;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = unit; ok && tile < total; tile += n_units) {
      const PTile t = pair_tile(tile, tile_start, goff, G, n_fb, kFbCols, kShorts);
      const int half = ((t.n_tok + 15) & ~15) >> 1;      // rows this CTA holds (multiple of 8)
      const int tok0 = static_cast<int>(rank) * half;    // its first token of the tile
      const int n_m = max(0, min(16, (half - 64 * gw) >> 2));  // warp instructions per stage
      int src[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const int tok = tok0 + 64 * gw + 4 * m + rsub;
        int r = -1;
        if (m < n_m && tok < t.n_tok) {
          r = __ldg(p.row_gather + t.r0 + tok) / p.gather_div;
          if (r >= p.a_rows) r = -1;
        }
        src[m] = r;
      }
      for (int kb = 0; kb < nk; ++kb) {
        const bool got = wait_bar_spin(bar_empty(stage), phase ^ 1u, abort_flag, p.status, wait_ns);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint32_t dst = sbase + PSmem::STAGE_T + stage * kTBytes;
        const int col = kb * BK + 8 * c;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          if (m < n_m) {
            const int j = 64 * gw + 4 * m + rsub;
            const bool live = src[m] >= 0 && col < p.Kdim;  // Kdim % 8 == 0: all in or out
            ptx::cp_async_16(dst + j * 128 + ((c ^ (j & 7)) << 4),
                             a + (live ? static_cast<size_t>(src[m]) * p.Kdim + col : 0),
                             live ? 16u : 0u);
          }
        }
        ptx::cp_async_mbar_arrive_noinc(leader ? bar_full(stage) : bar_gath(stage));
        if (++stage == kPStages) { stage = 0; phase ^= 1u; }
      }
    }
    ptx::cp_async_wait_all();   // nothing of this thread lands after the CTA's exit
  } else if (warp < kPairThreads / 32) {
    // ------------------------------------------------------------ epilogue
    // Two groups of four warps (2-5 and 6-9) take the tile's 32-token chunks in
    // turn, each with its own staging buffers and named barrier; all eight meet
    // once per tile (barrier 3) to decide together and to publish the tile's
    // destination rows and weights.
    const int eg = (warp - 2) >> 2;                              // epilogue group
    const int et = static_cast<int>(threadIdx.x) - 64 - 128 * eg;  // 0..127 in the group
    const int ea = static_cast<int>(threadIdx.x) - 64;           // 0..255 over both
    const int q = warp & 3;                                      // TMEM lane quarter
    const bool is_up = kGU && q < 2;
    // feature of this thread's TMEM lane within the CTA's output columns
    const int f = kGU ? (q & 1) * 32 + lane : q * 32 + lane;
    const int bar_g = 1 + eg;
    const uint32_t tempty_leader = ptx::mapa_shared(bar_tempty(0), 0);  // + 8 * acc
    const uint32_t epi = sbase + PSmem::EPI + eg * 8192;
    const uint32_t xch = epi;                     // gate/up: up rows, 64 x 32 bf16 (4 KB)
    const uint32_t ost = kGU ? epi + 4096 : epi;  // output staging, token-major
    // this thread's 16-bit slot in staging row j, for each j modulo the swizzle
    // period (16-byte pieces XOR-swizzled by the row)
    constexpr int kRowB = kGU ? 128 : 256;
    constexpr int kSw = kRowB / 16;
    uint32_t slot[kSw];
#pragma unroll
    for (int jj = 0; jj < kSw; ++jj) slot[jj] = ost + (((f >> 3) ^ jj) << 4) + (f & 7) * 2;
    uint32_t uses0 = 0, uses1 = 0;
    int acc = 0;
    // down: the destination row of this thread's token slot of the next tile,
    // loaded a tile ahead so its latency hides behind the accumulator wait
    auto dst_of = [&](const PTile& nt) {
      const int r = nt.r0 + ea;
      return ea < nt.n_tok ? (p.row_to_pair ? __ldg(p.row_to_pair + r) : r) : -1;
    };
    int nd = -1;
    if (!kGU && unit < total) nd = dst_of(pair_tile(unit, tile_start, goff, G, n_fb, kFbCols, kShorts));
    for (int tile = unit; tile < total; tile += n_units) {
      const PTile t = pair_tile(tile, tile_start, goff, G, n_fb, kFbCols, kShorts);
      // A short tile's two feature blocks are accumulated 128 columns apart;
      // group eg takes block eg, all its tokens in one chunk.  Otherwise the
      // groups take the tile's 32-token chunks in turn.
      const bool sh = kShorts && t.n_tok <= kShortTok;
      const bool has = sh ? eg < t.nblk : 32 * eg < t.n_tok;
      const int jbeg = sh ? 0 : 32 * eg;
      const int jstep = sh ? kTokBlock : 64;
      const uint32_t tcol = sh ? static_cast<uint32_t>(eg * 128) : 0u;
      // this CTA's first output column
      const int col0 = t.n0 + (sh ? eg * kFbCols : 0) + static_cast<int>(rank) * (kFbCols / 2);
      int* dst_t = s_dst + acc * kTokBlock;     // meta of this tile (double-buffered by slot)
      float* w_t = s_w + acc * kTokBlock;
      int d = -1;
      float w = 1.0f;
      if (!kGU) {
        d = nd;
        if (p.pair_weight && d >= 0) w = __ldg(p.pair_weight + d);
        if (tile + n_units < total)
          nd = dst_of(pair_tile(tile + n_units, tile_start, goff, G, n_fb, kFbCols, kShorts));
      }
      const bool landed =
          wait_bar(bar_tfull(acc), (acc ? uses1 : uses0) & 1u, abort_flag, p.status, wait_ns);
      if (!kGU && d >= 0) {
        // this buffer's last readers (two tiles ago) passed the previous tile's barrier 3
        dst_t[ea] = d;
        w_t[ea] = w;
      }
      // one decision for the eight warps; the barrier also publishes dst_t / w_t
      if (!ptx::bar_and(3, 256, landed)) {
        *abort_flag = 1;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kTokBlock);
      if (!has) {  // no chunk for this group: its warps free the accumulator now
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_remote_relaxed(tempty_leader + 8u * acc);
      }
#pragma unroll 1
      for (int j0 = jbeg; has && j0 < t.n_tok; j0 += jstep) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + tcol + static_cast<uint32_t>(j0), v);
        ptx::tmem_ld_wait();
        if (j0 + jstep >= t.n_tok) {  // this warp's last TMEM read of the tile: free the accumulator
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive_remote_relaxed(tempty_leader + 8u * acc);
        }
        if (kGU) {
          if (is_up) {
            // up values narrowed to bf16, row f of the exchange buffer (16-byte
            // pieces XOR-swizzled by (f / 2) % 4 against bank conflicts)
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
#pragma unroll
            for (int k = 0; k < 4; ++k)
              ptx::st_shared_v4(xch + f * 64 + ((k ^ ((f >> 1) & 3)) << 4), pk[4 * k],
                                pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
          }
          ptx::bar_sync(bar_g, 128);
          if (!is_up) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint4 u4 = ptx::ld_shared_v4(xch + f * 64 + ((k ^ ((f >> 1) & 3)) << 4));
              const uint32_t uw[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const int i = 4 * k + m;            // tokens 2i and 2i + 1
                // narrowing before the activation: gate (here) and up (there) are bf16
                const uint32_t gp =
                    pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                const float g0 = __uint_as_float(gp << 16), g1 = __uint_as_float(gp & 0xFFFF0000u);
                const float u0 = __uint_as_float(uw[m] << 16);
                const float u1 = __uint_as_float(uw[m] & 0xFFFF0000u);
                // SiLU is tolerance-checked: the fast reciprocal division serves
                const float a0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
                const float a1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
                const uint32_t ap = pack_bf16x2(a0, a1);
                const int j = 2 * i;
                ptx::st_shared_u16(slot[j & (kSw - 1)] + j * kRowB,
                                   static_cast<uint16_t>(ap & 0xFFFFu));
                ptx::st_shared_u16(slot[(j + 1) & (kSw - 1)] + (j + 1) * kRowB,
                                   static_cast<uint16_t>(ap >> 16));
              }
            }
          }
          ptx::bar_sync(bar_g, 128);
          // 32 token rows x 64 columns: eight threads store one row's 128 bytes
          uint16_t* out = static_cast<uint16_t*>(p.out);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int idx = et + 128 * i;
            const int j = idx >> 3, k = idx & 7;
            const int col = col0 + 8 * k;
            if (j0 + j < t.n_tok && col < p.N) {
              const uint4 val = ptx::ld_shared_v4(ost + j * 128 + ((k ^ (j & 7)) << 4));
              *reinterpret_cast<uint4*>(out + static_cast<size_t>(t.r0 + j0 + j) * p.N + col) =
                  val;
            }
          }
          ptx::bar_sync(bar_g, 128);
        } else {
          // the routing weight: one f32 multiply, then the one bf16 rounding
          float wv[32];
          if (p.pair_weight) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint4 w4 = ptx::ld_shared_v4(ptx::smem_u32(w_t + j0) + 16 * k);
              wv[4 * k] = __uint_as_float(w4.x);
              wv[4 * k + 1] = __uint_as_float(w4.y);
              wv[4 * k + 2] = __uint_as_float(w4.z);
              wv[4 * k + 3] = __uint_as_float(w4.w);
            }
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int j = 2 * i;
            float a = __uint_as_float(v[j]), b = __uint_as_float(v[j + 1]);
            if (p.pair_weight) {
              a = __fmul_rn(a, wv[j]);
              b = __fmul_rn(b, wv[j + 1]);
            }
            const uint32_t pk = pack_bf16x2(a, b);
            ptx::st_shared_u16(slot[j & (kSw - 1)] + j * kRowB, static_cast<uint16_t>(pk & 0xFFFFu));
            ptx::st_shared_u16(slot[(j + 1) & (kSw - 1)] + (j + 1) * kRowB,
                               static_cast<uint16_t>(pk >> 16));
          }
          ptx::bar_sync(bar_g, 128);
          // 32 token rows x 128 columns: sixteen threads store one row's 256 bytes
          uint16_t* out = static_cast<uint16_t*>(p.out);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int idx = et + 128 * i;
            const int j = idx >> 4, k = idx & 15;
            const int col = col0 + 8 * k;
            if (j0 + j < t.n_tok && col < p.N) {
              const uint4 val = ptx::ld_shared_v4(ost + j * 256 + ((k ^ (j & 15)) << 4));
              *reinterpret_cast<uint4*>(out + static_cast<size_t>(dst_t[j0 + j]) * p.N + col) =
                  val;
            }
          }
          ptx::bar_sync(bar_g, 128);
        }
      }
      if (acc) ++uses1;
      else ++uses0;
      acc ^= 1;
    }
  }

  // ---- exit: if either CTA of the pair gave up, drain before freeing memory
  __syncthreads();
  ptx::cluster_sync();
  const bool gave_up =
      *abort_flag != 0 ||
      ld_shared_cluster_u32(ptx::mapa_shared(ptx::smem_u32(const_cast<int*>(abort_flag)),
                                             rank ^ 1u)) != 0;
  if (gave_up) {
    if (warp == 1 && lane == 0 && leader && mma_any) {
      ptx::mma_commit_pair(bar_drain, 1);
      spin_bounded(bar_drain, 0);
    }
    if (warp == 0 && lane == 0) {
      const uint64_t t0 = ptx::globaltimer_ns();
      while (ptx::globaltimer_ns() - t0 < kCopyGraceNs) {
      }
    }
  }
  __syncthreads();
  ptx::cluster_sync();  // the peer may still use this CTA's shared memory or TMEM until here
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc2(tmem_base, 2 * kTokBlock);
  }
  if (kStaged && threadIdx.x == 0) {
    // the last CTA to finish records this launch's flag value for the next
    // launch (its flags then mean "ready" to nobody) and resets the count
    __threadfence();
    const unsigned int prev = atomicAdd(p.stage_ctl + 1, 1u);
    if (prev + 1u == gridDim.x) {
      p.stage_ctl[1] = 0u;
      *reinterpret_cast<volatile unsigned int*>(p.stage_ctl) = *s_epoch;
      __threadfence();
    }
  }
}

}  // namespace

// The pair kernels' grid: clusters of two CTAs, as many as can be resident.
template <int kEpi, int kSrc>
int launch_pair_kernel(const char* op, const CUtensorMap (&tt)[4], const CUtensorMap& tw,
                       PairParams p, long long tiles, cudaStream_t stream) {
  auto kern = pair_gemm_kernel<kEpi, kSrc>;
  constexpr int kNT = pair_threads(kSrc);
  const int smem = PSmem::ALLOC;
  static std::atomic<int> configured_dev[64] = {};
  static std::atomic<int> max_pairs_dev[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  const bool cache = dev >= 0 && dev < 64;
  if (!cache || !configured_dev[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return set_error(MOE_ERR_CUDA, "%s: cannot reserve %d bytes of shared memory: %s", op, smem,
                       cudaGetErrorString(cudaGetLastError()));
    if (cache) configured_dev[dev].store(1, std::memory_order_release);
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // a pair must sit in one GPC, so fewer than SMs / 2 pairs may fit at once;
  // launching more would leave a second, mostly idle wave
  int max_pairs = cache ? max_pairs_dev[dev].load(std::memory_order_relaxed) : 0;
  if (max_pairs <= 0) {
    max_pairs = num_sms() / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * max_pairs), 1, 1);
    cfg.blockDim = dim3(kNT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters > 0)
      max_pairs = clusters < max_pairs ? clusters : max_pairs;
    else
      cudaGetLastError();
    if (cache) max_pairs_dev[dev].store(max_pairs, std::memory_order_relaxed);
  }
  long long pairs = tiles < max_pairs ? tiles : max_pairs;
  if (pairs < 1) pairs = 1;
  DeviceDiag diag = device_diag();
  p.status = diag.status;
  p.launches = diag.launches;
  p.wait_ns = pipeline_wait_ns();
  return launch_status(launch_kernel(kern, dim3(static_cast<unsigned>(2 * pairs), 1, 1),
                                     dim3(kNT, 1, 1), smem, stream, attr, 1, tt[0], tt[1],
                                     tt[2], tt[3], tw, p),
                       op);
}

// Upper bound on the pair tiles of a call: token blocks of 256 per group times
// the feature blocks.
static long long pair_tile_bound(int P, int G, int N, int fb_cols) {
  const long long blocks = (P + kTokBlock - 1) / kTokBlock + (G < P ? G : P);
  return blocks * ((N + fb_cols - 1) / fb_cols);
}

// the token rows [rows, cols] behind four maps with 16-, 32-, 64- and 128-row
// boxes (the 16-row box feeds a short tile's side slot)
static int make_token_maps(CUtensorMap (&tt)[4], const void* base, int rows, int cols,
                           const char* op, const char* what) {
  int rc;
  for (int i = 0; i < 4; ++i)
    if ((rc = make_tmap(&tt[i], base, rows, cols, (kTokBoxMin / 2) << i, op, what)) != MOE_OK)
      return rc;
  return MOE_OK;
}

int launch_pair_gateup(const char* op, const void* a_bf16, int a_rows,
                       const int32_t* a_row_gather, int gather_div, const void* w13_bf16,
                       const int32_t* group_offsets, int P, int H, int I, int G, void* act_bf16,
                       cudaStream_t stream) {
  CUtensorMap tt[4], tw;
  int rc;
  if ((rc = make_tmap(&tw, w13_bf16, static_cast<long long>(G) * 2 * I, H, 64, op, "w13")) !=
      MOE_OK)
    return rc;
  if (a_row_gather) {
    for (int i = 0; i < 4; ++i) tt[i] = tw;  // unused: the gatherer warps copy the token rows
  } else if ((rc = make_token_maps(tt, a_bf16, P, H, op, "a")) != MOE_OK) {
    return rc;
  }
  PairParams p{};
  p.group_offsets = group_offsets;
  p.P = P;
  p.Kdim = H;
  p.N = I;
  p.G = G;
  p.w_rows_per_group = 2 * I;
  p.half_off = I;
  p.out = act_bf16;
  p.a = static_cast<const uint16_t*>(a_bf16);
  p.a_rows = a_rows;
  p.row_gather = a_row_gather;
  p.gather_div = gather_div;
  p.kid = MOE_KID_GEMM_GATEUP;
  const long long tiles = pair_tile_bound(P, G, I, 128);
  if (a_row_gather) return launch_pair_kernel<PEPI_GATEUP, SRC_GATHER>(op, tt, tw, p, tiles, stream);
  return launch_pair_kernel<PEPI_GATEUP, SRC_TMA>(op, tt, tw, p, tiles, stream);
}

int launch_pair_gateup_staged(const char* op, const void* x_bf16, int T,
                              const int32_t* sorted_pair, int K, void* x_perm_bf16,
                              const void* w13_bf16, const int32_t* group_offsets, int P, int H,
                              int I, int G, void* act_bf16, int32_t* stage_flags,
                              unsigned int* stage_ctl, cudaStream_t stream) {
  CUtensorMap tt[4], tw;
  int rc;
  if ((rc = make_tmap(&tw, w13_bf16, static_cast<long long>(G) * 2 * I, H, 64, op, "w13")) !=
      MOE_OK)
    return rc;
  if ((rc = make_token_maps(tt, x_perm_bf16, P, H, op, "x_perm")) != MOE_OK) return rc;
  PairParams p{};
  p.group_offsets = group_offsets;
  p.P = P;
  p.Kdim = H;
  p.N = I;
  p.G = G;
  p.w_rows_per_group = 2 * I;
  p.half_off = I;
  p.out = act_bf16;
  p.a = static_cast<const uint16_t*>(x_bf16);
  p.a_rows = T;
  p.row_gather = sorted_pair;
  p.gather_div = K;
  p.stage_out = static_cast<uint16_t*>(x_perm_bf16);
  p.stage_flags = stage_flags;
  p.stage_ctl = stage_ctl;
  p.kid = MOE_KID_GEMM_GATEUP;
  return launch_pair_kernel<PEPI_GATEUP, SRC_STAGED>(op, tt, tw, p, pair_tile_bound(P, G, I, 128),
                                                      stream);
}

int launch_pair_down(const char* op, const void* act_bf16, const void* w2_bf16,
                     const int32_t* group_offsets, const float* pair_weight,
                     const int32_t* row_to_pair, int P, int I, int H, int G, void* out_bf16,
                     cudaStream_t stream) {
  CUtensorMap tt[4], tw;
  int rc;
  if ((rc = make_token_maps(tt, act_bf16, P, I, op, "act")) != MOE_OK) return rc;
  if ((rc = make_tmap(&tw, w2_bf16, static_cast<long long>(G) * H, I, 128, op, "w2")) != MOE_OK)
    return rc;
  PairParams p{};
  p.group_offsets = group_offsets;
  p.P = P;
  p.Kdim = I;
  p.N = H;
  p.G = G;
  p.w_rows_per_group = H;
  p.half_off = 0;
  p.out = out_bf16;
  p.pair_weight = pair_weight;
  p.row_to_pair = row_to_pair;
  p.kid = MOE_KID_GEMM_DOWN;
  return launch_pair_kernel<PEPI_DOWN, SRC_TMA>(op, tt, tw, p, pair_tile_bound(P, G, H, 256),
                                             stream);
}

}  // namespace gemm
}  // namespace moe
