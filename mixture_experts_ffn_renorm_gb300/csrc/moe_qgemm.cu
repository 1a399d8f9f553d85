// moe_qgemm.cu -- keep-quant expert GEMMs: grouped matmuls that read the
// expert weights as GGUF Q8_0 / Q4_K blocks, with the activations quantized to
// 8-bit blocks and every block's dot product an exact integer sum, plus the
// activation quantizer.  These are kMatmulBTQuant / kMatmulBTQuantGrouped of
// vllm.cpp PR #523 ("What changed"): a grouped matmul over the expert ids that
// keeps the quantized weights as stored.
//
// GB300 has no fast 8-bit integer tensor-core path, and these ops matter where
// the weights dominate the bytes (decode: a few rows per expert), so the dot
// products run on the CUDA cores with dp4a.  The kernel is a persistent grid
// over units of (a row block of one expert: up to 8 activation rows, or 2 for
// decode-class calls) x (32 pairs of weight rows).  The unit's activation codes
// sit in shared memory; each warp streams its weight rows in K chunks, four
// rows to a slot, from HBM into a ring of shared-memory slots with TMA bulk
// copies, and its lanes multiply the rows with all of the unit's activation
// rows, so each weight byte crosses HBM once per row block.
//
// Weight blocks (little-endian, as stored in GGUF files):
//   Q8_0: 32 weights in 34 bytes: fp16 d, int8 q[32];          w = d*q
//   Q4_K: 256 weights in 144 bytes: fp16 d, fp16 dmin, 12 bytes of packed
//         6-bit scales sc_j and mins m_j, 128 bytes of 4-bit codes; sub-block
//         j (32 weights) has w = d*sc_j*q - dmin*m_j.
// Activations: Q8_0 blocks of 32 (for Q8_0 weights, scale rounded to fp16) or
// Q8_K blocks of 256 (for Q4_K weights, f32 scale), codes in an int8 [R, K]
// plane and scales in an f32 [R, K/block] plane.
#include <cuda_fp16.h>

#include <atomic>

#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace {

using namespace moe;

constexpr int kQWarps = 8;
constexpr int kQThreads = 32 * kQWarps;
constexpr int kMaxMR = 8;  // activation rows per unit: 8, or 2 for decode-class calls
constexpr int kItemsPerUnit = 32;                   // pairs of weight rows per unit
constexpr int kItemsPerWarp = kItemsPerUnit / kQWarps;
// weights of a row staged at a time: 1024 for Q8_0 (1088 bytes), 2048 for Q4_K (1152 bytes)
__host__ __device__ constexpr int chunk_k(int fmt) { return fmt == MOE_QFMT_Q8_0 ? 1024 : 2048; }
constexpr int kMaxK = 16384;
constexpr int kMaxG = 1024;

enum { QE_PLAIN = 0, QE_GATEUP = 1, QE_DOWN = 2 };

template <int kFmt>
struct QFmt;
template <>
struct QFmt<MOE_QFMT_Q8_0> {
  static constexpr int kBlk = 32, kBytes = 34;
};
template <>
struct QFmt<MOE_QFMT_Q4_K> {
  static constexpr int kBlk = 256, kBytes = 144;
};

// Per-warp ring of weight slots.  A slot holds one K chunk of four weight
// rows -- two items of two rows, one item per half-warp -- brought in by TMA
// bulk copies that complete on the slot's mbarrier.  A warp's items are
// consecutive, so when a row is a single chunk the slot's rows are two runs
// of adjacent rows in HBM (gate/up: the two gate rows and the two up rows;
// down: four rows) and arrive in one or two large copies: small bulk copies
// cost the copy engine far more per byte than large ones.  The slot ends in
// 16 spare bytes because the Q8_0 code reads take nine words and the ninth
// of a row's last block ends 4 bytes past the row.  The ring gets a fixed
// byte budget and the number of slots follows from the slot size.
constexpr int kWarpRingBytes = 9344;
constexpr int kMaxSlots = 8;
constexpr int kSlotRows = 4;

__host__ __device__ constexpr int align16(int n) { return (n + 15) & ~15; }

__host__ __device__ inline int q_blk(int fmt) { return fmt == MOE_QFMT_Q8_0 ? 32 : 256; }
__host__ __device__ inline int q_bytes(int fmt) { return fmt == MOE_QFMT_Q8_0 ? 34 : 144; }
// bytes of one staged row chunk (a chunk is at most chunk_k(fmt) weights); a
// multiple of 16 whenever K is a multiple of 256
__host__ __device__ inline int chunk_row_bytes(int fmt, int K) {
  return ((K < chunk_k(fmt) ? K : chunk_k(fmt)) / q_blk(fmt)) * q_bytes(fmt);
}
__host__ __device__ inline int slot_bytes(int fmt, int K) {
  return kSlotRows * chunk_row_bytes(fmt, K) + 16;
}
__host__ __device__ inline int ring_slots(int fmt, int K) {
  const int n = kWarpRingBytes / slot_bytes(fmt, K);
  return n < 2 ? 2 : (n > kMaxSlots ? kMaxSlots : n);
}

// shared-memory carve-up of one CTA (host and device compute it alike)
struct QSmem {
  int off_src, off_bars, off_codes, off_scale, off_xsum, off_ring, warp_ring, total;
  __host__ __device__ QSmem(int fmt, int K, int G, int mr) {
    off_src = align16((G + 1) * 4);
    off_bars = off_src + align16(mr * 4);  // per warp kMaxSlots mbarriers, then an abort flag
    off_codes = off_bars + align16(kQWarps * kMaxSlots * 8 + 4);
    off_scale = off_codes + mr * K;
    off_xsum = off_scale + align16(mr * (K / q_blk(fmt)) * 4);
    off_ring = off_xsum + (fmt == MOE_QFMT_Q4_K ? align16(mr * (K / 32) * 4) : 0);
    warp_ring = ring_slots(fmt, K) * slot_bytes(fmt, K);
    total = off_ring + kQWarps * warp_ring;
  }
};

struct QParams {
  const int8_t* aq;             // activation codes [a_rows, K]
  const float* ad;              // activation scales [a_rows, K / act block]
  int a_rows;
  const int32_t* a_row_gather;  // row r reads activation row a_row_gather[r] / gather_div
  int gather_div;
  const uint8_t* w;             // [G, rows_per_group, K / blk * bytes]
  const int32_t* group_offsets;
  int P, K, N, G;               // N: output columns (I for gate/up)
  int n_items, n_cb;            // pairs of weight rows; column blocks of kItemsPerUnit pairs
  void* out;
  const float* pair_weight;
  const int32_t* row_to_pair;
  unsigned long long* launches;
  unsigned int* status;
  int kid;
};

__device__ __forceinline__ float half_bits_to_f32(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}

__device__ __forceinline__ int group_lo(const int32_t* off, int g, int P) {
  return min(max(__ldg(off + g), 0), P);
}

// TMA bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to this CTA's shared memory, completing on mbarrier `bar`
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

constexpr unsigned long long kQWaitLimitNs = 1000000000ull;

// Bounded wait for phase `parity` of `bar`.  A wait that runs past the limit
// raises MOE_STATUS_TIMEOUT and the CTA's abort flag, and returns false; so
// does any wait once the flag is up.
__device__ __forceinline__ bool q_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       unsigned int* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > kQWaitLimitNs) {
      if (status) atomicOr(status, static_cast<unsigned int>(MOE_STATUS_TIMEOUT));
      *abort_flag = 1;
      return false;
    }
  }
}

// The 6-bit scales and mins of Q4_K sub-blocks 2c and 2c+1 (c = 0..3): the
// two bytes 2(c&1), 2(c&1)+1 of each scale word give them at once.  Sub-blocks
// 0-3 keep scale and min in the low six bits of bytes j (word s0) and j+4
// (s1); sub-blocks 4-7 take the low four bits from the nibbles of byte j+4
// (s2) and the top two from the top bits of bytes j-4 (s0) and j (s1).
__device__ __forceinline__ void q4k_pair_scales(uint32_t s0, uint32_t s1, uint32_t s2, int c,
                                                int& sc_l, int& sc_h, int& m_l, int& m_h) {
  const uint32_t sh = static_cast<uint32_t>(c & 1) * 16u;
  const uint32_t w0 = s0 >> sh, w1 = s1 >> sh, w2 = s2 >> sh;
  if (c < 2) {
    sc_l = static_cast<int>(w0 & 63u);
    sc_h = static_cast<int>((w0 >> 8) & 63u);
    m_l = static_cast<int>(w1 & 63u);
    m_h = static_cast<int>((w1 >> 8) & 63u);
  } else {
    sc_l = static_cast<int>((w2 & 15u) | ((w0 >> 2) & 0x30u));
    sc_h = static_cast<int>(((w2 >> 8) & 15u) | ((w0 >> 10) & 0x30u));
    m_l = static_cast<int>(((w2 >> 4) & 15u) | ((w1 >> 2) & 0x30u));
    m_h = static_cast<int>(((w2 >> 12) & 15u) | ((w1 >> 10) & 0x30u));
  }
}

// dp4a with the first operand's bytes unsigned (0..255) and the second's signed
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// sum over 32 bytes of (high nibble of q) * a: the nibbles are used in place
// (q & 0xF0 = 16 * nibble), so the result is 16 times the sum, exactly
__device__ __forceinline__ int dp4a8_hi16(const uint32_t (&q)[8], int4 a0, int4 a1) {
  const uint32_t kHi = 0xF0F0F0F0u;
  int x = dp4a_us(q[0] & kHi, a0.x, 0), y = dp4a_us(q[4] & kHi, a1.x, 0);
  x = dp4a_us(q[1] & kHi, a0.y, x);
  y = dp4a_us(q[5] & kHi, a1.y, y);
  x = dp4a_us(q[2] & kHi, a0.z, x);
  y = dp4a_us(q[6] & kHi, a1.z, y);
  x = dp4a_us(q[3] & kHi, a0.w, x);
  y = dp4a_us(q[7] & kHi, a1.w, y);
  return x + y;
}

__device__ __forceinline__ int dp4a8(const int (&q)[8], int4 a0, int4 a1) {
  // two chains of four for a shorter dependency path
  int x = __dp4a(q[0], a0.x, 0), y = __dp4a(q[4], a1.x, 0);
  x = __dp4a(q[1], a0.y, x);
  y = __dp4a(q[5], a1.y, y);
  x = __dp4a(q[2], a0.z, x);
  y = __dp4a(q[6], a1.z, y);
  x = __dp4a(q[3], a0.w, x);
  y = __dp4a(q[7], a1.w, y);
  return x + y;
}

// acc[w][r] += this lane's share of  sum_k W[w][k] * A[r][k]  over one chunk
// of K (weights k0 .. k0 + kc) for an item's two weight rows (the second at
// `rs` bytes after the first).  The 16 lanes of a half-warp share the item:
// the chunk is cut into K tasks -- a Q8_0 block, or a 32-byte (64 weights:
// two whole sub-blocks) or, for short rows, a 16-byte (32 weights) run of a
// Q4_K super-block's codes -- dealt to the half's lanes (li = 0..15) in turn;
// a lane works each of its K tasks on both rows, so the rows share the
// activation loads and give independent dependency chains.
template <int kFmt, int kMR>
__device__ __forceinline__ void chunk_dot(const uint8_t* slot, int rs, bool two, int k0, int kc,
                                          const int8_t* s_codes, const float* s_scale,
                                          const int* s_xsum, int K, int m, int li,
                                          float (&acc)[2][kMR]) {
  if (kFmt == MOE_QFMT_Q8_0) {
    const int nt = kc / 32;  // blocks in this chunk
    const int nb_row = K / 32;
#pragma unroll
    for (int i = 0; i < chunk_k(kFmt) / 32 / 16; ++i) {
      const int b = li + 16 * i;
      if (b >= nt) break;
      const int kb = k0 + 32 * b;
      const int base = 34 * b + 2;
      const uint32_t sh = static_cast<uint32_t>(base & 3) * 8u;
      int qw[2][8];
      float dw[2];
#pragma unroll
      for (int wr = 0; wr < 2; ++wr) {
        // the 32 codes start 2 bytes into the block, 2-byte aligned: read the
        // nine covering words and shift by 0 or 16 bits (a missing second row
        // reads the ring's own bytes and is never accumulated)
        const uint8_t* row = slot + wr * rs;
        const uint32_t* wp = reinterpret_cast<const uint32_t*>(row + (base & ~3));
        uint32_t u[9];
#pragma unroll
        for (int j = 0; j < 9; ++j) u[j] = wp[j];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          qw[wr][j] = static_cast<int>(__funnelshift_r(u[j], u[j + 1], sh));
        dw[wr] = half_bits_to_f32(*reinterpret_cast<const uint16_t*>(row + 34 * b));
      }
#pragma unroll
      for (int r = 0; r < kMR; ++r) {
        if (r >= m) break;
        const int4* ap = reinterpret_cast<const int4*>(s_codes + r * K + kb);
        const int4 a0 = ap[0], a1 = ap[1];
        const float dx = s_scale[r * nb_row + kb / 32];
        const int i0 = dp4a8(qw[0], a0, a1);
        const int i1 = dp4a8(qw[1], a0, a1);
        acc[0][r] = fmaf(__fmul_rn(dw[0], dx), static_cast<float>(i0), acc[0][r]);
        if (two) acc[1][r] = fmaf(__fmul_rn(dw[1], dx), static_cast<float>(i1), acc[1][r]);
      }
    }
  } else {
    const int nsb = kc / 256;
    const int nsb_row = K / 256;
    const uint32_t kLo = 0x0F0F0F0Fu;
    if (nsb * 4 >= 16) {
      // wide K tasks: 32 bytes of codes, sub-blocks 2c (low nibbles) and 2c+1
      // (high nibbles) whole, so this lane adds both min terms
#pragma unroll
      for (int i = 0; i < chunk_k(kFmt) / 256 * 4 / 16; ++i) {
        const int t = li + 16 * i;
        if (t >= nsb * 4) break;
        const int sb = t >> 2, c = t & 3;
        const int sbg = k0 / 256 + sb;
        const int kb = k0 + 256 * sb + 64 * c;
        int ql[2][8], scl[2], sch[2], ml[2], mh[2];
        uint32_t qr[2][8];  // raw code words: the high nibbles are used in place
        float d[2], dmin[2];
#pragma unroll
        for (int wr = 0; wr < 2; ++wr) {
          const uint8_t* blk = slot + wr * rs + 144 * sb;
          const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
          const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
          const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
          d[wr] = half_bits_to_f32(hdr.x);
          dmin[wr] = half_bits_to_f32(hdr.x >> 16);
          q4k_pair_scales(hdr.y, hdr.z, hdr.w, c, scl[wr], sch[wr], ml[wr], mh[wr]);
          qr[wr][0] = q0.x;
          qr[wr][1] = q0.y;
          qr[wr][2] = q0.z;
          qr[wr][3] = q0.w;
          qr[wr][4] = q1.x;
          qr[wr][5] = q1.y;
          qr[wr][6] = q1.z;
          qr[wr][7] = q1.w;
#pragma unroll
          for (int j = 0; j < 8; ++j) ql[wr][j] = static_cast<int>(qr[wr][j] & kLo);
        }
#pragma unroll
        for (int r = 0; r < kMR; ++r) {
          if (r >= m) break;
          const int4* ap = reinterpret_cast<const int4*>(s_codes + r * K + kb);
          const int4 l0 = ap[0], l1 = ap[1], h0 = ap[2], h1 = ap[3];
          const int* xs = s_xsum + r * (K / 32) + sbg * 8 + 2 * c;
          const int x_l = xs[0], x_h = xs[1];
          const float dx = s_scale[r * nsb_row + sbg];
#pragma unroll
          for (int wr = 0; wr < 2; ++wr) {
            const int il = dp4a8(ql[wr], l0, l1);
            const int ih = dp4a8_hi16(qr[wr], h0, h1) >> 4;  // exact: a multiple of 16
            const int s1 = scl[wr] * il + sch[wr] * ih;
            const int s2 = ml[wr] * x_l + mh[wr] * x_h;
            const float tv = __fsub_rn(__fmul_rn(d[wr], static_cast<float>(s1)),
                                       __fmul_rn(dmin[wr], static_cast<float>(s2)));
            if (wr == 0) acc[0][r] = fmaf(dx, tv, acc[0][r]);
            else if (two) acc[1][r] = fmaf(dx, tv, acc[1][r]);
          }
        }
      }
    } else {
      // narrow K tasks for short rows: 16 bytes of codes -- weights 64c + 16h + i
      // of sub-block 2c (low nibbles) and 64c + 32 + 16h + i of 2c+1 (high);
      // the h = 0 lane adds the two sub-blocks' min terms
#pragma unroll
      for (int i = 0; i < 2; ++i) {  // at most 3 super-blocks: 24 tasks
        const int t = li + 16 * i;
        if (t >= nsb * 8) break;
        const int sb = t >> 3, part = t & 7, c = part >> 1, h = part & 1;
        const int sbg = k0 / 256 + sb;
        const int kb = k0 + 256 * sb + 64 * c + 16 * h;
        int ql[2][4], scl[2], sch[2], ml[2], mh[2];
        uint32_t qr[2][4];  // raw code words: the high nibbles are used in place
        float d[2], dmin[2];
#pragma unroll
        for (int wr = 0; wr < 2; ++wr) {
          const uint8_t* blk = slot + wr * rs + 144 * sb;
          const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
          const uint4 q = *reinterpret_cast<const uint4*>(blk + 16 + 16 * part);
          d[wr] = half_bits_to_f32(hdr.x);
          dmin[wr] = half_bits_to_f32(hdr.x >> 16);
          q4k_pair_scales(hdr.y, hdr.z, hdr.w, c, scl[wr], sch[wr], ml[wr], mh[wr]);
          qr[wr][0] = q.x;
          qr[wr][1] = q.y;
          qr[wr][2] = q.z;
          qr[wr][3] = q.w;
#pragma unroll
          for (int j = 0; j < 4; ++j) ql[wr][j] = static_cast<int>(qr[wr][j] & kLo);
        }
#pragma unroll
        for (int r = 0; r < kMR; ++r) {
          if (r >= m) break;
          const int4 al = *reinterpret_cast<const int4*>(s_codes + r * K + kb);
          const int4 ah = *reinterpret_cast<const int4*>(s_codes + r * K + kb + 32);
          const int* xs = s_xsum + r * (K / 32) + sbg * 8 + 2 * c;
          const int x_l = h == 0 ? xs[0] : 0, x_h = h == 0 ? xs[1] : 0;
          const float dx = s_scale[r * nsb_row + sbg];
#pragma unroll
          for (int wr = 0; wr < 2; ++wr) {
            const uint32_t kHi = 0xF0F0F0F0u;
            int il = __dp4a(ql[wr][0], al.x, 0), ih = dp4a_us(qr[wr][0] & kHi, ah.x, 0);
            il = __dp4a(ql[wr][1], al.y, il);
            ih = dp4a_us(qr[wr][1] & kHi, ah.y, ih);
            il = __dp4a(ql[wr][2], al.z, il);
            ih = dp4a_us(qr[wr][2] & kHi, ah.z, ih);
            il = __dp4a(ql[wr][3], al.w, il);
            ih = dp4a_us(qr[wr][3] & kHi, ah.w, ih);
            const int s1 = scl[wr] * il + sch[wr] * (ih >> 4);  // ih is 16 x the sum
            const int s2 = ml[wr] * x_l + mh[wr] * x_h;
            const float tv = __fsub_rn(__fmul_rn(d[wr], static_cast<float>(s1)),
                                       __fmul_rn(dmin[wr], static_cast<float>(s2)));
            if (wr == 0) acc[0][r] = fmaf(dx, tv, acc[0][r]);
            else if (two) acc[1][r] = fmaf(dx, tv, acc[1][r]);
          }
        }
      }
    }
  }
}

// sum over the 16 lanes of a half-warp (both halves at once)
__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
  for (int s = 8; s >= 1; s >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, s);
  return v;
}

// Each CTA takes a contiguous range of units -- (row block, column block) with
// the column block fastest -- so consecutive units mostly share their
// activation rows, which are then loaded once.  Per unit a warp has
// kItemsPerWarp items, worked as slots of two items (one per half-warp), each
// slot in K chunks; the slots go through the warp's ring: the copies of slot
// k + S - 1 start before slot k is computed, so S - 1 slots stay in flight.
// Two cursors walk the slot sequence, one for the copies and one for the
// compute; each finds its unit's group once per unit.
struct QCursor {
  int u, s, ch;       // unit, slot of this warp within the unit, K chunk
  int rb, cb, g;      // the unit's row block, column block and group
  const uint8_t* wg;  // the group's weights
};

template <int kFmt, int kEpi, int kMR>
__global__ void __launch_bounds__(kQThreads, kFmt == MOE_QFMT_Q8_0 ? 3 : 2) qgemm_kernel(QParams p) {
  using F = QFmt<kFmt>;
  constexpr int kCK = chunk_k(kFmt);
  constexpr int kSlotsPerUnit = kItemsPerWarp / 2;
  extern __shared__ __align__(16) uint8_t smem[];
  const int K = p.K, G = p.G, P = p.P;
  const QSmem L(kFmt, K, G, kMR);
  int* rb_start = reinterpret_cast<int*>(smem);
  int* s_src = reinterpret_cast<int*>(smem + L.off_src);
  int8_t* s_codes = reinterpret_cast<int8_t*>(smem + L.off_codes);
  float* s_scale = reinterpret_cast<float*>(smem + L.off_scale);
  int* s_xsum = reinterpret_cast<int*>(smem + L.off_xsum);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, li = lane & 15;
  uint8_t* ring = smem + L.off_ring + warp * L.warp_ring;
  const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  const uint32_t bars = static_cast<uint32_t>(__cvta_generic_to_shared(smem + L.off_bars)) +
                        static_cast<uint32_t>(warp * kMaxSlots * 8);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(smem + L.off_bars + kQWarps * kMaxSlots * 8);
  const int crb = chunk_row_bytes(kFmt, K);  // a staged row chunk
  const int sbytes = slot_bytes(kFmt, K);
  const int S = ring_slots(kFmt, K);

  if (lane == 0) {
    for (int i = 0; i < S; ++i) ptx::mbar_init(bars + 8 * i, 1);
    ptx::fence_mbar_init();
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  count_launch(p.launches, p.kid);
  grid_dep_wait();
  grid_dep_launch();

  // row blocks of every group (groups clamped into [0, P]), as a prefix sum
  const int32_t* off = p.group_offsets;
  if (warp == 0) {
    const int per = (G + 31) / 32;
    int sum = 0;
    for (int i = 0; i < per; ++i) {
      const int g = lane * per + i;
      if (g < G) {
        const int lo = off ? group_lo(off, g, P) : 0;
        const int hi = off ? max(group_lo(off, g + 1, P), lo) : P;
        sum += (hi - lo + kMR - 1) / kMR;
      }
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - sum;
    for (int i = 0; i < per; ++i) {
      const int g = lane * per + i;
      if (g < G) {
        rb_start[g] = run;
        const int lo = off ? group_lo(off, g, P) : 0;
        const int hi = off ? max(group_lo(off, g + 1, P), lo) : P;
        run += (hi - lo + kMR - 1) / kMR;
      }
    }
    if (lane == 31) rb_start[G] = incl;
  }
  __syncthreads();

  const int nb_row = K / F::kBlk;
  const long long row_bytes = static_cast<long long>(nb_row) * F::kBytes;
  const long long group_bytes = (kEpi == QE_GATEUP ? 2LL * p.N : p.N) * row_bytes;
  // the second row of an item: the up row N rows on (gate/up), else the next row
  const long long second = kEpi == QE_GATEUP ? p.N * row_bytes : row_bytes;
  const int total = rb_start[G] * p.n_cb;  // the host bounds this below 2^31
  const int u0 = static_cast<int>(static_cast<long long>(total) * blockIdx.x / gridDim.x);
  const int u1 = static_cast<int>(static_cast<long long>(total) * (blockIdx.x + 1) / gridDim.x);
  const int nchunk = (K + kCK - 1) / kCK;
  constexpr int kChunkBytes = (kCK / F::kBlk) * F::kBytes;

  auto set_unit = [&](QCursor& c, int u) {
    c.u = u;
    c.s = 0;
    c.ch = 0;
    c.rb = u / p.n_cb;
    c.cb = u - c.rb * p.n_cb;
    int lo_g = 0, hi_g = G;  // the last group whose first row block is <= rb
    while (hi_g - lo_g > 1) {
      const int mid = (lo_g + hi_g) >> 1;
      if (rb_start[mid] <= c.rb) lo_g = mid;
      else hi_g = mid;
    }
    c.g = lo_g;
    c.wg = p.w + c.g * group_bytes;
  };
  auto advance = [&](QCursor& c) {
    if (++c.ch == nchunk) {
      c.ch = 0;
      if (++c.s == kSlotsPerUnit) {
        if (c.u + 1 < u1) set_unit(c, c.u + 1);
        else c.u = u1;  // past the end
      }
    }
  };
  // item of half h in the cursor's slot (a warp's items are consecutive), its
  // first weight row, and whether it has a second row
  auto item_of = [&](const QCursor& c, int h, int& wr0) {
    const int item = c.cb * kItemsPerUnit + warp * kItemsPerWarp + 2 * c.s + h;
    wr0 = kEpi == QE_GATEUP ? item : 2 * item;
    return item;
  };
  auto has_second = [&](int wr0) { return kEpi == QE_GATEUP || wr0 + 1 < p.N; };
  // Lane 0 starts the copies of the cursor's slot into ring place `place`;
  // the place's barrier completes when they have landed (at once when empty).
  // Slot layout, rows of crb bytes: gate/up [gate A, gate B, up A, up B],
  // down [A row 0, A row 1, B row 0, B row 1].
  auto issue = [&](const QCursor& c, int place) {
    if (lane != 0) return;
    const uint32_t bar = bars + 8 * place;
    const uint32_t dst = ring_s + static_cast<uint32_t>(place * sbytes);
    if (c.u >= u1) {
      ptx::mbar_arrive_expect_tx(bar, 0);
      return;
    }
    const int k0 = c.ch * kCK;
    const uint32_t bytes =
        static_cast<uint32_t>(((K - k0 < kCK ? K - k0 : kCK) / F::kBlk) * F::kBytes);
    const uint8_t* base = c.wg + static_cast<long long>(c.ch) * kChunkBytes;
    int wr0;
    const int itemA = item_of(c, 0, wr0);
    const bool one_chunk = nchunk == 1;  // then adjacent rows are adjacent in HBM too
    if (kEpi == QE_GATEUP) {
      const int n_it = min(2, max(0, p.n_items - itemA));  // items of the slot that exist
      ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(2 * n_it) * bytes);
      if (n_it == 0) return;
      const uint8_t* gate = base + itemA * row_bytes;
      if (one_chunk) {
        bulk_copy_g2s(dst, gate, n_it * bytes, bar);
        bulk_copy_g2s(dst + 2 * crb, gate + second, n_it * bytes, bar);
      } else {
        for (int h = 0; h < n_it; ++h) {
          bulk_copy_g2s(dst + h * crb, gate + h * row_bytes, bytes, bar);
          bulk_copy_g2s(dst + (2 + h) * crb, gate + second + h * row_bytes, bytes, bar);
        }
      }
    } else {
      const int n_rows = min(kSlotRows, max(0, p.N - wr0));  // rows of the slot that exist
      ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n_rows) * bytes);
      if (n_rows == 0) return;
      const uint8_t* src = base + wr0 * row_bytes;
      if (one_chunk) {
        bulk_copy_g2s(dst, src, n_rows * bytes, bar);
      } else {
        for (int j = 0; j < n_rows; ++j) bulk_copy_g2s(dst + j * crb, src + j * row_bytes, bytes, bar);
      }
    }
  };

  QCursor ci, cc;  // copy cursor (runs S - 1 slots ahead), compute cursor
  if (u0 < u1) {
    set_unit(ci, u0);
    set_unit(cc, u0);
  } else {
    ci.u = cc.u = u1;
  }
  __syncwarp();  // the ring's barriers are initialised
  for (int k = 0; k < S - 1; ++k) {
    issue(ci, k);
    if (ci.u < u1) advance(ci);
  }
  int cur_rb = -1, m = 0, row0 = 0;
  float acc[2][kMR];
#pragma unroll
  for (int r = 0; r < kMR; ++r) acc[0][r] = acc[1][r] = 0.0f;

  int place = 0;       // ring place of the compute cursor's slot
  uint32_t round = 0;  // completed passes over the ring: the barrier phase parity
  bool alive = true;   // false after a wait gave up: the warp then only keeps step
#pragma unroll 1
  while (cc.u < u1) {
    if (cc.s == 0 && cc.ch == 0 && cc.rb != cur_rb) {
      // a new row block: every warp reaches this slot together (the slot
      // sequence is the same in all warps), finishes with the old rows, and
      // the CTA loads the new activation rows
      const int glo = off ? group_lo(off, cc.g, P) : 0;
      const int ghi = off ? max(group_lo(off, cc.g + 1, P), glo) : P;
      row0 = glo + (cc.rb - rb_start[cc.g]) * kMR;
      m = min(kMR, ghi - row0);
      cur_rb = cc.rb;
      __syncthreads();
      if (threadIdx.x < kMR) {
        int src = -1;
        if (static_cast<int>(threadIdx.x) < m) {
          const int row = row0 + threadIdx.x;
          src = p.a_row_gather ? __ldg(p.a_row_gather + row) / p.gather_div : row;
          if (src < 0 || src >= p.a_rows) src = -1;  // reads zeros
        }
        s_src[threadIdx.x] = src;
      }
      __syncthreads();
      const int n16 = K / 16;
      for (int i = threadIdx.x; i < m * n16; i += kQThreads) {
        const int r = i / n16, c = i - r * n16;
        const int src = s_src[r];
        int4 v = make_int4(0, 0, 0, 0);
        if (src >= 0)
          v = __ldg(reinterpret_cast<const int4*>(p.aq + static_cast<long long>(src) * K) + c);
        reinterpret_cast<int4*>(s_codes + r * K)[c] = v;
      }
      for (int i = threadIdx.x; i < m * nb_row; i += kQThreads) {
        const int r = i / nb_row, c = i - r * nb_row;
        const int src = s_src[r];
        s_scale[i] = src >= 0 ? __ldg(p.ad + static_cast<long long>(src) * nb_row + c) : 0.0f;
      }
      __syncthreads();
      if (kFmt == MOE_QFMT_Q4_K) {
        const int nsub = K / 32;  // code sums of every 32-code sub-block
        for (int i = threadIdx.x; i < m * nsub; i += kQThreads) {
          const int r = i / nsub, j = i - r * nsub;
          const int4* ap = reinterpret_cast<const int4*>(s_codes + r * K + 32 * j);
          const int4 a0 = ap[0], a1 = ap[1];
          int sum = __dp4a(a0.x, 0x01010101, 0);
          sum = __dp4a(a0.y, 0x01010101, sum);
          sum = __dp4a(a0.z, 0x01010101, sum);
          sum = __dp4a(a0.w, 0x01010101, sum);
          sum = __dp4a(a1.x, 0x01010101, sum);
          sum = __dp4a(a1.y, 0x01010101, sum);
          sum = __dp4a(a1.z, 0x01010101, sum);
          sum = __dp4a(a1.w, 0x01010101, sum);
          s_xsum[i] = sum;
        }
        __syncthreads();
      }
    }
    // refill the place freed by the previous slot, then wait for this one
    if (alive) issue(ci, place == 0 ? S - 1 : place - 1);
    if (ci.u < u1) advance(ci);
    if (alive) alive = q_wait(bars + 8 * place, round & 1u, abort_flag, p.status);
    int wr0;
    const int item = item_of(cc, half, wr0);
    const bool valid = alive && item < p.n_items;
    const bool two = has_second(wr0);
    if (valid) {
      const int k0 = cc.ch * kCK;
      const int kc = K - k0 < kCK ? K - k0 : kCK;
      // the half's rows: gate/up at h and 2 + h, down at 2h and 2h + 1
      const uint8_t* r0 = ring + place * sbytes + (kEpi == QE_GATEUP ? half : 2 * half) * crb;
      chunk_dot<kFmt, kMR>(r0, kEpi == QE_GATEUP ? 2 * crb : crb, two, k0, kc, s_codes, s_scale,
                           s_xsum, K, m, li, acc);
    }
    if (cc.ch == nchunk - 1) {
      // reduce every row's sums over each half-warp, then lane li = r of a
      // half finishes row r of its item: the rows' epilogues run side by side
      float y0 = 0.0f, y1 = 0.0f;
#pragma unroll
      for (int r = 0; r < kMR; ++r) {
        if (r >= m) break;
        const float s0 = half_sum(acc[0][r]);
        const float s1 = half_sum(acc[1][r]);
        acc[0][r] = acc[1][r] = 0.0f;
        if (li == r) {
          y0 = s0;
          y1 = s1;
        }
      }
      if (valid && li < m) {
        const int row = row0 + li;
        const int wr1 = kEpi == QE_GATEUP ? p.N + item : wr0 + 1;
        if (kEpi == QE_PLAIN) {
          float* out = static_cast<float*>(p.out) + static_cast<long long>(row) * p.N;
          out[wr0] = y0;
          if (two) out[wr1] = y1;
        } else if (kEpi == QE_DOWN) {
          const int dst = p.row_to_pair ? __ldg(p.row_to_pair + row) : row;
          if (dst >= 0 && dst < P) {
            const float wgt = p.pair_weight ? __ldg(p.pair_weight + dst) : 1.0f;
            uint16_t* out = static_cast<uint16_t*>(p.out) + static_cast<long long>(dst) * p.N;
            out[wr0] = f32_to_bf16_bits(p.pair_weight ? __fmul_rn(y0, wgt) : y0);
            if (two) out[wr1] = f32_to_bf16_bits(p.pair_weight ? __fmul_rn(y1, wgt) : y1);
          }
        } else {
          // narrowing before the activation: gate and up are rounded to bf16 first
          const float gz = bf16_bits_to_f32(f32_to_bf16_bits(y0));
          const float uz = bf16_bits_to_f32(f32_to_bf16_bits(y1));
          const float sg = gz / (1.0f + __expf(-gz));
          static_cast<uint16_t*>(p.out)[static_cast<long long>(row) * p.N + wr0] =
              f32_to_bf16_bits(sg * uz);
        }
      }
    }
    __syncwarp();  // every lane is done with this place before it is refilled
    advance(cc);
    if (++place == S) {
      place = 0;
      ++round;
    }
  }
  // copies still in flight (issued ahead, or left by a wait that gave up) land
  // before the CTA exits: one bounded wait per outstanding place
  if (lane == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (int j = 0; j < S - 1; ++j) {
      const int pl = (place + j) % S;
      const uint32_t par = (round + (place + j >= S ? 1u : 0u)) & 1u;
      while (!ptx::mbar_try_wait(bars + 8 * pl, par) &&
             ptx::globaltimer_ns() - t0 < kQWaitLimitNs) {
      }
    }
  }
  __syncwarp();
}

// One thread per 8 values; kBlk / 8 consecutive threads share a block.
template <int kBlk, bool kF16Scale>
__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t* x, long long n8, int8_t* q,
                                                        float* d, unsigned long long* launches) {
  constexpr int kTpb = kBlk / 8;
  count_launch(launches, MOE_KID_QUANT_ACT);
  grid_dep_wait();
  grid_dep_launch();
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool active = t < n8;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (active) v = __ldg(reinterpret_cast<const uint4*>(x) + t);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float f[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  float amax = 0.0f;  // a NaN never compares greater: it is skipped
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a = fabsf(f[i]);
    if (a > amax) amax = a;
  }
#pragma unroll
  for (int s = kTpb / 2; s >= 1; s >>= 1) {
    const float o = __shfl_xor_sync(0xFFFFFFFFu, amax, s);
    if (o > amax) amax = o;
  }
  const float dd = __fdiv_rn(amax, 127.0f);
  const float id = dd != 0.0f ? __fdiv_rn(1.0f, dd) : 0.0f;
  uint32_t packed[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float r = roundf(__fmul_rn(f[i], id));  // half-way cases away from zero
    if (r != r) r = 0.0f;
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    const uint32_t b = static_cast<uint32_t>(static_cast<int>(r)) & 0xFFu;
    packed[i >> 2] |= b << (8 * (i & 3));
  }
  if (active) {
    reinterpret_cast<uint2*>(q)[t] = make_uint2(packed[0], packed[1]);
    if ((threadIdx.x & (kTpb - 1)) == 0)
      d[t / kTpb] = kF16Scale ? __half2float(__float2half_rn(dd)) : dd;
  }
}

int q_block(int fmt) { return fmt == MOE_QFMT_Q8_0 ? 32 : (fmt == MOE_QFMT_Q4_K ? 256 : 0); }

template <int kFmt, int kEpi, int kMR>
int launch_q_mr(const char* op, QParams& p, cudaStream_t stream) {
  static std::atomic<int> configured_dev{-1};
  auto kern = qgemm_kernel<kFmt, kEpi, kMR>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return check_launch(op);
  if (configured_dev.load(std::memory_order_acquire) != dev) {
    // the attribute is raised to the largest carve-up any call can need
    const QSmem Lmax(kFmt, kMaxK, kMaxG, kMR);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lmax.total) !=
        cudaSuccess)
      return check_launch(op);
    configured_dev.store(dev, std::memory_order_release);
  }
  const QSmem Lg(kFmt, p.K, p.G, kMR);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kQThreads, Lg.total) !=
          cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  const long long units = (static_cast<long long>((p.P + kMR - 1) / kMR) + p.G) * p.n_cb;
  if (units > 0x7FFFFFFFLL) return set_error(MOE_ERR_ARG, "%s: too many rows for one call", op);
  const long long cap = static_cast<long long>(per_sm) * sm_count();
  const int grid = static_cast<int>(units < cap ? units : cap);
  if (grid <= 0) return MOE_OK;
  const DeviceDiag diag = device_diag();
  p.launches = diag.launches;
  p.status = diag.status;
  return launch_status(
      launch_kernel(kern, dim3(grid), dim3(kQThreads), static_cast<size_t>(Lg.total), stream,
                    nullptr, 0, p),
      op);
}

// Row blocks of 2 when the groups hold 2 rows or fewer on average (decode):
// every unit then costs about the same, so the CTAs' equal shares of units
// take equal time; row blocks of 8 otherwise, so that weights are re-read less.
template <int kFmt, int kEpi>
int launch_q(const char* op, QParams& p, cudaStream_t stream) {
  if (static_cast<long long>(p.P) <= 2LL * p.G) return launch_q_mr<kFmt, kEpi, 2>(op, p, stream);
  return launch_q_mr<kFmt, kEpi, kMaxMR>(op, p, stream);
}

int check_q(const char* op, int qfmt, int P, int K, int N, int G, const int32_t* group_offsets,
            const void* aq, const float* ad, const void* w, const void* out) {
  if (qfmt != MOE_QFMT_Q8_0 && qfmt != MOE_QFMT_Q4_K)
    return set_error(MOE_ERR_ARG, "%s: qfmt=%d is neither MOE_QFMT_Q8_0 nor MOE_QFMT_Q4_K", op,
                     qfmt);
  if (P < 0 || N <= 0 || K <= 0 || G < 1 || G > kMaxG)
    return set_error(MOE_ERR_ARG, "%s: bad sizes P=%d K=%d N=%d G=%d (1 <= G <= %d)", op, P, K, N,
                     G, kMaxG);
  if (K % 256 != 0 || K > kMaxK)
    return set_error(MOE_ERR_ALIGN, "%s: the contraction length %d must be a multiple of 256 "
                     "and at most %d", op, K, kMaxK);
  if (!group_offsets && G != 1)
    return set_error(MOE_ERR_ARG, "%s: group_offsets is NULL with G=%d", op, G);
  if (P > 0 && (!aq || !ad || !w || !out))
    return set_error(MOE_ERR_ARG, "%s: NULL operand", op);
  if (!aligned16(aq) || !aligned16(w) || (reinterpret_cast<uintptr_t>(ad) & 3u))
    return set_error(MOE_ERR_ALIGN, "%s: codes and weights must be 16-byte aligned, scales "
                     "4-byte aligned", op);
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_quantize_act_q8(const void* x_bf16, int R, int K, int qfmt, int8_t* codes, float* scales,
                        void* stream) {
  clear_error();
  const char* op = "moe_quantize_act_q8";
  const int blk = q_block(qfmt);
  if (!blk)
    return set_error(MOE_ERR_ARG, "%s: qfmt=%d is neither MOE_QFMT_Q8_0 nor MOE_QFMT_Q4_K", op,
                     qfmt);
  if (R < 0 || K <= 0) return set_error(MOE_ERR_ARG, "%s: bad sizes R=%d K=%d", op, R, K);
  if (K % blk != 0)
    return set_error(MOE_ERR_ALIGN, "%s: K=%d is not a multiple of the block (%d)", op, K, blk);
  if (R == 0) return MOE_OK;
  if (!x_bf16 || !codes || !scales) return set_error(MOE_ERR_ARG, "%s: NULL operand", op);
  if (!aligned16(x_bf16) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u))
    return set_error(MOE_ERR_ALIGN, "%s: x and codes must be 16-byte aligned, scales 4-byte", op);
  const long long n8 = static_cast<long long>(R) * K / 8;
  const long long blocks = (n8 + 255) / 256;
  if (blocks > 0x7FFFFFFFLL) return set_error(MOE_ERR_ARG, "%s: too many rows", op);
  const auto x = static_cast<const uint16_t*>(x_bf16);
  unsigned long long* launches = device_diag().launches;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (qfmt == MOE_QFMT_Q8_0)
    e = launch_kernel(quant_act_kernel<32, true>, dim3(static_cast<unsigned>(blocks)), dim3(256),
                      0, s, nullptr, 0, x, n8, codes, scales, launches);
  else
    e = launch_kernel(quant_act_kernel<256, false>, dim3(static_cast<unsigned>(blocks)), dim3(256),
                      0, s, nullptr, 0, x, n8, codes, scales, launches);
  return launch_status(e, op);
}

int moe_grouped_gemm_q(const int8_t* a_codes, const float* a_scales, int a_rows,
                       const int32_t* a_row_gather, int gather_div, const uint8_t* w, int qfmt,
                       const int32_t* group_offsets, int P, int K, int N, int G, float* out_f32,
                       void* stream) {
  clear_error();
  const char* op = "moe_grouped_gemm_q";
  int rc;
  if ((rc = check_q(op, qfmt, P, K, N, G, group_offsets, a_codes, a_scales, w, out_f32)) != MOE_OK)
    return rc;
  if (a_row_gather && (gather_div < 1 || a_rows < 0))
    return set_error(MOE_ERR_ARG, "%s: gather_div=%d, a_rows=%d", op, gather_div, a_rows);
  if (reinterpret_cast<uintptr_t>(out_f32) & 3u)
    return set_error(MOE_ERR_ALIGN, "%s: out must be 4-byte aligned", op);
  if (P == 0) return MOE_OK;
  QParams p{};
  p.aq = a_codes;
  p.ad = a_scales;
  p.a_rows = a_row_gather ? a_rows : P;
  p.a_row_gather = a_row_gather;
  p.gather_div = a_row_gather ? gather_div : 1;
  p.w = w;
  p.group_offsets = group_offsets;
  p.P = P;
  p.K = K;
  p.N = N;
  p.G = G;
  p.n_items = (N + 1) / 2;
  p.n_cb = (p.n_items + kItemsPerUnit - 1) / kItemsPerUnit;
  p.out = out_f32;
  p.kid = MOE_KID_GEMM_Q;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return qfmt == MOE_QFMT_Q8_0 ? launch_q<MOE_QFMT_Q8_0, QE_PLAIN>(op, p, s)
                               : launch_q<MOE_QFMT_Q4_K, QE_PLAIN>(op, p, s);
}

int moe_grouped_gemm_gateup_silu_q(const int8_t* a_codes, const float* a_scales, int a_rows,
                                   const int32_t* a_row_gather, int gather_div,
                                   const uint8_t* w13, int qfmt, const int32_t* group_offsets,
                                   int P, int H, int I, int G, void* act_bf16, void* stream) {
  clear_error();
  const char* op = "moe_grouped_gemm_gateup_silu_q";
  int rc;
  if ((rc = check_q(op, qfmt, P, H, I, G, group_offsets, a_codes, a_scales, w13, act_bf16)) !=
      MOE_OK)
    return rc;
  if (a_row_gather && (gather_div < 1 || a_rows < 0))
    return set_error(MOE_ERR_ARG, "%s: gather_div=%d, a_rows=%d", op, gather_div, a_rows);
  if (reinterpret_cast<uintptr_t>(act_bf16) & 1u)
    return set_error(MOE_ERR_ALIGN, "%s: act must be 2-byte aligned", op);
  if (P == 0) return MOE_OK;
  QParams p{};
  p.aq = a_codes;
  p.ad = a_scales;
  p.a_rows = a_row_gather ? a_rows : P;
  p.a_row_gather = a_row_gather;
  p.gather_div = a_row_gather ? gather_div : 1;
  p.w = w13;
  p.group_offsets = group_offsets;
  p.P = P;
  p.K = H;
  p.N = I;
  p.G = G;
  p.n_items = I;
  p.n_cb = (I + kItemsPerUnit - 1) / kItemsPerUnit;
  p.out = act_bf16;
  p.kid = MOE_KID_GEMM_Q_GATEUP;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return qfmt == MOE_QFMT_Q8_0 ? launch_q<MOE_QFMT_Q8_0, QE_GATEUP>(op, p, s)
                               : launch_q<MOE_QFMT_Q4_K, QE_GATEUP>(op, p, s);
}

int moe_grouped_gemm_down_q(const int8_t* a_codes, const float* a_scales, const uint8_t* w2,
                            int qfmt, const int32_t* group_offsets, const float* pair_weight,
                            const int32_t* row_to_pair, int P, int I, int H, int G,
                            void* out_bf16, void* stream) {
  clear_error();
  const char* op = "moe_grouped_gemm_down_q";
  int rc;
  if ((rc = check_q(op, qfmt, P, I, H, G, group_offsets, a_codes, a_scales, w2, out_bf16)) !=
      MOE_OK)
    return rc;
  if (reinterpret_cast<uintptr_t>(out_bf16) & 1u)
    return set_error(MOE_ERR_ALIGN, "%s: out must be 2-byte aligned", op);
  if (P == 0) return MOE_OK;
  QParams p{};
  p.aq = a_codes;
  p.ad = a_scales;
  p.a_rows = P;
  p.gather_div = 1;
  p.w = w2;
  p.group_offsets = group_offsets;
  p.P = P;
  p.K = I;
  p.N = H;
  p.G = G;
  p.n_items = (H + 1) / 2;
  p.n_cb = (p.n_items + kItemsPerUnit - 1) / kItemsPerUnit;
  p.out = out_bf16;
  p.pair_weight = pair_weight;
  p.row_to_pair = row_to_pair;
  p.kid = MOE_KID_GEMM_Q_DOWN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return qfmt == MOE_QFMT_Q8_0 ? launch_q<MOE_QFMT_Q8_0, QE_DOWN>(op, p, s)
                               : launch_q<MOE_QFMT_Q4_K, QE_DOWN>(op, p, s);
}

}  // extern "C"
