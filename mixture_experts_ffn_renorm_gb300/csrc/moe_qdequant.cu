// moe_qdequant.cu -- keep-quant expert weights (GGUF Q8_0 / Q4_K blocks)
// expanded to bf16, so that batches with many rows per expert run on the bf16
// tensor-core GEMMs instead of the CUDA-core keep-quant kernels (GB300's HBM
// holds both copies of a layer's experts comfortably).  Every value is formed
// in binary32 and rounded to bf16 once:
//   Q8_0: bf16(d * q)                          (the product is exact)
//   Q4_K: bf16((d * sc_j) * q - dmin * m_j)    (exact products, one rounded
//                                               subtraction)
// One thread expands one 32-weight sub-block (Q4_K) or block (Q8_0) into
// 64 bytes of bf16; the grid covers every row's blocks.
#include <cuda_fp16.h>

#include "moe_common.cuh"

namespace {

using namespace moe;

__device__ __forceinline__ float fp16_bits(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return static_cast<uint32_t>(f32_to_bf16_bits(a)) |
         (static_cast<uint32_t>(f32_to_bf16_bits(b)) << 16);
}

// Q8_0: thread t expands block t (34 bytes at 2-byte alignment, read as 17 halves)
__global__ void __launch_bounds__(256) dequant_q8_0_kernel(const uint8_t* w, long long nblk,
                                                           uint16_t* out,
                                                           unsigned long long* launches) {
  count_launch(launches, MOE_KID_DEQUANT_Q);
  grid_dep_wait();
  grid_dep_launch();
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= nblk) return;
  const uint16_t* b = reinterpret_cast<const uint16_t*>(w + 34 * t);
  const float d = fp16_bits(__ldg(b));
  uint32_t o[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t two = __ldg(b + 1 + i);  // codes 2i (low byte) and 2i + 1
    const float q0 = static_cast<float>(static_cast<int8_t>(two & 0xFFu));
    const float q1 = static_cast<float>(static_cast<int8_t>(two >> 8));
    o[i] = pack2(__fmul_rn(d, q0), __fmul_rn(d, q1));
  }
  uint4* dst = reinterpret_cast<uint4*>(out + 32 * t);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

// Q4_K: thread t expands sub-block j = t % 8 of super-block t / 8.  Its codes
// are the low (j even) or high (j odd) nibbles of the 32 bytes 32 * (j / 2) ..
// of the super-block's codes; its 6-bit scale and min come from the 12 packed
// bytes (sub-blocks 0-3 in the low six bits of bytes j and j+4; sub-blocks 4-7
// low four bits from the nibbles of byte j+4, top two from bytes j-4 and j).
__global__ void __launch_bounds__(256) dequant_q4_k_kernel(const uint8_t* w, long long nsub,
                                                           uint16_t* out,
                                                           unsigned long long* launches) {
  count_launch(launches, MOE_KID_DEQUANT_Q);
  grid_dep_wait();
  grid_dep_launch();
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= nsub) return;
  const long long sb = t >> 3;
  const int j = static_cast<int>(t & 7);
  const uint8_t* blk = w + 144 * sb;
  const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(blk));
  const float d = fp16_bits(hdr.x), dmin = fp16_bits(hdr.x >> 16);
  const uint32_t sw[3] = {hdr.y, hdr.z, hdr.w};
  auto byte = [&](int i) { return static_cast<int>((sw[i >> 2] >> (8 * (i & 3))) & 0xFFu); };
  int sc, m;
  if (j < 4) {
    sc = byte(j) & 63;
    m = byte(j + 4) & 63;
  } else {
    sc = (byte(j + 4) & 15) | ((byte(j - 4) >> 6) << 4);
    m = (byte(j + 4) >> 4) | ((byte(j) >> 6) << 4);
  }
  const float dsc = __fmul_rn(d, static_cast<float>(sc));
  const float mn = __fmul_rn(dmin, static_cast<float>(m));
  const uint4* qp = reinterpret_cast<const uint4*>(blk + 16 + 32 * (j >> 1));
  const uint4 q0 = __ldg(qp), q1 = __ldg(qp + 1);
  const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  const int shift = (j & 1) * 4;
  uint32_t o[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t word = qw[i >> 1] >> (16 * (i & 1));  // codes 2i, 2i + 1 in its low bytes
    const float c0 = static_cast<float>((word >> shift) & 15u);
    const float c1 = static_cast<float>((word >> (8 + shift)) & 15u);
    o[i] = pack2(__fsub_rn(__fmul_rn(dsc, c0), mn), __fsub_rn(__fmul_rn(dsc, c1), mn));
  }
  uint4* dst = reinterpret_cast<uint4*>(out + 32 * t);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

}  // namespace

extern "C" int moe_dequantize_q_bf16(const uint8_t* w, int qfmt, long long rows, int K,
                                     void* out_bf16, void* stream) {
  clear_error();
  const char* op = "moe_dequantize_q_bf16";
  if (qfmt != MOE_QFMT_Q8_0 && qfmt != MOE_QFMT_Q4_K)
    return set_error(MOE_ERR_ARG, "%s: qfmt=%d is neither MOE_QFMT_Q8_0 nor MOE_QFMT_Q4_K", op,
                     qfmt);
  const int blk = qfmt == MOE_QFMT_Q8_0 ? 32 : 256;
  if (rows < 0 || K <= 0) return set_error(MOE_ERR_ARG, "%s: bad sizes rows=%lld K=%d", op, rows, K);
  if (K % blk != 0)
    return set_error(MOE_ERR_ALIGN, "%s: K=%d is not a multiple of the block (%d)", op, K, blk);
  if (rows == 0) return MOE_OK;
  if (!w || !out_bf16) return set_error(MOE_ERR_ARG, "%s: NULL operand", op);
  if (!aligned16(out_bf16) || (qfmt == MOE_QFMT_Q4_K ? !aligned16(w)
                                                      : (reinterpret_cast<uintptr_t>(w) & 1u)))
    return set_error(MOE_ERR_ALIGN, "%s: out must be 16-byte aligned, Q4_K blocks 16-byte and "
                     "Q8_0 blocks 2-byte aligned", op);
  const long long units = rows * (K / 32);  // threads: one per 32 weights
  const long long blocks = (units + 255) / 256;
  if (blocks > 0x7FFFFFFFLL) return set_error(MOE_ERR_ARG, "%s: too many rows", op);
  unsigned long long* launches = device_diag().launches;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto out = static_cast<uint16_t*>(out_bf16);
  const cudaError_t e =
      qfmt == MOE_QFMT_Q8_0
          ? launch_kernel(dequant_q8_0_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                          s, nullptr, 0, w, units, out, launches)
          : launch_kernel(dequant_q4_k_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                          s, nullptr, 0, w, units, out, launches);
  return launch_status(e, op);
}
