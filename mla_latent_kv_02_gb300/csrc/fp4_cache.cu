// NVFP4 latent cache: the quantising append and the dequantising gather.
//
// [P1] "撕开 DeepSeek MLA 源码…", opening section and §5: the latent cache is
// gathered in NVFP4 with 16-byte (uint4) vector loads, which fault when the
// page-table base is not 16-byte aligned or a byte offset (element offset
// / 2) is not a multiple of 8 — here every row is 416 = 26 x 16 bytes and the
// host rejects unaligned bases before any launch.  NVFP4 (NVIDIA's format):
// E2M1 elements, one E4M3 scale per 16 elements, one fp32 scale per tensor.
//
// Row (416 bytes): 256 bytes of codes (element 2i in the low nibble), 32
// block-scale bytes, 128 bytes of bf16 RoPE values.
//
// * kv_append_nvfp4: one warp per token, lane l owns block l (16 values): its
//   amax, s_b = E4M3(amax / (6 s_t)) and the 16 codes E2M1(x / (s_b s_t)),
//   each division and product one correctly rounded fp32 operation.
// * gather_nvfp4: one warp per token; lanes 0-15 load 32 codes each as one
//   16-byte vector and write 64 bytes of bf16, lanes 16-23 copy the RoPE
//   values.  Value = bf16(fp32(fp32(e2m1 * s_b) * s_t)).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fp8.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace f4 {

using namespace mla::dev;

constexpr int kWarps = 8;
constexpr int kRow = 416, kScaleOff = 256, kRopeOff = 288;

// Two fp32 values to an E2M1 pair (nearest even, saturating at 6); lo in the low nibble.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}
// One byte of two E2M1 codes (low nibble first) to an f16 pair, exactly.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t h;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
      : "=r"(h)
      : "r"(byte));
  return h;
}
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  const uint32_t h = e4m3x2_to_f16x2(code & 0xFFu);
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__global__ void __launch_bounds__(kWarps * 32)
    kv_append_nvfp4_kernel(const uint4* __restrict__ c_new, const uint4* __restrict__ k_new,
                           const int64_t* __restrict__ slots, int32_t n, float tensor_scale,
                           uint8_t* __restrict__ rows, int64_t num_slots, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const float six_st = __fmul_rn(6.f, tensor_scale);
  for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < n; t += (int64_t)gridDim.x * kWarps) {
    const int64_t slot = __ldg(slots + t);
    if (slot < 0 || slot >= num_slots) {
      if (lane == 0) atomicOr(err, (int32_t)MLA_DEVERR_SLOT_OOB);
      continue;
    }
    const uint4 a = __ldg(c_new + t * 64 + 2 * lane);
    const uint4 b = __ldg(c_new + t * 64 + 2 * lane + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t v = w[i] & 0x7FFF7FFFu;
      m = max(m, max(v & 0xFFFFu, v >> 16));
    }
    const float amax = __uint_as_float(m << 16);
    const uint32_t sb_code = f32x2_to_e4m3x2(__fdiv_rn(amax, six_st), 0.f) & 0xFFu;
    const float denom = __fmul_rn(e4m3_to_f32(sb_code), tensor_scale);
    uint32_t lo = 0, hi = 0;
    if (denom != 0.f) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        lo |= f32x2_to_e2m1x2(__fdiv_rn(bf_lo(w[i]), denom), __fdiv_rn(bf_hi(w[i]), denom)) << (8 * i);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        hi |= f32x2_to_e2m1x2(__fdiv_rn(bf_lo(w[4 + i]), denom), __fdiv_rn(bf_hi(w[4 + i]), denom)) << (8 * i);
    }
    uint8_t* row = rows + slot * kRow;
    *reinterpret_cast<uint2*>(row + 8 * lane) = make_uint2(lo, hi);
    row[kScaleOff + lane] = (uint8_t)sb_code;
    if (lane < 8) reinterpret_cast<uint4*>(row + kRopeOff)[lane] = __ldg(k_new + t * 8 + lane);
  }
}

// 8 codes (one 32-bit word) of one block to 8 bf16 (a uint4).
__device__ __forceinline__ uint4 dequant_word(uint32_t w, float sb, float st) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t h = e2m1x2_to_f16x2(w >> (8 * i));
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h));
    o[i] = pack_bf16x2(__fmul_rn(__fmul_rn(v.x, sb), st), __fmul_rn(__fmul_rn(v.y, sb), st));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(kWarps * 32)
    gather_nvfp4_kernel(const uint8_t* __restrict__ rows, float tensor_scale, int64_t num_pages,
                        const int32_t* __restrict__ block_table, int32_t max_pages, int32_t b, int32_t n_tokens,
                        uint4* __restrict__ out, int32_t* err) {
  const int lane = threadIdx.x & 31;
  for (int64_t j = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); j < n_tokens; j += (int64_t)gridDim.x * kWarps) {
    const int32_t pid = __ldg(block_table + (int64_t)b * max_pages + j / 64);
    if (pid < 0 || (int64_t)pid >= num_pages) {
      if (lane == 0) atomicOr(err, (int32_t)MLA_DEVERR_PAGE_OOB);
      continue;
    }
    const uint8_t* row = rows + ((int64_t)pid * 64 + j % 64) * kRow;
    uint4* dst = out + j * 72;
    if (lane < 16) {
      const uint4 c = __ldg(reinterpret_cast<const uint4*>(row) + lane);   // codes of blocks 2l, 2l+1
      const uint32_t s2 = __ldg(reinterpret_cast<const uint16_t*>(row + kScaleOff) + lane);
      const float s0 = e4m3_to_f32(s2 & 0xFFu), s1 = e4m3_to_f32(s2 >> 8);
      dst[4 * lane] = dequant_word(c.x, s0, tensor_scale);
      dst[4 * lane + 1] = dequant_word(c.y, s0, tensor_scale);
      dst[4 * lane + 2] = dequant_word(c.z, s1, tensor_scale);
      dst[4 * lane + 3] = dequant_word(c.w, s1, tensor_scale);
    } else if (lane < 24) {
      dst[64 + (lane - 16)] = __ldg(reinterpret_cast<const uint4*>(row + kRopeOff) + (lane - 16));
    }
  }
}

inline int blocks_for(int64_t items) {
  int64_t b = (items + kWarps - 1) / kWarps;
  if (b > 152 * 16) b = 152 * 16;
  return b < 1 ? 1 : (int)b;
}

}  // namespace f4

cudaError_t launch_kv_append_nvfp4(const uint16_t* c_kv_new, const uint16_t* k_r_new, const int64_t* slots,
                                   int32_t n, float tensor_scale, uint8_t* rows, int64_t num_slots,
                                   int32_t* dev_err, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  f4::kv_append_nvfp4_kernel<<<f4::blocks_for(n), f4::kWarps * 32, 0, stream>>>(
      reinterpret_cast<const uint4*>(c_kv_new), reinterpret_cast<const uint4*>(k_r_new), slots, n, tensor_scale,
      rows, num_slots, dev_err);
  return cudaGetLastError();
}

cudaError_t launch_gather_nvfp4(const uint8_t* rows, float tensor_scale, int64_t num_pages,
                                const int32_t* block_table, int32_t max_pages, int32_t b, int32_t n_tokens,
                                uint16_t* out, int32_t* dev_err, cudaStream_t stream) {
  if (n_tokens <= 0) return cudaSuccess;
  f4::gather_nvfp4_kernel<<<f4::blocks_for(n_tokens), f4::kWarps * 32, 0, stream>>>(
      rows, tensor_scale, num_pages, block_table, max_pages, b, n_tokens, reinterpret_cast<uint4*>(out), dev_err);
  return cudaGetLastError();
}

}  // namespace mla
