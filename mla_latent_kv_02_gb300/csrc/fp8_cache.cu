// FP8 (E4M3) latent cache: the quantising append and the dequantising gather.
//
// [P3] bjbfmj.com/news/60700: the byte formula L x (d_c + d_r) x b counts
// only the elements; quantisation scale factors are stored beside them.
// [P1] "撕开 DeepSeek MLA 源码…", opening section and §5: a quantised gather
// of the latent cache with 16-byte vector loads from 16-byte aligned bases.
//
// Layout: rows uint8 [num_pages][64][640] (512 E4M3 codes, then the 64 bf16
// RoPE values), scales fp32 [num_pages][64] (2^k per token).
//
// * kv_append_fp8: one warp per token.  Lane l holds latent values
//   [8l, 8l+8) and [256+8l, 256+8l+8); a warp max-reduction of |c| gives the
//   row's amax, the scale exponent follows from amax's exponent and mantissa
//   bits, and the scaled values (exact) are rounded to E4M3 by the hardware
//   conversion.  The RoPE key is copied bit for bit.
// * gather_paged_fp8: one warp per token; lane l loads 16 codes as one
//   16-byte vector and writes 32 bytes of bf16.
#include <cuda_runtime.h>

#include <cstdint>

#include "fp8.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace f8 {

using namespace mla::dev;

constexpr int kWarps = 8;

__device__ __forceinline__ uint32_t abs_max_bf16x2(uint32_t m, uint32_t v) {
  const uint32_t a = v & 0x7FFF7FFFu;
  return max(m, max(a & 0xFFFFu, a >> 16));
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Eight bf16 values (a uint4) times 2^n, rounded to eight E4M3 codes (a uint2).
__device__ __forceinline__ uint2 quant8(uint4 v, int n) {
  uint2 r;
  r.x = f32x2_to_e4m3x2(scale_pow2(bf16_lo(v.x), n), scale_pow2(bf16_hi(v.x), n)) |
        (f32x2_to_e4m3x2(scale_pow2(bf16_lo(v.y), n), scale_pow2(bf16_hi(v.y), n)) << 16);
  r.y = f32x2_to_e4m3x2(scale_pow2(bf16_lo(v.z), n), scale_pow2(bf16_hi(v.z), n)) |
        (f32x2_to_e4m3x2(scale_pow2(bf16_lo(v.w), n), scale_pow2(bf16_hi(v.w), n)) << 16);
  return r;
}

__global__ void __launch_bounds__(kWarps * 32)
    kv_append_fp8_kernel(const uint4* __restrict__ c_new, const uint4* __restrict__ k_new,
                         const int64_t* __restrict__ slots, int32_t n, uint8_t* __restrict__ rows,
                         float* __restrict__ scales, int64_t num_slots, int32_t* err) {
  const int lane = threadIdx.x & 31;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < n; t += (int64_t)gridDim.x * kWarps) {
    const int64_t slot = __ldg(slots + t);
    if (slot < 0 || slot >= num_slots) {
      if (lane == 0) atomicOr(err, (int32_t)MLA_DEVERR_SLOT_OOB);
      continue;
    }
    const uint4 a = __ldg(c_new + t * 64 + lane);
    const uint4 b = __ldg(c_new + t * 64 + 32 + lane);
    uint32_t m = 0;
    m = abs_max_bf16x2(m, a.x);
    m = abs_max_bf16x2(m, a.y);
    m = abs_max_bf16x2(m, a.z);
    m = abs_max_bf16x2(m, a.w);
    m = abs_max_bf16x2(m, b.x);
    m = abs_max_bf16x2(m, b.y);
    m = abs_max_bf16x2(m, b.z);
    m = abs_max_bf16x2(m, b.w);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    const int k = fp8_scale_exponent(__uint_as_float(m << 16));
    uint8_t* row = rows + slot * kFp8RowBytes;
    *reinterpret_cast<uint2*>(row + 8 * lane) = quant8(a, -k);
    *reinterpret_cast<uint2*>(row + 256 + 8 * lane) = quant8(b, -k);
    if (lane < 8) reinterpret_cast<uint4*>(row + kFp8Latent)[lane] = __ldg(k_new + t * 8 + lane);
    if (lane == 0) scales[slot] = k >= -126 ? exp2_int(k) : exp2_int(k + 64) * 0x1p-64f;
  }
}

__global__ void __launch_bounds__(kWarps * 32)
    gather_fp8_kernel(const uint8_t* __restrict__ rows, const float* __restrict__ scales, int64_t num_pages,
                      const int32_t* __restrict__ block_table, int32_t max_pages, int32_t b, int32_t n_tokens,
                      uint4* __restrict__ out, int32_t* err) {
  const int lane = threadIdx.x & 31;
  for (int64_t j = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); j < n_tokens; j += (int64_t)gridDim.x * kWarps) {
    const int32_t pid = __ldg(block_table + (int64_t)b * max_pages + j / 64);
    if (pid < 0 || (int64_t)pid >= num_pages) {
      if (lane == 0) atomicOr(err, (int32_t)MLA_DEVERR_PAGE_OOB);
      continue;
    }
    const int64_t slot = (int64_t)pid * 64 + j % 64;
    const uint8_t* row = rows + slot * kFp8RowBytes;
    const Fp8Scale sc = fp8_row_scale(__ldg(scales + slot));
    const uint4 c = __ldg(reinterpret_cast<const uint4*>(row) + lane);   // codes [16 lane, 16 lane + 16)
    uint4* dst = out + j * 72;
    dst[2 * lane] = dequant8(make_uint2(c.x, c.y), sc);
    dst[2 * lane + 1] = dequant8(make_uint2(c.z, c.w), sc);
    if (lane < 8) dst[64 + lane] = __ldg(reinterpret_cast<const uint4*>(row + kFp8Latent) + lane);
  }
}

inline int blocks_for(int64_t items) {
  int64_t b = (items + kWarps - 1) / kWarps;
  if (b > 152 * 16) b = 152 * 16;
  return b < 1 ? 1 : (int)b;
}

}  // namespace f8

cudaError_t launch_kv_append_fp8(const uint16_t* c_kv_new, const uint16_t* k_r_new, const int64_t* slots, int32_t n,
                                 uint8_t* rows, float* scales, int64_t num_slots, int32_t* dev_err,
                                 cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  f8::kv_append_fp8_kernel<<<f8::blocks_for(n), f8::kWarps * 32, 0, stream>>>(
      reinterpret_cast<const uint4*>(c_kv_new), reinterpret_cast<const uint4*>(k_r_new), slots, n, rows, scales,
      num_slots, dev_err);
  return cudaGetLastError();
}

cudaError_t launch_gather_fp8(const uint8_t* rows, const float* scales, int64_t num_pages,
                              const int32_t* block_table, int32_t max_pages, int32_t b, int32_t n_tokens,
                              uint16_t* out, int32_t* dev_err, cudaStream_t stream) {
  if (n_tokens <= 0) return cudaSuccess;
  f8::gather_fp8_kernel<<<f8::blocks_for(n_tokens), f8::kWarps * 32, 0, stream>>>(
      rows, scales, num_pages, block_table, max_pages, b, n_tokens, reinterpret_cast<uint4*>(out), dev_err);
  return cudaGetLastError();
}

}  // namespace mla
