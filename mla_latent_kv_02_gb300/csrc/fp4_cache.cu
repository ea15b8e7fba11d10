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
// * gather_nvfp4: one half-warp per token; in each of four steps lane l of
//   the half dequantises code word 16 v + l (8 elements) and the 16 lanes
//   write 256 contiguous bytes of bf16; lanes 0-7 copy the RoPE values.
//   Value = bf16(fp32(fp32(e2m1 * s_b) * s_t)).
// * gather_nvfp4_batch: many sequences into one packed output in one launch
//   (the same values; one half-warp per token).
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

// One token's row, dequantised by the 16 lanes (hl) of a half-warp into dst
// (72 uint4 = 576 bf16).  In step v lane hl takes code word 16 v + hl
// (elements 8 (16 v + hl) .. + 7, block (16 v + hl) / 2), so each store
// instruction writes 256 contiguous bytes; lanes 0-7 also copy the RoPE
// values.  Every load is issued before the first store.
__device__ __forceinline__ void gather_row_half(const uint8_t* __restrict__ row, uint4* __restrict__ dst, int hl,
                                                float tensor_scale) {
  uint32_t cw[4], sb[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    cw[v] = __ldg(reinterpret_cast<const uint32_t*>(row) + 16 * v + hl);
    sb[v] = __ldg(row + kScaleOff + ((16 * v + hl) >> 1));
  }
  uint4 rp = make_uint4(0u, 0u, 0u, 0u);
  if (hl < 8) rp = __ldg(reinterpret_cast<const uint4*>(row + kRopeOff) + hl);
#pragma unroll
  for (int v = 0; v < 4; ++v) dst[16 * v + hl] = dequant_word(cw[v], e4m3_to_f32(sb[v]), tensor_scale);
  if (hl < 8) dst[64 + hl] = rp;
}

__global__ void __launch_bounds__(kWarps * 32)
    gather_nvfp4_kernel(const uint8_t* __restrict__ rows, float tensor_scale, int64_t num_pages,
                        const int32_t* __restrict__ block_table, int32_t max_pages, int32_t b, int32_t n_tokens,
                        uint4* __restrict__ out, int32_t* err) {
  const int lane = threadIdx.x & 31, hl = lane & 15;
  const int64_t stride = (int64_t)gridDim.x * kWarps * 2;
  for (int64_t j0 = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * 2; j0 < n_tokens; j0 += stride) {
    const int64_t j = j0 + (lane >> 4);  // one token per half-warp
    if (j >= n_tokens) continue;
    const int32_t pid = __ldg(block_table + (int64_t)b * max_pages + j / 64);
    if (pid < 0 || (int64_t)pid >= num_pages) {
      if (hl == 0) atomicOr(err, (int32_t)MLA_DEVERR_PAGE_OOB);
      continue;
    }
    gather_row_half(rows + ((int64_t)pid * 64 + j % 64) * kRow, out + j * 72, hl, tensor_scale);
  }
}

// Batched gather: token g of the packed output belongs to the sequence i with
// off[i] <= g < off[i + 1] (found by bisection of the small offsets array)
// and sits at position g - off[i] of sequence seq_ids[i].  One half-warp per
// token (gather_row_half), two tokens per warp.
__global__ void __launch_bounds__(kWarps * 32)
    gather_nvfp4_batch_kernel(const uint8_t* __restrict__ rows, float tensor_scale, int64_t num_pages,
                              const int32_t* __restrict__ block_table, int32_t B, int32_t max_pages,
                              const int32_t* __restrict__ seq_ids, const int64_t* __restrict__ off, int32_t nb,
                              int64_t total, uint4* __restrict__ out, int32_t* err) {
  const int lane = threadIdx.x & 31, hl = lane & 15;
  const int64_t stride = (int64_t)gridDim.x * kWarps * 2;
  for (int64_t g0 = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * 2; g0 < total; g0 += stride) {
    const int64_t g = g0 + (lane >> 4);
    if (g >= total) continue;
    int lo = 0, hi = nb;  // off[lo] <= g < off[hi] when the offsets are consistent
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(off + mid) <= g) lo = mid;
      else hi = mid;
    }
    const int64_t o0 = __ldg(off + lo), o1 = __ldg(off + lo + 1);
    const int64_t j = g - o0;
    const int32_t sid = __ldg(seq_ids + lo);
    if (!(o0 <= g && g < o1) || sid < 0 || sid >= B || j / 64 >= max_pages) {
      if (hl == 0) atomicOr(err, (int32_t)MLA_DEVERR_BATCH);
      continue;
    }
    const int32_t pid = __ldg(block_table + (int64_t)sid * max_pages + j / 64);
    if (pid < 0 || (int64_t)pid >= num_pages) {
      if (hl == 0) atomicOr(err, (int32_t)MLA_DEVERR_PAGE_OOB);
      continue;
    }
    gather_row_half(rows + ((int64_t)pid * 64 + j % 64) * kRow, out + g * 72, hl, tensor_scale);
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
  f4::gather_nvfp4_kernel<<<f4::blocks_for(((int64_t)n_tokens + 1) / 2), f4::kWarps * 32, 0, stream>>>(
      rows, tensor_scale, num_pages, block_table, max_pages, b, n_tokens, reinterpret_cast<uint4*>(out), dev_err);
  return cudaGetLastError();
}

cudaError_t launch_gather_nvfp4_batch(const uint8_t* rows, float tensor_scale, int64_t num_pages,
                                      const int32_t* block_table, int32_t B, int32_t max_pages, const int32_t* seq_ids,
                                      const int64_t* out_offsets, int32_t nb, int64_t total_tokens, uint16_t* out,
                                      int32_t* dev_err, cudaStream_t stream) {
  if (total_tokens <= 0 || nb <= 0) return cudaSuccess;
  f4::gather_nvfp4_batch_kernel<<<f4::blocks_for((total_tokens + 1) / 2), f4::kWarps * 32, 0, stream>>>(
      rows, tensor_scale, num_pages, block_table, B, max_pages, seq_ids, out_offsets, nb, total_tokens,
      reinterpret_cast<uint4*>(out), dev_err);
  return cudaGetLastError();
}

}  // namespace mla
