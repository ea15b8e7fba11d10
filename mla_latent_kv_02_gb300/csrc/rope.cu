// Decoupled RoPE in fp32, fused into the cache append, and for the query
// rows.  [P1] "撕开 DeepSeek MLA 源码…" §1: a 64-d shared RoPE key carries
// the position apart from the 512-d latent; §3: the plugin settings fix the
// RoPE compute dtype to fp32; §4: a failed equivalence check traced to RoPE
// computed in fp16 (phase error) is fixed by generating the RoPE table in
// fp32 and multiply-adding in fp32.  Rotation (the pages print none; the
// standard rotary embedding): consecutive pairs (x[2i], x[2i+1]) turned by
// p * base^(-2i/64).
//
// * rope_table: entry (p, i) = (cos, sin) of the angle, computed in double
//   and rounded once to fp32.
// * kv_append_rope: one warp per new token; the latent row is copied bit for
//   bit, lane i rotates pair i of k_pe in fp32 (fused multiply-add) and
//   rounds to bf16, so a row is one coalesced 1152-byte write.
// * rope_q: eight threads per (token, head) row of q_pe, four pairs each.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace rope {

constexpr int kPairs = 32;   // 64 RoPE dims
constexpr int kLatVec = 64;  // 512 bf16 = 64 x 16 B
constexpr int kRowVec = 72;  // 576 bf16 per cached token
constexpr int kWarps = 8;

__global__ void __launch_bounds__(256) rope_table_kernel(float2* __restrict__ table, int32_t max_pos, double base) {
  const int64_t n = (int64_t)max_pos * kPairs;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += (int64_t)gridDim.x * blockDim.x) {
    const int32_t p = (int32_t)(k / kPairs), i = (int32_t)(k % kPairs);
    const double a = (double)p * pow(base, -2.0 * (double)i / 64.0);
    table[k] = make_float2((float)cos(a), (float)sin(a));
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Pair (x0, x1) turned by (c, s) in fp32, rounded to a bf16 pair.
__device__ __forceinline__ uint32_t rotate_pair(uint32_t x, float2 cs) {
  const float x0 = bf16_lo(x), x1 = bf16_hi(x);
  const float y0 = fmaf(x0, cs.x, -x1 * cs.y);
  const float y1 = fmaf(x0, cs.y, x1 * cs.x);
  return dev::pack_bf16x2(y0, y1);
}

__global__ void __launch_bounds__(kWarps * 32)
    kv_append_rope_kernel(const uint4* __restrict__ c_new, const uint32_t* __restrict__ k_pe,
                          const int32_t* __restrict__ positions, const float2* __restrict__ table, int32_t max_pos,
                          const int64_t* __restrict__ slots, int32_t n, uint4* __restrict__ cache, int64_t num_slots,
                          int32_t* err) {
  const int lane = threadIdx.x & 31;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < n; t += (int64_t)gridDim.x * kWarps) {
    const int64_t slot = __ldg(slots + t);
    const int32_t p = __ldg(positions + t);
    if (slot < 0 || slot >= num_slots || p < 0 || p >= max_pos) {
      if (lane == 0) atomicOr(err, (int32_t)((slot < 0 || slot >= num_slots) ? MLA_DEVERR_SLOT_OOB : MLA_DEVERR_POS_OOB));
      continue;
    }
    uint4* dst = cache + slot * kRowVec;
    dst[lane] = __ldg(c_new + t * kLatVec + lane);
    dst[lane + 32] = __ldg(c_new + t * kLatVec + lane + 32);
    const uint32_t r = rotate_pair(__ldg(k_pe + t * kPairs + lane), __ldg(table + (int64_t)p * kPairs + lane));
    reinterpret_cast<uint32_t*>(dst + kLatVec)[lane] = r;
  }
}

// One thread per 16-byte chunk (four pairs) of a (token, head) row: eight
// threads cover a row, so a warp moves 512 contiguous bytes of q_pe with one
// load each and reads its four table pairs as two 16-byte loads.
__global__ void __launch_bounds__(256)
    rope_q_kernel(const uint4* __restrict__ q_pe, const int32_t* __restrict__ positions,
                  const float4* __restrict__ table, int32_t max_pos, uint4* __restrict__ q_r, int64_t chunks,
                  int32_t* err) {
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < chunks; k += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = k >> 3;
    const int c = (int)(k & 7);
    const int32_t p = __ldg(positions + row / MLA_NUM_HEADS);
    if (p < 0 || p >= max_pos) {
      if (c == 0 && row % MLA_NUM_HEADS == 0) atomicOr(err, (int32_t)MLA_DEVERR_POS_OOB);
      continue;
    }
    const uint4 x = __ldg(q_pe + k);
    const float4 t0 = __ldg(table + (int64_t)p * (kPairs / 2) + 2 * c);
    const float4 t1 = __ldg(table + (int64_t)p * (kPairs / 2) + 2 * c + 1);
    uint4 y;
    y.x = rotate_pair(x.x, make_float2(t0.x, t0.y));
    y.y = rotate_pair(x.y, make_float2(t0.z, t0.w));
    y.z = rotate_pair(x.z, make_float2(t1.x, t1.y));
    y.w = rotate_pair(x.w, make_float2(t1.z, t1.w));
    q_r[k] = y;
  }
}

inline int blocks_for(int64_t items) {
  int64_t b = (items + kWarps - 1) / kWarps;
  if (b > 152 * 16) b = 152 * 16;
  return b < 1 ? 1 : (int)b;
}

}  // namespace rope

cudaError_t launch_rope_table(float* table, int32_t max_pos, double base, cudaStream_t stream) {
  if (max_pos <= 0) return cudaSuccess;
  const int64_t n = (int64_t)max_pos * rope::kPairs;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  rope::rope_table_kernel<<<(int)blocks, 256, 0, stream>>>(reinterpret_cast<float2*>(table), max_pos, base);
  return cudaGetLastError();
}

cudaError_t launch_kv_append_rope(const uint16_t* c_kv_new, const uint16_t* k_pe_new, const int32_t* positions,
                                  const float* table, int32_t max_pos, const int64_t* slots, int32_t n,
                                  uint16_t* kv_cache, int64_t num_slots, int32_t* dev_err, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  rope::kv_append_rope_kernel<<<rope::blocks_for(n), rope::kWarps * 32, 0, stream>>>(
      reinterpret_cast<const uint4*>(c_kv_new), reinterpret_cast<const uint32_t*>(k_pe_new), positions,
      reinterpret_cast<const float2*>(table), max_pos, slots, n, reinterpret_cast<uint4*>(kv_cache), num_slots,
      dev_err);
  return cudaGetLastError();
}

cudaError_t launch_rope_q(const uint16_t* q_pe, const int32_t* positions, const float* table, int32_t max_pos,
                          uint16_t* q_r, int32_t T, int32_t* dev_err, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int64_t chunks = (int64_t)T * MLA_NUM_HEADS * 8;
  int64_t blocks = (chunks + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  rope::rope_q_kernel<<<(int)blocks, 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(q_pe), positions, reinterpret_cast<const float4*>(table), max_pos,
      reinterpret_cast<uint4*>(q_r), chunks, dev_err);
  return cudaGetLastError();
}

}  // namespace mla
