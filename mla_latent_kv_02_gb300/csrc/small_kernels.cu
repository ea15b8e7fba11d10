// Step A1 (append a token's [c_KV | k_R] row at its slot) and the paged
// gather used to check what the decode kernel reads, bit for bit.
//
// [P2] "DeepSeek的推理为什么比别人便宜一个数量级？…", closing inference-flow
// summary: each step's new latent joins the cache; [P1] "撕开 DeepSeek MLA
// 源码…" §3: pages of 64 tokens, 576 bf16 per token (1152 B, 72 16-byte
// vectors); §5: 16-byte aligned vector access.
//
// One warp per token: 72 coalesced 16-byte copies per row.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace small {

constexpr int kRowVec = 72;    // 576 bf16 = 72 x 16 B
constexpr int kLatVec = 64;    // 512 bf16
constexpr int kRopeVec = 8;    // 64 bf16
constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
    kv_append_kernel(const uint4* __restrict__ c_new, const uint4* __restrict__ k_new,
                     const int64_t* __restrict__ slots, int32_t n, uint4* __restrict__ cache, int64_t num_slots,
                     int32_t* err) {
  const int lane = threadIdx.x & 31;
  for (int64_t i = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); i < n; i += (int64_t)gridDim.x * kWarps) {
    // the row's 72 16-byte pieces (up to three per lane) and its slot are
    // requested together: one memory round trip before the stores
    uint4 v[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int k = lane + 32 * j;
      if (k < kRowVec) v[j] = k < kLatVec ? __ldg(c_new + i * kLatVec + k) : __ldg(k_new + i * kRopeVec + (k - kLatVec));
    }
    const int64_t slot = __ldg(slots + i);
    if (slot < 0 || slot >= num_slots) {
      if (lane == 0) atomicOr(err, (int32_t)MLA_DEVERR_SLOT_OOB);
      continue;
    }
    uint4* dst = cache + slot * kRowVec;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int k = lane + 32 * j;
      if (k < kRowVec) dst[k] = v[j];
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32)
    gather_kernel(const uint4* __restrict__ cache, int64_t num_pages, const int32_t* __restrict__ block_table,
                  int32_t max_pages, int32_t b, int32_t n_tokens, uint4* __restrict__ out, int32_t* err) {
  const int lane = threadIdx.x & 31;
  for (int64_t j = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); j < n_tokens; j += (int64_t)gridDim.x * kWarps) {
    const int32_t pid = __ldg(block_table + (int64_t)b * max_pages + j / 64);
    if (pid < 0 || (int64_t)pid >= num_pages) {
      if (lane == 0) atomicOr(err, (int32_t)MLA_DEVERR_PAGE_OOB);
      continue;
    }
    const uint4* src = cache + ((int64_t)pid * 64 + j % 64) * kRowVec;
    for (int k = lane; k < kRowVec; k += 32) out[j * kRowVec + k] = __ldg(src + k);
  }
}

// The packed gather of several sequences (the decompress branch of a
// batch): a warp finds its token's sequence by bisection of the offsets.
__global__ void __launch_bounds__(kWarps * 32)
    gather_batch_kernel(const uint4* __restrict__ cache, int64_t num_pages, const int32_t* __restrict__ block_table,
                        int32_t max_pages, const __grid_constant__ GatherBatch g, uint4* __restrict__ out,
                        int32_t* err) {
  const int lane = threadIdx.x & 31;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < g.total;
       t += (int64_t)gridDim.x * kWarps) {
    int lo = 0, hi = g.nb - 1;  // the last sequence whose offset is <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (g.off[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    const int64_t j = t - g.off[lo];
    if (j < 0 || j >= g.n[lo]) {  // offsets inconsistent with the lengths
      if (lane == 0) atomicOr(err, (int32_t)MLA_DEVERR_BATCH);
      continue;
    }
    const int32_t pid = __ldg(block_table + (int64_t)g.b[lo] * max_pages + j / 64);
    if (pid < 0 || (int64_t)pid >= num_pages) {
      if (lane == 0) atomicOr(err, (int32_t)MLA_DEVERR_PAGE_OOB);
      continue;
    }
    const uint4* src = cache + ((int64_t)pid * 64 + j % 64) * kRowVec;
    for (int k = lane; k < kRowVec; k += 32) out[t * kRowVec + k] = __ldg(src + k);
  }
}

inline int blocks_for(int64_t items) {
  int64_t b = (items + kWarps - 1) / kWarps;
  if (b > 152 * 16) b = 152 * 16;
  return b < 1 ? 1 : (int)b;
}

}  // namespace small

cudaError_t launch_kv_append(const uint16_t* c_kv_new, const uint16_t* k_r_new, const int64_t* slots, int32_t n,
                             uint16_t* kv_cache, int64_t num_slots, int32_t* dev_err, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  small::kv_append_kernel<<<small::blocks_for(n), small::kWarps * 32, 0, stream>>>(
      reinterpret_cast<const uint4*>(c_kv_new), reinterpret_cast<const uint4*>(k_r_new), slots, n,
      reinterpret_cast<uint4*>(kv_cache), num_slots, dev_err);
  return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t* kv_cache, int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                          int32_t b, int32_t n_tokens, uint16_t* out, int32_t* dev_err, cudaStream_t stream) {
  if (n_tokens <= 0) return cudaSuccess;
  small::gather_kernel<<<small::blocks_for(n_tokens), small::kWarps * 32, 0, stream>>>(
      reinterpret_cast<const uint4*>(kv_cache), num_pages, block_table, max_pages, b, n_tokens,
      reinterpret_cast<uint4*>(out), dev_err);
  return cudaGetLastError();
}

cudaError_t launch_gather_batch(const uint16_t* kv_cache, int64_t num_pages, const int32_t* block_table,
                                int32_t max_pages, const GatherBatch& g, uint16_t* out, int32_t* dev_err,
                                cudaStream_t stream) {
  if (g.total <= 0 || g.nb <= 0) return cudaSuccess;
  small::gather_batch_kernel<<<small::blocks_for(g.total), small::kWarps * 32, 0, stream>>>(
      reinterpret_cast<const uint4*>(kv_cache), num_pages, block_table, max_pages, g, reinterpret_cast<uint4*>(out),
      dev_err);
  return cudaGetLastError();
}

}  // namespace mla
