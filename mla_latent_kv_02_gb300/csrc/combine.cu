// Step A4: merge of the split-KV partials.  The pages print no softmax
// kernel; the attention of [P1] "撕开 DeepSeek MLA 源码…" §4 path B is an exact
// softmax over the visible tokens, and a row whose tokens were cut into
// pieces is the log-sum-exp weighted mean of the pieces' normalised outputs:
//   o_lat = Σ_i 2^(lse_i - m) o_i / Σ_i 2^(lse_i - m),   lse = (m + log2 Σ_i 2^(lse_i - m)) ln 2,
// with o_i the fp32 normalised partial of piece i, lse_i its log2-sum-exp
// and m = max_i lse_i.
//
// One CTA = one split row and HPC heads; TPH threads per head, each with QPT
// of the head's 128 column quads (float4), loaded for two pieces at once.
// Many split rows: 16 heads x 16 threads x 8 quads (one wave covers the
// merge); few (one or sixteen query rows cut into many pieces): one head x
// 128 threads x 1 quad, so that the few rows spread over many SMs.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace comb {

using namespace mla::dev;

constexpr int kH = 128, kDC = 512;

template <int HPC, int QPT>
__global__ void __launch_bounds__(HPC * 128 / QPT) combine_kernel(const CombineArgs a) {
  constexpr int kTPH = 128 / QPT;  // threads per head
  const int r = blockIdx.x, tid = threadIdx.x;
  const int h = blockIdx.y * HPC + tid / kTPH, q0 = tid % kTPH;
  const int row = a.split_rows[4 * r], s0 = a.split_rows[4 * r + 1], n = a.split_rows[4 * r + 2];
  if (row < 0 || row >= a.T || s0 < 0 || n < 1 || s0 + n > a.num_partials) {
    if (tid == 0) atomicOr(a.dev_err, (int32_t)MLA_DEVERR_PLAN);
    return;
  }
  // One pass over the pieces, two at a time, with a running maximum: both
  // pieces' outputs and log-sum-exps are loaded together, so a row of two
  // pieces costs one round of loads.
  float mx = -INFINITY, wsum = 0.f;
  float4 acc[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  const uint64_t last_use = l2_policy_evict_first();  // the partials' only read
#pragma unroll 1
  for (int i = 0; i < n; i += 2) {
    const bool two = i + 1 < n;
    const float la = __ldg(a.part_lse + (size_t)(s0 + i) * kH + h);
    const float lb = two ? __ldg(a.part_lse + (size_t)(s0 + i + 1) * kH + h) : -INFINITY;
    const float4* pa = reinterpret_cast<const float4*>(a.part_o + ((size_t)(s0 + i) * kH + h) * kDC) + q0;
    float4 va[QPT], vb[QPT];
#pragma unroll
    for (int k = 0; k < QPT; ++k) va[k] = ld_global_v4_hint(pa + kTPH * k, last_use);
    if (two) {
      const float4* pb = pa + (size_t)kH * kDC / 4;
#pragma unroll
      for (int k = 0; k < QPT; ++k) vb[k] = ld_global_v4_hint(pb + kTPH * k, last_use);
    } else {
#pragma unroll
      for (int k = 0; k < QPT; ++k) vb[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float mn = fmaxf(mx, fmaxf(la, lb));
    const float sc = exp2f(mx - mn), wa = exp2f(la - mn), wb = two ? exp2f(lb - mn) : 0.f;
    mx = mn;
    wsum = wsum * sc + wa + wb;
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      acc[k].x = acc[k].x * sc + wa * va[k].x + wb * vb[k].x;
      acc[k].y = acc[k].y * sc + wa * va[k].y + wb * vb[k].y;
      acc[k].z = acc[k].z * sc + wa * va[k].z + wb * vb[k].z;
      acc[k].w = acc[k].w * sc + wa * va[k].w + wb * vb[k].w;
    }
  }
  const float inv = 1.f / wsum;
  uint2* dst = reinterpret_cast<uint2*>(a.o_lat + ((size_t)row * kH + h) * kDC) + q0;
#pragma unroll
  for (int k = 0; k < QPT; ++k)
    dst[kTPH * k] = make_uint2(pack_bf16x2(acc[k].x * inv, acc[k].y * inv), pack_bf16x2(acc[k].z * inv, acc[k].w * inv));
  if (q0 == 0 && a.lse) a.lse[(size_t)row * kH + h] = (mx + log2f(wsum)) * 0.6931471805599453f;
}

}  // namespace comb

cudaError_t launch_combine(const CombineArgs& args, int num_split_rows, cudaStream_t stream) {
  if (num_split_rows <= 0) return cudaSuccess;
  if (num_split_rows >= 32)
    comb::combine_kernel<16, 8><<<dim3(num_split_rows, comb::kH / 16), 16 * 16, 0, stream>>>(args);
  else
    comb::combine_kernel<1, 1><<<dim3(num_split_rows, comb::kH), 128, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace mla
