// Decompress branch (f2): expansion of the cached latent into per-head keys
// and values in one pass ([P1] "撕开 DeepSeek MLA 源码…" §4 path A,
// K = c_KV·W_UK per head; [P2] MLA section, V = c_KV·W_UV):
//   K_c[h, t, :] = c[t, :]·W_UK[h]^T,   V_c[h, t, :] = c[t, :]·W_UV[h]
// (head-major outputs, one head's rows contiguous for the attention's loads).
//
// A GEMM with a short contraction (512): per 128 x 128 output tile the
// operands weigh as much as the math, so a CTA that loads both for every tile
// is bound by what its SM can take in from L2, not by the tensor pipe.  Two
// CTAs on neighbouring SMs therefore share each MMA (tcgen05 .cta_group::2,
// M = 256 tokens): each CTA keeps its 128 latent rows resident in shared
// memory (all 512 columns, 128 KB) while the pair walks the heads, and loads
// only its half of each head's W_UK and W_UV (N split 64 + 64), 128 KB per
// head per CTA for 2 x 128 x 256 x 512 flops — a third of what a lone CTA
// streams for the same work.
//
// Work unit = (256-token block, head); the pairs take contiguous ranges of
// units in block-major order, so a pair reloads its rows once or twice.
// Warps: 0 TMA producer (both CTAs: rows, then per head the W halves through
// a 5-stage ring, every copy completing on the even CTA's barriers);
// 1 TMEM allocation and, in the even CTA, the MMA issue; 2-5 the epilogue
// (thread = token row = TMEM lane): two 256-column accumulators in TMEM
// (K_c and V_c of one head) alternate, so the epilogue of head h — bf16
// rounding into 128-byte-swizzled boxes, TMA stores — runs under the MMAs of
// head h+1.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace expand {

using namespace mla::dev;

constexpr int kKCh = 512 / 64;                  // 64-wide chunks of the latent
constexpr int kAChunk = 128 * 64 * 2;           // 16 KB: 128 rows x 64, 128-byte swizzle
constexpr int kABytes = kKCh * kAChunk;         // 128 KB: this CTA's rows, resident
constexpr int kBHalf = 64 * 64 * 2;             // 8 KB: this CTA's half of one W chunk
constexpr int kStage = 2 * kBHalf;              // W_UK half | W_UV half
constexpr int kStages = 5;
constexpr int kBoxBytes = 128 * 64 * 2;         // one [128 tokens x 64] bf16 output box
constexpr int kOutBufs = 1;
constexpr int kOffB = kABytes;
constexpr int kOffOut = kOffB + kStages * kStage;
constexpr int kOffBar = kOffOut + kOutBufs * kBoxBytes;
// full[kStages] | empty[kStages] | a_full | a_empty | acc_full[2] | acc_empty[2] | fin
constexpr int kBarFull = 0, kBarEmpty = kStages, kBarAFull = 2 * kStages, kBarAEmpty = kBarAFull + 1,
              kBarAccFull = kBarAEmpty + 1, kBarAccEmpty = kBarAccFull + 2, kBarFin = kBarAccEmpty + 2,
              kNumBars = kBarFin + 1;
constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // abort flag | TMEM slot | W stage uses issued | row loads issued
constexpr int kSmem = kOffMisc + 32 + 1024;
static_assert(kSmem <= 232448, "shared memory");
static_assert(2 * kSmem > 232448, "one CTA per SM: the pair allocates all 512 TMEM columns");
constexpr int kThreads = 192;
constexpr int kTokBlock = 256;                   // tokens per pair and unit
constexpr uint32_t kIdescK = idesc_bf16_f32(256, 128, false, false);  // W_UK read K-major
constexpr uint32_t kIdescV = idesc_bf16_f32(256, 128, false, true);   // W_UV read MN-major
constexpr uint32_t kEpiBar = 1;                  // named barrier of the four epilogue warps

// Number of the first `issued` round-robin uses that fell on stage s.
__device__ __forceinline__ int uses_of(int issued, int s, int stages) {
  return issued > s ? (issued - 1 - s) / stages + 1 : 0;
}

// Retires the last phase of a barrier fed by both CTAs (each `bytes`), armed
// by the even CTA: `mine` / `peer` = uses issued by the even / odd CTA (they
// differ by at most one).  Counts the bytes of the side that never issued,
// arming the phase first if the even CTA did not, then waits (bounded) until
// the copies in flight have landed.
__device__ __forceinline__ void retire_last_phase(uint32_t bar, int mine, int peer, uint32_t bytes) {
  const int n = mine > peer ? mine : peer;
  if (n == 0) return;
  if (mine < n) {
    mbar_arrive_expect_tx(bar, 2u * bytes);
    mbar_complete_tx(bar, bytes);
  } else if (peer < n) {
    mbar_complete_tx(bar, bytes);
  }
  wait_phase_drain(bar, (uint32_t)((n - 1) & 1));
}

// a_map: latent rows {512, 1, n} (box 64 x 1 x 128); k_map: W_UK {512, 128, 128 heads}
// (box 64 x 64 x 1); v_map: W_UV {128, 512, 128 heads} (box 64 x 64 x 1);
// kc_map / vc_map: K_c and V_c {128, n, 128 heads} (box 64 x 128 x 1, stores).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    expand_kv_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap k_map,
                     const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap kc_map,
                     const __grid_constant__ CUtensorMap vc_map, int32_t n, int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + kOffBar;
  auto BAR = [&](int i) { return bars + 8u * (uint32_t)i; };
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(gbase + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kOffMisc + 8);
  volatile int32_t* w_issued = reinterpret_cast<volatile int32_t*>(gbase + kOffMisc + 16);
  volatile int32_t* a_issued = reinterpret_cast<volatile int32_t*>(gbase + kOffMisc + 20);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const int64_t units = (int64_t)((n + kTokBlock - 1) / kTokBlock) * 128;
  const int64_t pairs = gridDim.x / 2, pair = blockIdx.x / 2;
  const int64_t u0 = pair * units / pairs, u1 = (pair + 1) * units / pairs;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *w_issued = 0;
    *a_issued = 0;
    for (int i = 0; i < kNumBars; ++i) mbar_init(BAR(i), i == kBarAccEmpty || i == kBarAccEmpty + 1 ? 8u : 1u);
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any copy or arrival targets them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&a_map);
      prefetch_tmap(&k_map);
      prefetch_tmap(&v_map);
      const uint32_t lead_afull = mapa(BAR(kBarAFull), 0);
      const uint64_t wpol = l2_policy_evict_last();  // W: read by every pair, kept in L2 past the output stream
      int g = 0, na = 0, cur = -1;
      bool ok = true;
      for (int64_t u = u0; u < u1 && ok; ++u) {
        const int tb = (int)(u >> 7), h = (int)(u & 127);
        if (tb != cur) {
          if (na > 0 && !wait_phase(BAR(kBarAEmpty), (uint32_t)((na - 1) & 1), err, abort_flag)) break;
          if (even) mbar_arrive_expect_tx(BAR(kBarAFull), 2u * kABytes);
          const int m0 = tb * kTokBlock + 128 * (int)rank;
          for (int kc = 0; kc < kKCh; ++kc) tma_load_3d_pair(base + kc * kAChunk, &a_map, kc * 64, 0, m0, lead_afull);
          *a_issued = ++na;
          cur = tb;
        }
        for (int kc = 0; kc < kKCh; ++kc, ++g) {
          const int s = g % kStages, use = g / kStages;
          if (use > 0 && !wait_phase(BAR(kBarEmpty + s), (uint32_t)((use - 1) & 1), err, abort_flag)) {
            ok = false;
            break;
          }
          if (even) mbar_arrive_expect_tx(BAR(kBarFull + s), 2u * kStage);
          const uint32_t dst = base + kOffB + s * kStage, lead_full = mapa(BAR(kBarFull + s), 0);
          tma_load_3d_pair_hint(dst, &k_map, kc * 64, 64 * (int)rank, h, lead_full, wpol);
          tma_load_3d_pair_hint(dst + kBHalf, &v_map, 64 * (int)rank, kc * 64, h, lead_full, wpol);
          *w_issued = g + 1;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && even) {
      int g = 0, na = 0, cur = -1, j = 0;
      bool ok = true;
      for (int64_t u = u0; u < u1 && ok; ++u, ++j) {
        const int tb = (int)(u >> 7);
        if (tb != cur) {
          if (na > 0) tc_commit_pair(BAR(kBarAEmpty), 3);  // old rows free once the MMAs reading them end
          if (!wait_phase(BAR(kBarAFull), (uint32_t)(na & 1), err, abort_flag)) break;
          ++na;
          cur = tb;
        }
        const int buf = j & 1, use = j >> 1;
        if (use > 0 && !wait_phase<true>(BAR(kBarAccEmpty + buf), (uint32_t)((use - 1) & 1), err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + 256u * buf;
        for (int kc = 0; kc < kKCh; ++kc, ++g) {
          const int s = g % kStages;
          if (!wait_phase(BAR(kBarFull + s), (uint32_t)((g / kStages) & 1), err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + kc * kAChunk, sb = base + kOffB + s * kStage;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (kc | kk) ? 1u : 0u;
            const uint64_t a = sdesc_sw128(sa + kk * 32, 16, 1024);
            mma_ss_pair(d, a, sdesc_sw128(sb + kk * 32, 16, 1024), kIdescK, acc);
            mma_ss_pair(d + 128, a, sdesc_sw128(sb + kBHalf + kk * 2048, 8192, 1024), kIdescV, acc);
          }
          tc_commit_pair(BAR(kBarEmpty + s), 3);
        }
        if (ok) tc_commit_pair(BAR(kBarAccFull + buf), 3);
      }
      tc_commit_pair(BAR(kBarFin), 3);  // completes once every MMA above has
    }
    __syncwarp();
  } else {
    // Epilogue: thread = token row (TMEM lane); the four warps decide together
    // whether a unit's accumulators are ready, so none is left at a barrier.
    const int q = warp & 3;
    const uint32_t r = (uint32_t)(q * 32 + lane);
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t lead_empty[2] = {mapa(BAR(kBarAccEmpty), 0), mapa(BAR(kBarAccEmpty + 1), 0)};
    const bool issuer = warp == 2 && lane == 0;
    const uint64_t opol = l2_policy_evict_first();  // K_c / V_c: written once, read by the next kernel
    int j = 0, nbox = 0;
    for (int64_t u = u0; u < u1; ++u, ++j) {
      const int tb = (int)(u >> 7), h = (int)(u & 127);
      const int buf = j & 1;
      const bool ready = wait_phase(BAR(kBarAccFull + buf), (uint32_t)((j >> 1) & 1), err, abort_flag);
      if (!named_bar_and(kEpiBar, 128, ready)) break;
      tc_fence_after();
      const int m0 = tb * kTokBlock + 128 * (int)rank;
#pragma unroll 1
      for (int bx = 0; bx < 4; ++bx, ++nbox) {  // K_c columns 0-63, 64-127, then V_c
        const uint32_t box = base + kOffOut + (nbox % kOutBufs) * kBoxBytes;
        if (issuer) bulk_wait_read<kOutBufs - 1>();  // the store from this buffer kOutBufs boxes back has read it
        named_bar_sync(kEpiBar, 128);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t v[32];
          tmem_ld32_sync(tl + 256u * buf + 64u * bx + 32u * hf, v);
          stage_row_bf16_sw128(box, r, hf, v);
        }
        if (bx == 3) {  // this warp has read both accumulators: hand them back to the MMA
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(lead_empty[buf]);
        }
        fence_proxy_async_smem();
        named_bar_sync(kEpiBar, 128);
        if (issuer && m0 < n) {
          tma_store_3d_hint(bx < 2 ? &kc_map : &vc_map, box, (bx & 1) * 64, m0, h, opol);
          bulk_commit_group();
        }
      }
    }
    if (issuer) bulk_wait_all_read();
  }

  // Teardown.  Every copy either CTA issued completes on the even CTA's
  // barriers; after an abort some of those phases may lack one side's bytes,
  // so the even CTA's producer retires each ring's last phase before anyone
  // exits.  Then every MMA has completed (fin) before TMEM is released.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (even && warp == 0 && lane == 0) {
    const int wp = (int)ld_cluster_u32(mapa(smem_u32(const_cast<int32_t*>(w_issued)), 1));
    const int ap = (int)ld_cluster_u32(mapa(smem_u32(const_cast<int32_t*>(a_issued)), 1));
    const int wm = *w_issued, am = *a_issued;
    for (int s = 0; s < kStages; ++s)
      retire_last_phase(BAR(kBarFull + s), uses_of(wm, s, kStages), uses_of(wp, s, kStages), kStage);
    retire_last_phase(BAR(kBarAFull), am, ap, kABytes);
  }
  if (warp == 1 && lane == 0) wait_phase_drain(BAR(kBarFin), 0);
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace expand

cudaError_t launch_expand_kv(const CUtensorMap& a_map, const CUtensorMap& k_map, const CUtensorMap& v_map,
                             const CUtensorMap& kc_map, const CUtensorMap& vc_map, int32_t n, int32_t* err,
                             cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(expand::expand_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       expand::kSmem);
  if (e != cudaSuccess) return e;
  static int max_pairs = 0;
  if (max_pairs == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(expand::kThreads, 1, 1);
    cfg.dynamicSmemBytes = expand::kSmem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int c = 0;
    e = cudaOccupancyMaxActiveClusters(&c, expand::expand_kv_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (c <= 0) return cudaErrorInvalidConfiguration;
    max_pairs = c;
  }
  const int64_t units = (int64_t)((n + expand::kTokBlock - 1) / expand::kTokBlock) * 128;
  const int pairs = (int)(units < max_pairs ? units : max_pairs);
  expand::expand_kv_kernel<<<2 * pairs, expand::kThreads, expand::kSmem, stream>>>(a_map, k_map, v_map, kc_map,
                                                                                   vc_map, n, err);
  return cudaGetLastError();
}

}  // namespace mla
