// Decompress branch (f2): expansion of the cached latent into per-head keys
// and values in one pass ([P1] "撕开 DeepSeek MLA 源码…" §4 path A,
// K = c_KV·W_UK per head; [P2] MLA section, V = c_KV·W_UV):
//   K_c[h, t, :] = c[t, :]·W_UK[h]^T,   V_c[h, t, :] = c[t, :]·W_UV[h]
// (head-major outputs, one head's rows contiguous for the attention's loads).
//
// One CTA = one head and 128 tokens: two 128 x 128 fp32 accumulators in
// TMEM (K and V, 256 columns), so two CTAs share an SM and one's epilogue
// runs while the other's MMAs do (with one CTA of 256 tokens per SM, all 512
// columns in use, the epilogue stalled the tensor pipe: 520 against 470 us
// on the chunked-prefill expansion).  Each 64-wide K-chunk of the latent is
// loaded once for both outputs, so a CTA moves 384 KB for 34 MFLOP, the two
// W tiles coming from L2 for all but the first token block of a head.  Warp
// 0 lane 0 issues TMA, warp 1 lane 0 the MMAs; all four warps run the
// epilogue (thread = token row = TMEM lane), which rounds each accumulator
// to bf16 into the drained ring as two 128-token x 64-column boxes in the
// TMA's 128-byte-swizzled layout and writes each with one TMA store.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace expand {

using namespace mla::dev;

constexpr int kHalves = 1;                      // 128-token blocks per CTA
constexpr int kM = 128 * kHalves, kKCh = 512 / 64;
constexpr int kTile = 128 * 64 * 2;              // 16 KB: 128 rows x 64, 128-byte swizzle
constexpr int kStage = (kHalves + 2) * kTile;    // A rows of each half | W_UK chunk | W_UV chunk
constexpr int kStages = 2;
constexpr int kCtasPerSm = 2;
constexpr int kTmemCols = 256 * kHalves;         // K and V of each half
constexpr int kOffBar = kStages * kStage;
constexpr int kOffMisc = kOffBar + 8 * (2 * kStages + 1);
constexpr int kSmem = kOffMisc + 16 + 1024;
static_assert(kCtasPerSm * kSmem <= 232448 && kCtasPerSm * kTmemCols <= 512, "the CTAs of an SM do not fit");
constexpr uint32_t kIdescK = idesc_bf16_f32(128, 128, false, false);  // W_UK read K-major
constexpr uint32_t kIdescV = idesc_bf16_f32(128, 128, false, true);   // W_UV read MN-major

constexpr int kBoxBytes = 128 * 64 * 2;         // one [128 tokens x 64] bf16 output box
static_assert(4 * kHalves * kBoxBytes <= kStages * kStage, "the output boxes are staged in the drained ring");

// a_map: latent rows {512, 1, n} (box 64 x 1 x 128); k_map: W_UK {512, 128, 128 heads}
// (box 64 x 128 x 1); v_map: W_UV {128, 512, 128 heads} (box 64 x 64 x 1);
// kc_map / vc_map: K_c and V_c {128, n, 128 heads} (box 64 x 128 x 1, stores).
__global__ void __launch_bounds__(128, kCtasPerSm)
    expand_kv_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap k_map,
                     const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap kc_map,
                     const __grid_constant__ CUtensorMap vc_map, int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + kOffBar;
  const uint32_t full0 = bars, empty0 = bars + 8 * kStages, done = bars + 16 * kStages;
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(gbase + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kOffMisc + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int m0 = blockIdx.x * kM;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&a_map);
      prefetch_tmap(&k_map);
      prefetch_tmap(&v_map);
      prefetch_tmap(&kc_map);
      prefetch_tmap(&vc_map);
      int issued = 0;
      for (int kc = 0; kc < kKCh; ++kc) {
        const int st = kc % kStages, use = kc / kStages;
        if (use > 0 && !wait_phase(empty0 + 8 * st, (use - 1) & 1, err, abort_flag)) break;
        const uint32_t dst = base + st * kStage;
        const uint32_t fb = full0 + 8 * st;
        mbar_arrive_expect_tx(fb, (uint32_t)kStage);
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf) tma_load_3d(dst + hf * kTile, &a_map, kc * 64, 0, m0 + 128 * hf, fb);
        tma_load_3d(dst + kHalves * kTile, &k_map, kc * 64, 0, h, fb);
        tma_load_3d(dst + (kHalves + 1) * kTile, &v_map, 0, kc * 64, h, fb);
        tma_load_3d(dst + (kHalves + 1) * kTile + 8192, &v_map, 64, kc * 64, h, fb);
        ++issued;
      }
      for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
        wait_phase_drain(full0 + 8 * (k % kStages), (k / kStages) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      for (int kc = 0; kc < kKCh; ++kc) {
        const int st = kc % kStages;
        if (!wait_phase(full0 + 8 * st, (kc / kStages) & 1, err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = base + st * kStage;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t acc = (kc | kk) ? 1u : 0u;
          const uint64_t bk = sdesc_sw128(sa + kHalves * kTile + kk * 32, 16, 1024);
          const uint64_t bv = sdesc_sw128(sa + (kHalves + 1) * kTile + kk * 2048, 8192, 1024);
#pragma unroll
          for (int hf = 0; hf < kHalves; ++hf) {
            const uint64_t a = sdesc_sw128(sa + hf * kTile + kk * 32, 16, 1024);
            mma_ss(tmem + 256 * hf, a, bk, kIdescK, acc);
            mma_ss(tmem + 256 * hf + 128, a, bv, kIdescV, acc);
          }
        }
        tc_commit(empty0 + 8 * st);
      }
      tc_commit(done);
      if (!ok) wait_phase_drain(done, 0);
    }
    __syncwarp();
  }

  // Epilogue: thread = token row of each 128-token half, all four warps; the
  // decision to store is the whole CTA's, since a box holds every warp's rows.
  bool w = wait_phase(done, 0, err, abort_flag) && !*abort_flag;
  w = __syncthreads_and(w) != 0;
  tc_fence_after();
  if (w) {
    // Every MMA has completed (done), so no load is in flight and the ring is free.
    const uint32_t r = (uint32_t)(warp * 32 + lane);
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int q = 0; q < 2 * kHalves; ++q) {    // K rows 0-127, V rows 0-127, K rows 128-255, V rows 128-255
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t box = base + (q * 2 + b) * kBoxBytes;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t v[32];
          tmem_ld32_sync(tl + q * 128 + b * 64 + hf * 32, v);
          stage_row_bf16_sw128(box, r, hf, v);
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        const CUtensorMap* out = (q & 1) ? &vc_map : &kc_map;
        const int t0 = m0 + (q >> 1) * 128;
        tma_store_3d(out, base + (q * 2) * kBoxBytes, 0, t0, h);
        tma_store_3d(out, base + (q * 2 + 1) * kBoxBytes, 64, t0, h);
        bulk_commit_group();
      }
    }
    if (threadIdx.x == 0) bulk_wait_all_read();  // the staging ring is released at exit
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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
  dim3 grid((n + expand::kM - 1) / expand::kM, 128);
  expand::expand_kv_kernel<<<grid, 128, expand::kSmem, stream>>>(a_map, k_map, v_map, kc_map, vc_map, err);
  return cudaGetLastError();
}

}  // namespace mla
