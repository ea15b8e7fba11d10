// Steps A2 (query absorption) and A5 (V up-projection) as per-head GEMMs on
// the tcgen05 tensor cores:
//   A2  q_abs[t, h, :] = q_c[t, h, :] · W_UK[h]     (K = 128 -> N = 512)
//       ([P1] "撕开 DeepSeek MLA 源码…" §4 path B, einsum 'qhd,hdc->qhc')
//   A5  out[t, h, :]   = o_lat[t, h, :] · W_UV[h]   (K = 512 -> N = 128)
//       ([P2] "DeepSeek的推理为什么比别人便宜一个数量级？…", MLA section: V = c·W_UV)
//
// One CTA computes a 128-row tile of tokens for one head and one of NSPLIT
// column blocks: D[128 x N/NSPLIT] fp32 in TMEM, A (activation rows,
// K-major) and W (row-major [K x N], read as an MN-major operand) staged by
// TMA with 128-byte swizzle through a K-chunk ring.  When split, two CTAs
// fit on an SM, so one CTA's stores overlap another's loads.  The epilogue
// rounds D to bf16 into the drained ring, one 64-column box at a time in the
// TMA's 128-byte-swizzled layout, and writes each box with one TMA store
// (whole 128-byte lines; a thread-per-row store would put 32 rows, 128 KiB
// apart, in every warp instruction).  Rows past T are zero-filled by the
// loads and clipped by the stores.  For small T the kernel streams the
// 16 MiB of weights once (HBM bound).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace gemm {

using namespace mla::dev;

template <int N, int K, int STAGES, int NSPLIT>
struct Cfg {
  static constexpr int kNC = N / NSPLIT;  // columns of this CTA
  static constexpr int kKCh = K / 64;
  static constexpr int kABytes = 128 * 64 * 2;
  static constexpr int kBBytes = 64 * kNC * 2;
  static constexpr int kStage = kABytes + kBBytes;
  static constexpr int kOffBar = STAGES * kStage;
  static constexpr int kOffMisc = kOffBar + 8 * (2 * STAGES + 1);
  static constexpr int kSmem = kOffMisc + 16 + 1024;
  static constexpr int kMmaN = kNC < 256 ? kNC : 256;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(128, kMmaN, false, true);
  static_assert((NSPLIT == 1 ? 1 : 2) * kSmem <= 232448, "a split head GEMM needs two CTAs per SM");
  static_assert(kNC % 64 == 0 && kNC >= 64, "column block is a multiple of 64");
  static constexpr int kBoxBytes = 128 * 64 * 2;  // one [128 x 64] bf16 output box
  static_assert((kNC / 64) * kBoxBytes <= STAGES * kStage, "the output boxes are staged in the drained ring");
};

template <int N, int K, int STAGES, int NSPLIT>
__global__ void __launch_bounds__(128, 2)
    head_gemm_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap w_map,
                     const __grid_constant__ CUtensorMap c_map, int32_t* err) {
  using C = Cfg<N, K, STAGES, NSPLIT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + C::kOffBar;
  const uint32_t full0 = bars, empty0 = bars + 8 * STAGES, done = bars + 16 * STAGES;
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(gbase + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int m0 = blockIdx.x * 128;
  const int n0 = blockIdx.z * C::kNC;  // first output column of this CTA

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), C::kNC);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&a_map);
      prefetch_tmap(&w_map);
      prefetch_tmap(&c_map);
      int issued = 0;
      for (int kc = 0; kc < C::kKCh; ++kc) {
        const int st = kc % STAGES, use = kc / STAGES;
        if (use > 0 && !wait_phase(empty0 + 8 * st, (use - 1) & 1, err, abort_flag)) break;
        const uint32_t dst = base + st * C::kStage;
        mbar_arrive_expect_tx(full0 + 8 * st, (uint32_t)C::kStage);
        tma_load_3d(dst, &a_map, kc * 64, h, m0, full0 + 8 * st);
#pragma unroll
        for (int nb = 0; nb < C::kNC / 64; ++nb)
          tma_load_3d(dst + C::kABytes + nb * 8192, &w_map, n0 + nb * 64, kc * 64, h, full0 + 8 * st);
        ++issued;
      }
      for (int k = (issued > STAGES ? issued - STAGES : 0); k < issued; ++k)
        wait_phase_drain(full0 + 8 * (k % STAGES), (k / STAGES) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      for (int kc = 0; kc < C::kKCh; ++kc) {
        const int st = kc % STAGES;
        if (!wait_phase(full0 + 8 * st, (kc / STAGES) & 1, err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = base + st * C::kStage;
        const uint32_t sb = sa + C::kABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
          for (int nh = 0; nh < C::kNC / C::kMmaN; ++nh)
            mma_ss(tmem + nh * C::kMmaN, sdesc_sw128(sa + kk * 32, 16, 1024),
                   sdesc_sw128(sb + nh * (C::kMmaN / 64) * 8192 + kk * 2048, 8192, 1024), C::kIdesc,
                   (kc | kk) ? 1u : 0u);
        tc_commit(empty0 + 8 * st);
      }
      tc_commit(done);  // also fires (after in-flight MMAs) when the loop stopped early
      if (!ok) wait_phase_drain(done, 0);
    }
    __syncwarp();
  }

  // Epilogue: thread = tile row (TMEM lane), all four warps; the decision to
  // store is taken by the whole CTA, since the boxes need every warp's rows.
  bool w = wait_phase(done, 0, err, abort_flag) && !*abort_flag;
  w = __syncthreads_and(w) != 0;
  tc_fence_after();
  if (w) {
    // Every MMA has completed (done), so no load is in flight and the ring is free.
    const uint32_t r = (uint32_t)(warp * 32 + lane);
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int b = 0; b < C::kNC / 64; ++b) {
      const uint32_t box = base + b * C::kBoxBytes;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[32];
        tmem_ld32_sync(tl + b * 64 + hf * 32, v);
        stage_row_bf16_sw128(box, r, hf, v);
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        tma_store_3d(&c_map, box, n0 + b * 64, h, m0);
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
    tmem_dealloc(tmem, C::kNC);
  }
}

template <int N, int K, int STAGES, int NSPLIT>
cudaError_t run(const CUtensorMap& a_map, const CUtensorMap& w_map, const CUtensorMap& c_map, int32_t T,
                int32_t* err, cudaStream_t stream) {
  using C = Cfg<N, K, STAGES, NSPLIT>;
  auto* kern = head_gemm_kernel<N, K, STAGES, NSPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((T + 127) / 128, 128, NSPLIT);
  kern<<<grid, 128, C::kSmem, stream>>>(a_map, w_map, c_map, err);
  return cudaGetLastError();
}

}  // namespace gemm

cudaError_t launch_head_gemm(HeadGemm kind, const CUtensorMap& a_map, const CUtensorMap& w_map,
                             const CUtensorMap& c_map, int32_t T, int32_t* err, cudaStream_t stream) {
  if (kind == HeadGemm::kAbsorbQ) return gemm::run<512, 128, 2, 2>(a_map, w_map, c_map, T, err, stream);
  return gemm::run<128, 512, 4, 1>(a_map, w_map, c_map, T, err, stream);
}

}  // namespace mla
