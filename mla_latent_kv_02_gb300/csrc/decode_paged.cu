// Steps A3 + A4: absorbed paged MLA attention (split-KV) and the combine.
//
// Method ([P1] "撕开 DeepSeek MLA 源码：C++ 与 TensorRT-LLM 算子设计优化全景与 TaoToken 实践",
// §4 path B and §3 constants): per query row t and head h,
//   s_j = (q_abs[t,h]·c_KV[j] + q_R[t,h]·k_R[j]) · scale,
//   o_lat[t,h] = Σ_j softmax(s)_j · c_KV[j],   lse[t,h] = ln Σ_j e^{s_j}.
//
// GB300 design (one CTA pair = one 2-CTA cluster per work range):
//  * The fp32 latent accumulator O[128 heads × 512] is exactly one SM's TMEM
//    (128 lanes × 512 columns), so the pair splits the latent columns: CTA r
//    owns O[:, 256r : 256r+256) and streams only its columns of each 64-token
//    page by TMA — no byte of the cache is read twice.
//  * The score contraction (576 = 9 chunks of 64) is split the same way: CTA 0
//    takes latent chunks 0-3, CTA 1 latent chunks 4-7 plus the RoPE chunk.  Each
//    CTA computes a partial S = Q_r·K_r^T (tcgen05, M = 128 heads, N = 64
//    tokens, A = Q from TMEM, B = the page tile in shared memory) and the two
//    partials are exchanged through distributed shared memory (st.async into
//    the peer, completing on the peer's mbarrier).  Both CTAs then hold the
//    same full S (fp32 addition is commutative), run the same online softmax,
//    write P (bf16) into TMEM and accumulate O_r += P·V_r (tcgen05, N = 256,
//    B = the same page tile read as an MN-major operand).
//  * Online softmax with lazy rescaling: the running reference max only moves
//    when a tile's max exceeds it by more than 8 (log2 units), so P stays
//    below 256 and O in TMEM is rescaled only on those rare tiles.
//  * Warp roles: warp 0 TMA producer, warp 1 TMEM allocation + MMA issue,
//    warps 2-5 softmax/epilogue (thread = head row = TMEM lane).
//  * Work: the plan cuts all rows' 64-token tiles into equal contiguous ranges,
//    one per cluster; a row cut by a boundary is written as fp32 partials
//    (normalised O and log2-sum-exp) and merged by the combine kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace decode {

using namespace mla::dev;

constexpr int kH = 128, kDC = 512, kDR = 64, kPage = 64;
constexpr int kChunk = 64;                                // elements in one 128-byte swizzled row
constexpr int kChunkBytes = kPage * kChunk * 2;           // [64 tokens x 64] bf16 = 8 KB
constexpr int kMaxQKChunks = 5;
constexpr int kStageBytes = kMaxQKChunks * kChunkBytes;   // 40 KB
constexpr int kStages = 4;
constexpr int kXBytes = kH * kPage * 4;                   // one CTA's fp32 partial S
constexpr int kOffKV = 0;
constexpr int kOffX = kStages * kStageBytes;
constexpr int kOffBar = kOffX + 2 * kXBytes;
constexpr int kOffMisc = kOffBar + 8 * 32;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;          // + slack to align the base to 1024 B
static_assert(kSmemBytes <= 232448, "decode kernel exceeds 227 KB of shared memory");

constexpr uint32_t kColO = 0, kColS = 256, kColQ = 320, kColP = 480, kTmemCols = 512;
constexpr int kThreads = 192;

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, false, true);

enum : int {
  B_KV_FULL = 0,
  B_KV_EMPTY = kStages,
  B_S_FULL = 2 * kStages,
  B_S_FREE,
  B_P_FULL,
  B_O_DONE,
  B_Q_READY,
  B_O_FREE,
  B_X_FULL0,
  B_X_FULL1,
  B_DRAIN,
  B_COUNT
};
static_assert(B_COUNT <= 32, "barrier area too small");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(gbase + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kOffMisc + 8);
  int32_t* seg_range = reinterpret_cast<int32_t*>(gbase + kOffMisc + 16);
  const uint32_t bars = base + kOffBar;
#define BAR(i) (bars + 8u * (uint32_t)(i))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cid = blockIdx.x >> 1;
  const int nq = rank ? 5 : 4;      // score-contraction chunks held by this CTA
  const int chunk0 = rank ? 4 : 0;  // first of them within the 576-wide token row
  int32_t* err = a.dev_err;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(BAR(B_KV_FULL + i), 1);
      mbar_init(BAR(B_KV_EMPTY + i), 1);
    }
    mbar_init(BAR(B_S_FULL), 1);
    mbar_init(BAR(B_S_FREE), 128);
    mbar_init(BAR(B_P_FULL), 128);
    mbar_init(BAR(B_O_DONE), 1);
    mbar_init(BAR(B_Q_READY), 128);
    mbar_init(BAR(B_O_FREE), 128);
    mbar_init(BAR(B_X_FULL0), 1);
    mbar_init(BAR(B_X_FULL1), 1);
    mbar_init(BAR(B_DRAIN), 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    // Validate this cluster's plan range; an inconsistent plan is skipped whole
    // (by every role alike) and reported instead of being dereferenced.
    int32_t sb = a.seg_off[cid], se = a.seg_off[cid + 1];
    bool good = sb >= 0 && se >= sb && se <= a.num_segments;
    for (int s = sb; good && s < se; ++s) {
      const int32_t* sg = a.segs + 8 * s;
      const int32_t row = sg[0], b = sg[1], pb = sg[2], pe = sg[3], vis = sg[4], slot = sg[5];
      good = row >= 0 && row < a.T && b >= 0 && b < a.B && pb >= 0 && pe > pb && pe <= a.max_pages && vis >= 1 &&
             (int64_t)(pe - 1) * kPage < (int64_t)vis && slot >= -1 && slot < a.num_partials;
    }
    if (!good) {
      atomicOr(err, (int32_t)MLA_DEVERR_PLAN);
      sb = se = 0;
    }
    seg_range[0] = sb;
    seg_range[1] = se;
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&kv_map);
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any st.async reaches them
  const uint32_t tmem = *tmem_slot;

  const int s_begin = seg_range[0];
  const int s_end = seg_range[1];

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t g = 0;
      bool ok = true;
      for (int s = s_begin; s < s_end && ok; ++s) {
        const int32_t* sg = a.segs + 8 * s;
        const int b = sg[1], pb = sg[2], pe = sg[3];
        const int32_t* bt = a.block_table + (int64_t)b * a.max_pages;
        for (int pg = pb; pg < pe; ++pg) {
          const uint32_t st = g % kStages, use = g / kStages;
          if (use > 0 && !wait_phase(BAR(B_KV_EMPTY + st), (use - 1) & 1u, err, abort_flag)) {
            ok = false;
            break;
          }
          int32_t pid = __ldg(bt + pg);
          if (pid < 0 || (int64_t)pid >= a.num_pages) {
            atomicOr(err, (int32_t)MLA_DEVERR_PAGE_OOB);
            pid = 0;
          }
          const uint32_t dst = base + kOffKV + st * kStageBytes;
          mbar_arrive_expect_tx(BAR(B_KV_FULL + st), (uint32_t)(nq * kChunkBytes));
          for (int i = 0; i < nq; ++i)
            tma_load_2d(dst + i * kChunkBytes, &kv_map, (chunk0 + i) * kChunk, pid * kPage, BAR(B_KV_FULL + st));
          ++g;
        }
      }
      // Loads still in flight must land before this CTA may exit.
      for (uint32_t k = (g > (uint32_t)kStages ? g - kStages : 0u); k < g; ++k)
        wait_phase_drain(BAR(B_KV_FULL + k % kStages), (k / kStages) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      uint32_t g = 0;
      int segi = 0;
      bool ok = true, pend = false, pend_first = false;
      uint32_t pend_g = 0;
      int pend_seg = 0;
      auto issue_pv = [&](uint32_t gp, bool first, int si) -> bool {
        if (!wait_phase(BAR(B_P_FULL), gp & 1u, err, abort_flag)) return false;
        if (first && !wait_phase(BAR(B_O_FREE), (uint32_t)si & 1u, err, abort_flag)) return false;
        tc_fence_after();
        const uint32_t v = base + kOffKV + (gp % kStages) * kStageBytes;
        // O_r[128 x 256] += P[128 x 64] · V_r[64 x 256]; V_r is MN-major: 4 atoms
        // of 64 columns 8 KB apart (LBO), 8-token row groups 1 KB apart (SBO).
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(tmem + kColO, tmem + kColP + kk * 8, sdesc_sw128(v + kk * 2048, 8192, 1024), kIdescPV,
                 (first && kk == 0) ? 0u : 1u);
        tc_commit(BAR(B_KV_EMPTY + gp % kStages));
        tc_commit(BAR(B_O_DONE));
        return true;
      };
      for (int s = s_begin; s < s_end && ok; ++s, ++segi) {
        const int32_t* sg = a.segs + 8 * s;
        const int pb = sg[2], pe = sg[3];
        if (!wait_phase(BAR(B_Q_READY), (uint32_t)segi & 1u, err, abort_flag)) {
          ok = false;
          break;
        }
        for (int pg = pb; pg < pe; ++pg) {
          const uint32_t st = g % kStages;
          if (!wait_phase(BAR(B_KV_FULL + st), (g / kStages) & 1u, err, abort_flag) ||
              (g > 0 && !wait_phase(BAR(B_S_FREE), (g - 1) & 1u, err, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kv = base + kOffKV + st * kStageBytes;
          // S_partial[128 x 64] = Q_r[128 x 64*nq] · K_r^T, K-major, 16 per step.
          for (int i = 0; i < nq; ++i)
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tmem + kColS, tmem + kColQ + i * 32 + kk * 8,
                     sdesc_sw128(kv + i * kChunkBytes + kk * 32, 16, 1024), kIdescQK, (i | kk) ? 1u : 0u);
          tc_commit(BAR(B_S_FULL));
          if (pend && !issue_pv(pend_g, pend_first, pend_seg)) {
            ok = false;
            break;
          }
          pend = true;
          pend_g = g;
          pend_first = (pg == pb);
          pend_seg = segi;
          ++g;
        }
      }
      if (ok && pend) ok = issue_pv(pend_g, pend_first, pend_seg);
      // Every MMA must be finished before TMEM is released.
      tc_commit(BAR(B_DRAIN));
      wait_phase_drain(BAR(B_DRAIN), 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax + epilogue
    const int q4 = warp & 3;
    const int h = q4 * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);  // this warp's TMEM lane quarter
    const uint32_t xrow = base + kOffX + (uint32_t)h * 256u;
    const uint32_t swz = (uint32_t)(h & 7);
    const float scale_log2 = a.scale_log2;
    __syncwarp();

    auto load_q = [&](int s) {
      const int row = a.segs[8 * s];
      const uint4* src = reinterpret_cast<const uint4*>(a.q_abs + ((size_t)row * kH + h) * kDC + rank * 256);
      uint32_t r[32];
#pragma unroll
      for (int part = 0; part < 4; ++part) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = __ldg(src + part * 8 + v);
          r[4 * v] = x.x;
          r[4 * v + 1] = x.y;
          r[4 * v + 2] = x.z;
          r[4 * v + 3] = x.w;
        }
        tmem_st32(tl + kColQ + part * 32, r);
      }
      if (rank == 1) {
        const uint4* srr = reinterpret_cast<const uint4*>(a.q_r + ((size_t)row * kH + h) * kDR);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = __ldg(srr + v);
          r[4 * v] = x.x;
          r[4 * v + 1] = x.y;
          r[4 * v + 2] = x.z;
          r[4 * v + 3] = x.w;
        }
        tmem_st32(tl + kColQ + 128, r);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(BAR(B_Q_READY));
    };

    mbar_arrive(BAR(B_O_FREE));  // O is free for the first segment
    if (s_begin < s_end) load_q(s_begin);
    uint32_t g = 0;
    bool ok = true;
    for (int s = s_begin; s < s_end && ok; ++s) {
      const int32_t* sg = a.segs + 8 * s;
      const int row = sg[0], pb = sg[2], pe = sg[3], vis = sg[4], slot = sg[5];
      float m = -INFINITY, l = 0.f;
      for (int pg = pb; pg < pe; ++pg, ++g) {
        bool w = wait_phase(BAR(B_S_FULL), g & 1u, err, abort_flag);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[64];
        {
          uint32_t r[32];
          tmem_ld32_sync(tl + kColS, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[i] = __uint_as_float(r[i]);
          tmem_ld32_sync(tl + kColS + 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[32 + i] = __uint_as_float(r[i]);
        }
        tc_fence_before();
        mbar_arrive(BAR(B_S_FREE));
        if (pg == pe - 1 && s + 1 < s_end) load_q(s + 1);  // all QK of this segment are done

        // ---- exchange partial scores with the peer CTA
        const uint32_t xb = g & 1u;
        if (h == 0) mbar_arrive_expect_tx(BAR(B_X_FULL0 + xb), (uint32_t)kXBytes);
        const uint32_t my_row = xrow + xb * (uint32_t)kXBytes;
        const uint32_t rrow = mapa(my_row, peer);
        const uint32_t rbar = mapa(BAR(B_X_FULL0 + xb), peer);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          st_async_v4(rrow + (((uint32_t)k ^ swz) << 4), sv[4 * k], sv[4 * k + 1], sv[4 * k + 2], sv[4 * k + 3], rbar);
        w = wait_phase<true>(BAR(B_X_FULL0 + xb), (g >> 1) & 1u, err, abort_flag);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float4 v = ld_shared_v4(my_row + (((uint32_t)k ^ swz) << 4));
          sv[4 * k] += v.x;
          sv[4 * k + 1] += v.y;
          sv[4 * k + 2] += v.z;
          sv[4 * k + 3] += v.w;
        }

        // ---- scale (log2 domain), causal/length mask, online softmax
        const int valid = vis - pg * kPage;
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float x = (j < valid) ? sv[j] * scale_log2 : -INFINITY;
          sv[j] = x;
          mt = fmaxf(mt, x);
        }
        float factor = 1.f;
        bool resc = false;
        if (pg == pb) {
          m = mt;
        } else if (mt > m + 8.f) {
          factor = exp2f(m - mt);
          m = mt;
          l *= factor;
          resc = true;
        }
        // P (single TMEM buffer) and an O rescale both need PV of the previous tile done.
        if (g > 0) {
          w = wait_phase(BAR(B_O_DONE), (g - 1) & 1u, err, abort_flag);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int c = 0; c < 256; c += 32) {
            uint32_t r[32];
            tmem_ld32_sync(tl + kColO + c, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * factor);
            tmem_st32(tl + kColO + c, r);
          }
        }
        uint32_t pk[32];
        float rs = 0.f;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const __nv_bfloat162 v = __floats2bfloat162_rn(exp2f(sv[2 * jj] - m), exp2f(sv[2 * jj + 1] - m));
          pk[jj] = *reinterpret_cast<const uint32_t*>(&v);
          rs += __low2float(v) + __high2float(v);
        }
        l += rs;
        tmem_st32(tl + kColP, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(B_P_FULL));
      }
      if (!ok) break;

      // ---- epilogue of this segment: wait for the last P·V, normalise, store
      bool w = wait_phase(BAR(B_O_DONE), (g - 1) & 1u, err, abort_flag);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = 1.f / l;
      if (slot < 0) {
        uint4* dst = reinterpret_cast<uint4*>(a.o_lat + ((size_t)row * kH + h) * kDC + rank * 256);
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          uint32_t r[32];
          tmem_ld32_sync(tl + kColO + c, r);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[c / 8 + v] = make_uint4(
                pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv, __uint_as_float(r[8 * v + 1]) * inv),
                pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv, __uint_as_float(r[8 * v + 3]) * inv),
                pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv, __uint_as_float(r[8 * v + 5]) * inv),
                pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv, __uint_as_float(r[8 * v + 7]) * inv));
        }
      } else {
        float4* dst = reinterpret_cast<float4*>(a.part_o + ((size_t)slot * kH + h) * kDC + rank * 256);
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          uint32_t r[32];
          tmem_ld32_sync(tl + kColO + c, r);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[c / 4 + v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                         __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(B_O_FREE));
      if (rank == 0) {
        const float lse2 = m + log2f(l);
        if (slot < 0) {
          if (a.lse) a.lse[(size_t)row * kH + h] = lse2 * 0.6931471805599453f;
        } else {
          a.part_lse[(size_t)slot * kH + h] = lse2;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // neither CTA leaves while its peer may still address its shared memory
#undef BAR
}

// Merge split rows: lse = log2 Σ 2^{lse_s} (log2 domain), o = Σ 2^{lse_s - lse} o_s.
__global__ void __launch_bounds__(128) combine_kernel(const CombineArgs a) {
  const int r = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int row = a.split_rows[4 * r], s0 = a.split_rows[4 * r + 1], n = a.split_rows[4 * r + 2];
  if (row < 0 || row >= a.T || s0 < 0 || n < 1 || s0 + n > a.num_partials) {
    if (tid == 0) atomicOr(a.dev_err, (int32_t)MLA_DEVERR_PLAN);
    return;
  }
  float mx = -INFINITY;
  for (int i = 0; i < n; ++i) mx = fmaxf(mx, __ldg(a.part_lse + (size_t)(s0 + i) * kH + h));
  float wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = 0; i < n; ++i) {
    const float w = exp2f(__ldg(a.part_lse + (size_t)(s0 + i) * kH + h) - mx);
    const float4 v = __ldg(reinterpret_cast<const float4*>(a.part_o + ((size_t)(s0 + i) * kH + h) * kDC) + tid);
    wsum += w;
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  const float inv = 1.f / wsum;
  uint2 out;
  out.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  out.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(a.o_lat + ((size_t)row * kH + h) * kDC)[tid] = out;
  if (tid == 0 && a.lse) a.lse[(size_t)row * kH + h] = (mx + log2f(wsum)) * 0.6931471805599453f;
}

}  // namespace decode

int decode_smem_bytes() { return decode::kSmemBytes; }
int decode_threads() { return decode::kThreads; }

cudaError_t decode_prepare() {
  return cudaFuncSetAttribute(decode::decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              decode::kSmemBytes);
}

cudaError_t decode_max_clusters(int* out) {
  cudaError_t e = decode_prepare();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(decode::kThreads, 1, 1);
  cfg.dynamicSmemBytes = decode::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, (const void*)decode::decode_kernel, &cfg);
}

cudaError_t launch_decode(const CUtensorMap& kv_map, const DecodeArgs& args, int num_clusters,
                          cudaStream_t stream) {
  cudaError_t e = decode_prepare();
  if (e != cudaSuccess) return e;
  decode::decode_kernel<<<2 * num_clusters, decode::kThreads, decode::kSmemBytes, stream>>>(kv_map, args);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& args, int num_split_rows, cudaStream_t stream) {
  if (num_split_rows <= 0) return cudaSuccess;
  decode::combine_kernel<<<dim3(num_split_rows, decode::kH), 128, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace mla
