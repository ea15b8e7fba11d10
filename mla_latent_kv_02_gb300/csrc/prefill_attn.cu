// Decompress branch (f2): causal multi-head attention over the expanded
// cache, the pages' "path A" for long query chunks.
//
// [P1] "撕开 DeepSeek MLA 源码…" §3 (kPrefillThresh = 256: a chunk of at
// least that many query tokens is not absorbed but decompressed) and §4
// path A: K = c_KV·W_UK per head, s = (q_c·K + q_R·k_R)·(d_hc + d_r)^-1/2;
// [P2] MLA section: V = c_KV·W_UV; out = softmax(s)·V per head.
//
// One CTA = one head h and 128 query rows of one sequence of the batch
// (blockIdx.z; its rows and cache tokens sit at offsets of the packed
// arrays); query row i sits at position N - M + i and sees keys
// [0, N - M + i].  Keys of a sequence's last tile that belong to the next
// sequence are past N - 1 and always masked; query rows past M compute as
// the last row and are not stored.  Key tiles of 128 tokens stream by TMA
// through a 3-deep ring of K = [K_c[h, ., 0:128] | k_R] (192 columns,
// K-major) and a 2-deep ring of V = V_c[h, ., :] (MN-major); K_c and V_c are
// head-major, so a head's tile is 32 contiguous KB.  tcgen05:
//   S(j) = Q·K(j)^T   M = 128, N = 128, K = 192   (A = Q from TMEM)
//   O   += P(j)·V(j)  M = 128, N = 128, K = 128   (A = P from TMEM)
// TMEM: O 128 | S 128 | P 2 x 64 | Q 96 columns.  QK^T(j+1) waits only
// until the softmax has read S(j) into registers; P(j) is written while
// P·V(j-1) still reads the other P buffer (P(j) waits for P·V(j-2)).  Q
// sits in TMEM (copied from the third K stage, its landing place, before
// K(2) loads there), which frees shared memory for the third K stage.  The
// row sum l is kept per half by the softmax threads (the rounded bf16 P,
// summed in fp32) and the halves' sums are added at the end.
// Warps: 0 TMA producer, 1 TMEM allocation + QK^T issue,
// 10 P·V issue (an MMA issue blocks while the tensor pipe's queue is full, so
// one thread issuing both would hold P·V(j) behind QK^T(j+1)),
// 2-9 softmax and epilogue: two warps per query row (thread = TMEM lane),
// each with 64 of a tile's 128 key columns; the two halves of a row swap
// their maxima through shared memory and the named barrier of their lane
// quarter once per tile.  P·V(j) is issued only after every MMA of
// QK^T(j + 2) (QK^T first in the tensor pipe, so the key stages free
// sooner).  The softmax
// follows the decode kernel's: fp16 raw scores, a lazily moved reference max
// (8 log2 units), P = 2^(c2 (s - m)) with one fused multiply-add, bf16 P.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace prefill {

using namespace mla::dev;

constexpr int kBM = 128, kBN = 128;                // query rows, key tokens per tile
constexpr int kChunkBytes = 128 * 64 * 2;          // [128 rows x 64] bf16, 128-byte swizzle: 16 KB
constexpr int kKBytes = 3 * kChunkBytes;           // K_c (2 chunks) | k_R (1 chunk); q_c | q_r the same way
constexpr int kVBytes = 2 * kChunkBytes;           // V_c (2 chunks of 64 columns)
constexpr int kStages = 3;                         // depth of the K ring
constexpr int kVStages = 2;                        // depth of the V ring
constexpr int kQStage = 2;                         // the K stage Q lands in (K(2) loads there after Q's copy)
constexpr int kPvLag = 2;                          // P·V(j) is issued after every MMA of QK^T(j + kPvLag) (0: no order)
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kStages * kKBytes;
constexpr int kAlignedBytes = kOffV + kVStages * kVBytes;
constexpr int kNumBars = 26;
constexpr int kOffXMax = 8 * kNumBars + 64;         // float [2 tile parities][2 halves][128 rows]
constexpr int kOffXSum = kOffXMax + 2 * 2 * 128 * 4; // float [2 halves][128 rows]: the halves' row sums
constexpr int kSmallBytes = kOffXSum + 2 * 128 * 4;
constexpr int kSmemBytes = kSmallBytes + kAlignedBytes + 1024;
static_assert(kSmemBytes <= 232448, "shared memory layout does not fit");

// TMEM: O, the score buffer, two P buffers (tile j's in buffer j mod 2), Q
constexpr uint32_t kColO = 0, kColS = 128, kColP = 256, kColQ = 384, kTmemCols = 512;
constexpr int kSoftWarp0 = 2;
constexpr int kSoftWarps = 8;                      // two warps per TMEM lane quarter, 64 key columns each
constexpr int kPvWarp = kSoftWarp0 + kSoftWarps;
constexpr int kThreads = 32 * (kPvWarp + 1);
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);

enum : int {
  B_Q_FULL = 0,
  B_Q_TMEM,                         // Q copied into TMEM, one arrival per softmax warp
  B_K_FULL,                         // kStages each: K and V have their own rings, so a K
  B_K_EMPTY = B_K_FULL + kStages,   // stage frees when QK^T is done, before P·V
  B_V_FULL = B_K_EMPTY + kStages,
  B_V_EMPTY = B_V_FULL + kVStages,
  B_S_FULL = B_V_EMPTY + kVStages,  // 2 (tile parity)
  B_S_FREE = B_S_FULL + 2,          // 2 (tile parity), one arrival per softmax warp
  B_P_FULL = B_S_FREE + 2,          // 2 (P buffer), one arrival per softmax warp
  B_O_DONE = B_P_FULL + 2,          // 2 (tile parity): P·V of tile j complete
  B_DRAIN = B_O_DONE + 2,
  B_DRAIN_PV,
  B_XSUM,                           // the halves' row sums, one arrival per softmax warp
  B_COUNT
};
static_assert(B_COUNT <= kNumBars, "barrier area too small");

__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<const __half2*>(&u); }
__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }

// q_map: q_c [M, 128, 128] as {128, 128 heads, M}; r_map: q_r {64, 128, M};
// k_map / v_map: K_c / V_c [128, N, 128] as {128, N, 128 heads}; kr_map: the
// gathered cache rows [N, 576] as {576, N} (k_R at column 512).  Boxes of
// 64 columns x 128 rows, 128-byte swizzle.
__global__ void __launch_bounds__(kThreads, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap r_map,
                        const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap kr_map,
                        const __grid_constant__ CUtensorMap v_map, const PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t bars = raw;
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem_raw + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + 8 * kNumBars + 8);
  volatile int32_t* qk_issued = reinterpret_cast<volatile int32_t*>(smem_raw + 8 * kNumBars + 16);
  const uint32_t base = (raw + kSmallBytes + 1023u) & ~1023u;
#define BAR(i) (bars + 8u * (uint32_t)(i))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y;
  const int i0 = qt * kBM;
  const PrefillSeq sq = a.seq[blockIdx.z];
  if (i0 >= sq.M) return;                             // this sequence has fewer query tiles
  const int M = sq.M, N = sq.N;
  const int kv_base = N - M;                          // position of query row 0
  const int last_row = min(i0 + kBM, M) - 1;
  const int n_tiles = (kv_base + last_row) / kBN + 1;  // tiles any row of this CTA sees
  int32_t* err = a.dev_err;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *qk_issued = -1;
    mbar_init(BAR(B_Q_FULL), 1);
    mbar_init(BAR(B_Q_TMEM), kSoftWarps);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(BAR(B_K_FULL + i), 1);
      mbar_init(BAR(B_K_EMPTY + i), 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(BAR(B_V_FULL + i), 1);
      mbar_init(BAR(B_V_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(B_S_FULL + i), 1);
      mbar_init(BAR(B_S_FREE + i), kSoftWarps);
    }
    mbar_init(BAR(B_P_FULL), kSoftWarps);
    mbar_init(BAR(B_P_FULL + 1), kSoftWarps);
    mbar_init(BAR(B_O_DONE), 1);
    mbar_init(BAR(B_O_DONE + 1), 1);
    mbar_init(BAR(B_XSUM), kSoftWarps);
    mbar_init(BAR(B_DRAIN), 1);
    mbar_init(BAR(B_DRAIN_PV), 1);
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
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&q_map);
      prefetch_tmap(&k_map);
      prefetch_tmap(&v_map);
      const uint32_t qdst = base + kOffK + kQStage * kKBytes;
      mbar_arrive_expect_tx(BAR(B_Q_FULL), (uint32_t)kKBytes);
      tma_load_3d(qdst, &q_map, 0, h, sq.q_off + i0, BAR(B_Q_FULL));
      tma_load_3d(qdst + kChunkBytes, &q_map, 64, h, sq.q_off + i0, BAR(B_Q_FULL));
      tma_load_3d(qdst + 2 * kChunkBytes, &r_map, 0, h, sq.q_off + i0, BAR(B_Q_FULL));
      // K(nk) as soon as its stage is free (QK^T(nk-3) done; K(2)'s stage once
      // Q has left it for TMEM), V(nv) as soon as its stage is free (P·V(nv-2)
      // done); a tile's K goes before its V.
      int nk = 0, nv = 0;
      bool ok = true;
      uint64_t t_last = cycles();
      uint32_t spins = 0;
      while (ok && nv < n_tiles) {
        bool progressed = false;
        if (nk < n_tiles && (nk < kStages ? (nk != kQStage || mbar_test_wait(BAR(B_Q_TMEM), 0))
                                          : mbar_test_wait(BAR(B_K_EMPTY + nk % kStages), ((nk - kStages) / kStages) & 1))) {
          const int st = nk % kStages, t0 = sq.kv_off + nk * kBN;
          const uint32_t dst = base + kOffK + st * kKBytes;
          mbar_arrive_expect_tx(BAR(B_K_FULL + st), (uint32_t)kKBytes);
          tma_load_3d(dst, &k_map, 0, t0, h, BAR(B_K_FULL + st));
          tma_load_3d(dst + kChunkBytes, &k_map, 64, t0, h, BAR(B_K_FULL + st));
          tma_load_2d(dst + 2 * kChunkBytes, &kr_map, 512, t0, BAR(B_K_FULL + st));
          ++nk;
          progressed = true;
        }
        if (nv < nk && (nv < kVStages || mbar_test_wait(BAR(B_V_EMPTY + nv % kVStages), ((nv - kVStages) / kVStages) & 1))) {
          const int st = nv % kVStages, t0 = sq.kv_off + nv * kBN;
          const uint32_t dst = base + kOffV + st * kVBytes;
          mbar_arrive_expect_tx(BAR(B_V_FULL + st), (uint32_t)kVBytes);
          tma_load_3d(dst, &v_map, 0, t0, h, BAR(B_V_FULL + st));
          tma_load_3d(dst + kChunkBytes, &v_map, 64, t0, h, BAR(B_V_FULL + st));
          ++nv;
          progressed = true;
        }
        if (progressed) {
          spins = 0;
          t_last = cycles();
        } else if ((++spins & 255u) == 0u) {
          if (*abort_flag) {
            ok = false;
          } else if (cycles() - t_last > kWaitLimitCycles) {
            atomicOr(err, (int32_t)MLA_DEVERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
          }
        }
      }
      // loads still in flight land before the CTA may exit
      wait_phase_drain(BAR(B_Q_FULL), 0);
      for (int k = (nk > kStages ? nk - kStages : 0); k < nk; ++k)
        wait_phase_drain(BAR(B_K_FULL + k % kStages), (k / kStages) & 1);
      for (int k = (nv > kVStages ? nv - kVStages : 0); k < nv; ++k)
        wait_phase_drain(BAR(B_V_FULL + k % kVStages), (k / kVStages) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- QK^T issue
    // S(j) = Q·K(j)^T once K(j) has landed and the softmax has read S(j-1)
    // out of the score buffer.
    if (lane == 0) {
      const uint64_t kdesc0 = sdesc_sw128(base + kOffK, 16, 1024);
      bool ok = wait_phase<false, false>(BAR(B_Q_TMEM), 0, err, abort_flag);
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j % kStages, sb = j & 1;
        ok = wait_phase<false, false>(BAR(B_K_FULL + st), (j / kStages) & 1, err, abort_flag) &&
             (j < 1 || wait_phase<false, false>(BAR(B_S_FREE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, err, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint64_t dk = kdesc0 + (uint64_t)((st * kKBytes) >> 4);
#pragma unroll
        for (int c = 0; c < 3; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + kColS, tmem + kColQ + c * 32 + kk * 8,
                   dk + (uint64_t)((c * kChunkBytes + kk * 32) >> 4), kIdescQK, (c | kk) ? 1u : 0u);
        tc_commit(BAR(B_S_FULL + sb));
        tc_commit(BAR(B_K_EMPTY + st));
        *qk_issued = j;
      }
      // every MMA of this thread has finished before TMEM is released
      tc_commit(BAR(B_DRAIN));
      wait_phase_drain(BAR(B_DRAIN), 0);
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ---------------------------------------------------------------- P·V issue
    // O += P(j)·V(j) once the softmax has written P(j) (buffer j mod 2) and
    // V(j) has landed.
    if (lane == 0) {
      const uint64_t vdesc0 = sdesc_sw128(base + kOffV, (uint32_t)kChunkBytes, 1024);
      bool ok = true;
      for (int t = 0; ok && t < n_tiles; ++t) {
        ok = wait_phase<false, false>(BAR(B_P_FULL + (t & 1)), (t >> 1) & 1, err, abort_flag) &&
             wait_phase<false, false>(BAR(B_V_FULL + t % kVStages), (t / kVStages) & 1, err, abort_flag);
        if (!ok) break;
        // QK^T first in the tensor pipe: P·V(t) waits until every MMA of
        // QK^T(t + kPvLag) is issued (which needs nothing P·V(t) produces),
        // so the key stages free sooner
        if (kPvLag > 0 && t + kPvLag < n_tiles && *qk_issued < t + kPvLag) {
          const uint64_t t0 = cycles();
          for (uint32_t it = 1; *qk_issued < t + kPvLag; ++it) {
            if ((it & 255u) == 0u && (*abort_flag || cycles() - t0 > kWaitLimitCycles)) {
              if (!*abort_flag) atomicOr(err, (int32_t)MLA_DEVERR_TIMEOUT);
              *abort_flag = 1;
              ok = false;
              break;
            }
          }
          if (!ok) break;
        }
        tc_fence_after();
        const uint64_t dv = vdesc0 + (uint64_t)(((t % kVStages) * kVBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t acc = (t == 0 && kk == 0) ? 0u : 1u;
          mma_ts(tmem + kColO, tmem + kColP + (t & 1) * 64 + kk * 8, dv + (uint64_t)((kk * 2048) >> 4), kIdescPV, acc);
        }
        tc_commit(BAR(B_V_EMPTY + t % kVStages));
        tc_commit(BAR(B_O_DONE + (t & 1)));
      }
      tc_commit(BAR(B_DRAIN_PV));
      wait_phase_drain(BAR(B_DRAIN_PV), 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax + epilogue
    const int q4 = warp & 3;                       // TMEM lane quarter this warp may access
    const int half = (warp - kSoftWarp0) >> 2;     // key columns [64 half, 64 half + 64) of each tile
    const int r = q4 * 32 + lane;                  // query row of the tile = TMEM lane
    const int i = i0 + r;                          // query index in the chunk
    const int pos = kv_base + min(i, M - 1);       // rows past M act as the last row and are not stored
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    float* xmax = reinterpret_cast<float*>(smem_raw + kOffXMax);
    const float c2 = a.scale_log2;
    const float rescale_thr = 8.f / c2;            // lazy rescale: 8 in log2 units
    const __half2 c2h = __float2half2_rn(c2);
    float m = -INFINITY;
    float l = 0.f;                                 // this half's row sum of P, at the reference max m
    bool ok = true;
    {
      // Q into TMEM: row r's dims in packed pairs, half 0 the q_c chunks, half 1 q_r
      bool w = wait_phase<false, true>(BAR(B_Q_FULL), 0, err, abort_flag);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
      } else {
        const uint32_t qsrc = base + kOffK + kQStage * kKBytes + (uint32_t)r * 128u;
#pragma unroll 1
        for (int cc = 2 * half; cc < 2 + half; ++cc) {
          uint32_t v[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 x = ld_shared_v4(qsrc + cc * kChunkBytes + (((uint32_t)u ^ ((uint32_t)r & 7u)) << 4));
            v[4 * u] = __float_as_uint(x.x);
            v[4 * u + 1] = __float_as_uint(x.y);
            v[4 * u + 2] = __float_as_uint(x.z);
            v[4 * u + 3] = __float_as_uint(x.w);
          }
          tmem_st32(tl + kColQ + 32 * cc, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_Q_TMEM));
      }
    }
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int sb = j & 1;
      bool w = wait_phase<false, true>(BAR(B_S_FULL + sb), (j >> 1) & 1, err, abort_flag);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t own[32];                            // raw scores as fp16 pairs, then P as bf16 pairs
      {
        uint32_t s[64];
        tmem_ld64_sync(tl + kColS + half * 64, s);
#pragma unroll
        for (int k = 0; k < 32; ++k)
          own[k] = cvt_f16x2_satfinite(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_S_FREE + sb));
      // causal mask: token j*128 + 64 half + c is visible iff it is <= pos
      const int valid = pos - j * kBN - 64 * half + 1;
      if (valid < 64) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          if (2 * k >= valid) own[k] = (own[k] & 0xFFFF0000u) | 0xFC00u;
          if (2 * k + 1 >= valid) own[k] = (own[k] & 0x0000FFFFu) | 0xFC000000u;
        }
      }
      __half2 mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = as_h2(own[k]);
#pragma unroll
      for (int k = 8; k < 32; ++k) mx[k & 7] = __hmax2(mx[k & 7], as_h2(own[k]));
      const __half2 mh = __hmax2(__hmax2(__hmax2(mx[0], mx[1]), __hmax2(mx[2], mx[3])),
                                 __hmax2(__hmax2(mx[4], mx[5]), __hmax2(mx[6], mx[7])));
      // swap the halves' maxima through a tile-parity buffer and the named
      // barrier of this lane quarter's two warps: a warp writes tile j+2's
      // value only after passing tile j+1's barrier, which its partner
      // reaches after reading tile j's values.  A warp that leaves the loop
      // early arrives once (below), which releases its partner's current or
      // next sync; the partner cannot reach a second one, since QK^T of the
      // tile after needs both warps' score reads (the abort check before the
      // sync only makes it leave sooner).
      xmax[(sb * 2 + half) * 128 + r] = fmaxf(__low2float(mh), __high2float(mh));
      if (*abort_flag) {
        ok = false;
        break;
      }
      named_bar_sync(1 + q4, 64);
      const float mt = fmaxf(xmax[(sb * 2) * 128 + r], xmax[(sb * 2 + 1) * 128 + r]);
      float factor = 1.f;
      bool resc = false;
      if (j == 0) {
        m = mt;
      } else if (mt > m + rescale_thr) {
        factor = exp2f((m - mt) * c2);
        m = mt;
        resc = true;
      }
      const __half2 mc2 = __float2half2_rn(-m * c2);
      float rs0 = 0.f, rs1 = 0.f;                  // row sum of the bf16 P the tensor core accumulates
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float2 p = __half22float2(as_h2(ex2_f16x2(as_u32(__hfma2(as_h2(own[k]), c2h, mc2)))));
        own[k] = pack_bf16x2(p.x, p.y);
        rs0 += __uint_as_float(own[k] << 16);
        rs1 += __uint_as_float(own[k] & 0xFFFF0000u);
      }
      l = fmaf(l, factor, rs0 + rs1);
      // P buffer j mod 2 was last read by P·V(j-2); waited first, it also keeps
      // a rescale's wait for P·V(j-1) below within one phase of its barrier
      if (j >= 2) {
        w = wait_phase<false, true>(BAR(B_O_DONE + (j & 1)), ((j >> 1) - 1) & 1, err, abort_flag);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, resc)) {
        // a rescale of O needs P·V(j-1) done (P·V(j) waits for this tile's P)
        w = wait_phase<false, true>(BAR(B_O_DONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, err, abort_flag);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // each half rescales its 64 output columns
#pragma unroll 1
        for (int c = 64 * half; c < 64 * half + 64; c += 32) {
          uint32_t o[32];
          tmem_ld32_sync(tl + kColO + c, o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * factor);
          tmem_st32(tl + kColO + c, o);
        }
      }
      tmem_st32(tl + kColP + (j & 1) * 64 + 32 * half, own);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_P_FULL + (j & 1)));
    }
    if (!ok) named_bar_arrive(1 + q4, 64);
    // ---- epilogue: out[i, h, 64 half : 64 half + 64] = O / l, l the sum of
    //      the two halves' row sums (swapped through shared memory)
    if (ok && n_tiles > 0) {
      float* xsum = reinterpret_cast<float*>(smem_raw + kOffXSum);
      xsum[half * 128 + r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_XSUM));
      const int nl = n_tiles - 1;
      bool w = wait_phase<false, true>(BAR(B_XSUM), 0, err, abort_flag) &&
               wait_phase<false, true>(BAR(B_O_DONE + (nl & 1)), (nl >> 1) & 1, err, abort_flag);
      if (__all_sync(0xffffffffu, w)) {
        tc_fence_after();
        const float inv = 1.f / (xsum[r] + xsum[128 + r]);
        uint4* dst = reinterpret_cast<uint4*>(a.out + ((size_t)(sq.q_off + min(i, M - 1)) * 128 + h) * 128);
#pragma unroll 1
        for (int c = 64 * half; c < 64 * half + 64; c += 32) {
          uint32_t o[32];
          tmem_ld32_sync(tl + kColO + c, o);
          if (i < M) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c / 8 + v] = make_uint4(
                  pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv),
                  pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv),
                  pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv),
                  pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv));
          }
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
#undef BAR
}

}  // namespace prefill
}  // namespace mla

namespace mla {

int prefill_smem_bytes() { return prefill::kSmemBytes; }

cudaError_t launch_prefill_attn(const CUtensorMap& q_map, const CUtensorMap& r_map, const CUtensorMap& k_map,
                                const CUtensorMap& kr_map, const CUtensorMap& v_map, const PrefillArgs& args,
                                cudaStream_t stream) {
  int max_m = 0;
  for (int i = 0; i < args.nb; ++i) max_m = args.seq[i].M > max_m ? args.seq[i].M : max_m;
  if (args.nb <= 0 || max_m <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(prefill::prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       prefill::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((max_m + prefill::kBM - 1) / prefill::kBM, 128, args.nb);
  prefill::prefill_attn_kernel<<<grid, prefill::kThreads, prefill::kSmemBytes, stream>>>(q_map, r_map, k_map,
                                                                                        kr_map, v_map, args);
  return cudaGetLastError();
}

}  // namespace mla
