// Step A3: absorbed paged MLA attention (split-KV); the combine (A4) is in combine.cu.
//
// Method ([P1] "撕开 DeepSeek MLA 源码：C++ 与 TensorRT-LLM 算子设计优化全景与 TaoToken 实践",
// §4 path B and §3 constants): per query row t and head h,
//   s_j = (q_abs[t,h]·c_KV[j] + q_R[t,h]·k_R[j]) · scale,
//   o_lat[t,h] = Σ_j softmax(s)_j · c_KV[j],   lse[t,h] = ln Σ_j e^{s_j}.
//
// GB300 design (one 2-CTA cluster per work range):
//  * The fp32 latent accumulator O[128 heads × 512] is exactly one SM's TMEM
//    (128 lanes × 512 columns), so the pair splits the latent columns: CTA r
//    owns O[:, 256r : 256r+256) and streams only its columns of each 64-token
//    page by TMA — no byte of the cache is read twice.
//  * The score contraction (576) is split evenly: CTA r takes latent chunks
//    4r..4r+3 (64 columns each, 128-byte swizzle) and RoPE dims [32r, 32r+32)
//    (64-byte swizzle).  Each CTA computes a partial S = Q_r·K_r^T (tcgen05,
//    M = 128 heads, N = 64 tokens, A = Q from TMEM, B = the page tile in shared
//    memory).  The partials are exchanged unscaled as fp16 (the scale times
//    log2 e enters once, in the exponent of P): each
//    warp stages its rows and one bulk copy per warp pushes them into the peer
//    CTA, completing on the peer's mbarrier.  Both CTAs add the same two
//    rounded halves, so they hold bit-identical S and take identical softmax
//    decisions.
//  * Softmax in packed fp16 (add, max, subtract, 2^x with one MUFU issue per
//    pair), P converted to bf16 and written to TMEM; O_r += P·V_r (tcgen05,
//    N = 256, B = the same page tile read as an MN-major operand) and the row
//    sums l += P·1 (N = 16 against a tile of ones), so l matches exactly the
//    bf16 P the tensor core accumulated.
//  * Exchange ring: kXBufs receive buffers per CTA; tile t lands in buffer
//    t mod kXBufs, and the rows this CTA sends for tile t are staged in its own
//    buffer (t + kXLead) mod kXBufs.  Pushing tile t needs only the peer's tile
//    t - kXLead to have arrived: that arrival proves the peer's copy out of
//    the buffer tile t goes to has finished, and that the peer had consumed
//    what it held.  No release message crosses the cluster.
//  * Two softmax warpgroups take alternate tiles, each tile whole (thread =
//    head row = TMEM lane, all 64 tokens): while one waits for the peer's half
//    of its tile, the other computes.  The only hand-off between them is the
//    row's reference max, passed from tile g-1 to tile g through a tagged
//    shared-memory slot.  QK^T and P·V are issued by two warps, each as soon
//    as its own inputs are ready.
//  * Online softmax with lazy rescaling: the running reference max only moves
//    when a tile's max exceeds it by more than 8 (log2 units), so P stays
//    below 256 and O and l in TMEM are rescaled only on those rare tiles.
//  * Warp roles: warp 0 TMA producer, warp 1 TMEM allocation + QK^T issue,
//    warps 2-9 softmax/epilogue (two warpgroups), warp 10 P·V issue.
//  * Work: the plan cuts all rows' 64-token tiles into equal contiguous ranges,
//    one per cluster; a row cut by a boundary is written as fp32 partials
//    (normalised O and log2-sum-exp) and merged by the combine kernel.
//  * Every wait in the loop is bounded (DecodeArgs::wait_limit); on expiry the
//    kernel raises an abort flag that every role polls, drains its own TMA
//    loads and MMAs, waits until the score copies the peer already issued
//    into this CTA have landed, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fp8.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace decode {

using namespace mla::dev;

constexpr int kH = 128, kDC = 512, kDR = 64, kPage = 64;
constexpr int kChunk = 64;                                // elements in one 128-byte swizzled row
constexpr int kChunkBytes = kPage * kChunk * 2;           // [64 tokens x 64] bf16 = 8 KB
constexpr int kRopeHalf = 32;                             // RoPE dims per CTA
constexpr int kRopeBytes = kPage * kRopeHalf * 2;         // [64 tokens x 32] bf16 = 4 KB, 64-byte rows
constexpr int kXBytes = kH * kPage * 2;                   // one CTA's fp16 partial S (16 KB)
// Softmax: two warpgroups take alternate tiles whole (thread = head row).
constexpr int kSWarps = 8;
constexpr int kWords = kPage / 2;                         // fp16x2 words of a row's 64 scores
constexpr int kXRow = kPage * 2;                          // one row of a partial S tile (128 bytes)
constexpr int kXWarp = 32 * kXRow;                        // one warp's 32 rows (4 KB)
constexpr int kXBufs = 4;                                 // exchange ring depth
constexpr int kXLead = kXBufs - 2;                        // staging buffer offset
static_assert(kXLead >= 1 && kXLead <= kXBufs - 2, "the exchange ring needs two tiles between staging and reuse");
constexpr int kOnesBytes = 16 * kChunk * 2;               // [16 x 64] bf16 ones for the row sums

// FP8 stage (one page, this CTA's half): the 32 KB latent area, whose first
// 16 KB first receive the 64 token rows of 256 E4M3 codes and are then
// overwritten by their bf16 values; the RoPE half (64-byte swizzle); the 64
// token scales.
constexpr int kF8Codes = kPage * 256;                     // 16 KB
constexpr int kF8RopeOff = 4 * kChunkBytes;               // 32 KB
constexpr int kF8ScaleOff = kF8RopeOff + kRopeBytes;
constexpr int kF8Payload = kF8Codes + kRopeBytes + kPage * 4;  // bytes the TMA delivers per stage
constexpr int kF8StageBytes = 37 * 1024;                  // keeps every stage 1024-byte aligned
constexpr int kConvWarps = 4;
constexpr uint32_t kConvBarrier = 1;                      // named barrier of the converter warps
static_assert(kF8ScaleOff + kPage * 4 <= kF8StageBytes, "FP8 stage too small");

// Shared memory: a small region (barriers, row-max slots, flags) at the
// start, then the 1024-byte aligned region (page ring, FP8 staging ring,
// exchange ring, the ones tile).
constexpr int kNumBars = 32;
constexpr int kSmallBar = 0;
constexpr int kSmallPair = kSmallBar + 8 * kNumBars;      // uint2 [4][128]: {reference max bits, tile}
constexpr int kSmallMisc = kSmallPair + 4 * kH * 8;
// misc: +0 abort flag, +8 TMEM address, +16 segment range [2], +32 copies
// issued per softmax warp [8], +64 the peer's copies [8] (written by the
// peer), +96 the abort flags of this CTA and the peer [2], +104 the last tile
// armed on each exchange buffer [4], +120 the last tile whose QK^T MMAs are
// all issued (FP8).
constexpr int kMiscPush = 32, kMiscPeerPush = 64, kMiscAborts = 96, kMiscArmed = 104, kMiscQkIssued = 120;
constexpr int kSmallBytes = kSmallMisc + 128;

// The two cache formats.  bf16: the producer's TMA fills a 4-deep ring of
// [latent half | RoPE half] stages.  FP8: the TMA fills the same 4-deep ring
// with [codes | RoPE half | scales], and a converter warpgroup dequantises
// the codes in place (all codes read into registers, a barrier, then the
// bf16 rows written over them).  Warp roles:
//   bf16: 0 producer, 1 QK^T, 2-9 softmax, 10 P·V                (352 threads)
//   FP8:  0 producer, 1 QK^T, 2 P·V, 3 idle, 4-11 softmax,
//         12-15 converters; warpgroups 0 and 3 give registers to 1 and 2 (512)
template <bool kF8>
struct Cfg;
template <>
struct Cfg<false> {
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = 4 * kChunkBytes + kRopeBytes;  // 36 KB
  static constexpr int kSoftWarp0 = 2, kPvWarp = 2 + kSWarps, kConvWarp0 = 1 << 20;
  static constexpr int kThreads = 32 * (kPvWarp + 1);
};
template <>
struct Cfg<true> {
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = kF8StageBytes;                 // 37 KB
  static constexpr int kSoftWarp0 = 4, kPvWarp = 2, kConvWarp0 = 12;
  static constexpr int kThreads = 512;
};

template <bool kF8>
struct Layout : Cfg<kF8> {
  using C = Cfg<kF8>;
  static constexpr int kOffKV = 0;
  static constexpr int kOffX = C::kStages * C::kStageBytes;
  static constexpr int kOffOnes = kOffX + kXBufs * kXBytes;
  static constexpr int kAlignedBytes = kOffOnes + kOnesBytes;
  static constexpr int kSmemBytes = kSmallBytes + kAlignedBytes + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory layout does not fit");
  enum : int {
    B_KV_FULL = 0,
    B_KV_EMPTY = C::kStages,
    // S_FULL and O_DONE come in pairs by tile parity: each softmax warpgroup
    // waits only on its own tiles' phases, in order (a parity test cannot tell
    // a phase from the one two before it, and the warpgroups run apart).
    B_S_FULL0 = 2 * C::kStages,
    B_S_FULL1,
    B_S_FREE,
    B_P_FULL,
    B_O_DONE0,
    B_O_DONE1,
    B_Q_READY,
    B_O_FREE,
    B_X_FULL0,                      // exchange buffer i filled by the peer
    B_DRAIN = B_X_FULL0 + kXBufs,
    B_DRAIN_PV,
    B_F8_FULL,                      // FP8: stage i's codes, RoPE half and scales landed
    B_COUNT = B_F8_FULL + (kF8 ? C::kStages : 0)
  };
  static_assert(B_COUNT <= kNumBars, "barrier area too small");
};

constexpr uint32_t kColO = 0, kColS = 256, kColSum = 320, kColQ = 336, kColP = 480, kTmemCols = 512;
// The producer and the two MMA-issuing threads poll (mbarrier.test_wait)
// rather than sleep: their wake-up sits on the score chain.
constexpr bool kIssueSuspend = false;
constexpr uint32_t kTileThreads = 128;                    // the warpgroup that handles one tile

// bf16 operands for the bf16 cache; f16 for the FP8 cache (an E4M3 value is
// an exact f16, and P is computed in f16 in both).
template <bool kF8>
struct Idesc {
  static constexpr uint32_t kQK = kF8 ? idesc_f16_f32(128, 64, false, false) : idesc_bf16_f32(128, 64, false, false);
  static constexpr uint32_t kPV = kF8 ? idesc_f16_f32(128, 256, false, true) : idesc_bf16_f32(128, 256, false, true);
  static constexpr uint32_t kSum = kF8 ? idesc_f16_f32(128, 16, false, false) : idesc_bf16_f32(128, 16, false, false);
};

// Walks the 64-token tiles of a cluster's segments in order; a segment's
// fields are read from the plan once, when the cursor enters it.
struct TileCursor {
  const int32_t* segs;
  int s, s_end, pg, pb, pe, row, vis, slot;
  __device__ __forceinline__ void init(const int32_t* sg, int sb, int se) {
    segs = sg;
    s = sb;
    s_end = se;
    if (s < s_end) load();
  }
  __device__ __forceinline__ void load() {
    // {row, b, page_begin, page_end} and {visible, out_slot, 0, 0}: 16-byte aligned
    const int4 lo = __ldg(reinterpret_cast<const int4*>(segs + 8 * s));
    const int4 hi = __ldg(reinterpret_cast<const int4*>(segs + 8 * s) + 1);
    row = lo.x;
    pb = lo.z;
    pe = lo.w;
    vis = hi.x;
    slot = hi.y;
    pg = pb;
  }
  __device__ __forceinline__ bool valid() const { return s < s_end; }
  __device__ __forceinline__ bool first() const { return pg == pb; }
  __device__ __forceinline__ bool last() const { return pg == pe - 1; }
  __device__ __forceinline__ void next() {
    if (++pg == pe) {
      ++s;
      if (s < s_end) load();
    }
  }
};

__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<const __half2*>(&u); }
__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }

// kv_map / rope_map: bf16 cache — latent chunks (3D, 128-byte swizzle) and
// RoPE halves; FP8 cache — code rows (uint8, 256-byte boxes, no swizzle) and
// RoPE halves of the 640-byte rows.
template <bool kF8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<kF8>::kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap rope_map,
                  const DecodeArgs a) {
  using L = Layout<kF8>;
  constexpr int kStages = L::kStages, kStageBytes = L::kStageBytes, kThreads = L::kThreads;
  constexpr int kPvWarp = L::kPvWarp, kSoftWarp0 = L::kSoftWarp0, kConvWarp0 = L::kConvWarp0;
  constexpr int kOffKV = L::kOffKV, kOffX = L::kOffX, kOffOnes = L::kOffOnes;
  constexpr int kAlignedBytes = L::kAlignedBytes, kSmemBytes = L::kSmemBytes;
  constexpr int B_KV_FULL = L::B_KV_FULL, B_KV_EMPTY = L::B_KV_EMPTY, B_S_FULL0 = L::B_S_FULL0,
                B_S_FULL1 = L::B_S_FULL1, B_S_FREE = L::B_S_FREE, B_P_FULL = L::B_P_FULL,
                B_O_DONE0 = L::B_O_DONE0, B_O_DONE1 = L::B_O_DONE1, B_Q_READY = L::B_Q_READY,
                B_O_FREE = L::B_O_FREE, B_X_FULL0 = L::B_X_FULL0, B_DRAIN = L::B_DRAIN, B_DRAIN_PV = L::B_DRAIN_PV,
                B_F8_FULL = L::B_F8_FULL;
  constexpr uint32_t kIdescQK = Idesc<kF8>::kQK, kIdescPV = Idesc<kF8>::kPV, kIdescSum = Idesc<kF8>::kSum;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t bars = raw + kSmallBar;
  const uint32_t pair = raw + kSmallPair;  // uint2 slots, accessed with volatile ld/st
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem_raw + kSmallMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + kSmallMisc + 8);
  int32_t* seg_range = reinterpret_cast<int32_t*>(smem_raw + kSmallMisc + 16);
  uint32_t* push_cnt = reinterpret_cast<uint32_t*>(smem_raw + kSmallMisc + kMiscPush);
  volatile uint32_t* peer_push = reinterpret_cast<volatile uint32_t*>(smem_raw + kSmallMisc + kMiscPeerPush);
  volatile int32_t* aborts = reinterpret_cast<volatile int32_t*>(smem_raw + kSmallMisc + kMiscAborts);
  int32_t* armed = reinterpret_cast<int32_t*>(smem_raw + kSmallMisc + kMiscArmed);
  volatile int32_t* qk_issued = reinterpret_cast<volatile int32_t*>(smem_raw + kSmallMisc + kMiscQkIssued);
  const uint32_t base = (raw + kSmallBytes + 1023u) & ~1023u;
  const bool layout_fits = base + kAlignedBytes <= raw + kSmemBytes;
#define BAR(i) (bars + 8u * (uint32_t)(i))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cid = blockIdx.x >> 1;
  int32_t* err = a.dev_err;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(BAR(B_KV_FULL + i), kF8 ? kConvWarps : 1);  // FP8: one arrival per converter warp
      mbar_init(BAR(B_KV_EMPTY + i), 1);
      if (kF8) mbar_init(BAR(B_F8_FULL + i), 1);
    }
    mbar_init(BAR(B_S_FULL0), 1);
    mbar_init(BAR(B_S_FULL1), 1);
    mbar_init(BAR(B_S_FREE), kTileThreads / 32);  // one arrival per warp
    mbar_init(BAR(B_P_FULL), kTileThreads / 32);
    mbar_init(BAR(B_O_DONE0), 1);
    mbar_init(BAR(B_O_DONE1), 1);
    mbar_init(BAR(B_Q_READY), kTileThreads);
    mbar_init(BAR(B_O_FREE), kTileThreads);
    for (int i = 0; i < kXBufs; ++i) {
      mbar_init(BAR(B_X_FULL0 + i), 1);
      armed[i] = -1;
    }
    for (int i = 0; i < kSWarps; ++i) {
      push_cnt[i] = 0u;
      peer_push[i] = 0u;
    }
    aborts[0] = aborts[1] = 0;
    *qk_issued = -1;
    mbar_init(BAR(B_DRAIN), 1);
    mbar_init(BAR(B_DRAIN_PV), 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 64) {
    // Validate this cluster's plan range; an inconsistent plan (or a shared
    // memory window that cannot hold the aligned layout) is skipped whole, by
    // every role alike, and reported instead of being dereferenced.
    int32_t sb = a.seg_off[cid], se = a.seg_off[cid + 1];
    bool good = layout_fits && sb >= 0 && se >= sb && se <= a.num_segments;
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
  // Row-max slots start with an impossible tile tag; the ones tile feeds the
  // row-sum MMA (written by the generic proxy, read by the tensor core).
  for (int i = threadIdx.x; i < 4 * kH; i += kThreads) st_shared_v2_volatile(pair + 8u * i, 0u, 0xFFFFFFFFu);
  if (layout_fits) {
    uint32_t* ones = reinterpret_cast<uint32_t*>(smem_raw + (base - raw) + kOffOnes);
    const uint32_t one2 = kF8 ? 0x3C003C00u : 0x3F803F80u;  // f16 / bf16 1.0 pairs
    for (int i = threadIdx.x; i < kOnesBytes / 4; i += kThreads) ones[i] = one2;
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&kv_map);
    prefetch_tmap(&rope_map);
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any copy or arrive reaches them
  const uint32_t tmem = *tmem_slot;

  const int s_begin = seg_range[0];
  const int s_end = seg_range[1];

  // Each role is a lambda so that the FP8 layout can give each warpgroup its
  // register budget at the top of a branch that reaches only its own roles.
  auto role_producer = [&]() {
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
          int32_t pid = __ldg(bt + pg);  // in flight while the stage drains
          if (pg == pe - 1 && s + 1 < s_end) {
            // The next segment's query row is read right after this segment's
            // last QK^T: warm L2 with it (each CTA one half of q_abs[row],
            // CTA 0 also q_r[row]) so that load is not a DRAM round trip.
            const size_t qrow = (size_t)a.segs[8 * (s + 1)];
            const uint8_t* qa = reinterpret_cast<const uint8_t*>(a.q_abs) + qrow * (kH * kDC * 2);
            prefetch_l2_bulk(qa + rank * (kH * kDC), kH * kDC);
            if (rank == 0) prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(a.q_r) + qrow * (kH * kDR * 2), kH * kDR * 2);
          }
          if (use > 0 && !wait_phase<false, kIssueSuspend>(BAR(B_KV_EMPTY + st), (use - 1) & 1u, err, abort_flag, a.wait_limit, a.wait_every)) {
            ok = false;
            break;
          }
          if (pid < 0 || (int64_t)pid >= a.num_pages) {
            atomicOr(err, (int32_t)MLA_DEVERR_PAGE_OOB);
            pid = 0;
          }
          const uint32_t dst = base + kOffKV + st * kStageBytes;
          if constexpr (kF8) {
            // this CTA's 256 codes of each of the page's 64 rows, its RoPE
            // half, and the page's 64 token scales
            mbar_arrive_expect_tx(BAR(B_F8_FULL + st), (uint32_t)kF8Payload);
            tma_load_2d(dst, &kv_map, (int)(256 * rank), pid * kPage, BAR(B_F8_FULL + st));
            tma_load_2d(dst + kF8RopeOff, &rope_map, 256 + (int)rank * kRopeHalf, pid * kPage, BAR(B_F8_FULL + st));
            bulk_load_g2s(dst + kF8ScaleOff, a.kv_scales + (size_t)pid * kPage, kPage * 4, BAR(B_F8_FULL + st));
          } else {
            mbar_arrive_expect_tx(BAR(B_KV_FULL + st), (uint32_t)kStageBytes);
            // latent chunks 4r..4r+3 in one 3D box, then the RoPE half
            tma_load_3d(dst, &kv_map, 0, pid * kPage, (int)(4 * rank), BAR(B_KV_FULL + st));
            tma_load_2d(dst + 4 * kChunkBytes, &rope_map, kDC + (int)rank * kRopeHalf, pid * kPage,
                        BAR(B_KV_FULL + st));
          }
          ++g;
        }
      }
      // Loads still in flight must land before this CTA may exit.
      for (uint32_t k = (g > (uint32_t)kStages ? g - kStages : 0u); k < g; ++k)
        wait_phase_drain(BAR((kF8 ? B_F8_FULL : B_KV_FULL) + k % kStages), (k / kStages) & 1u);
    }
    __syncwarp();
  };
  auto role_qk = [&]() {
    // ---------------------------------------------------------------- QK^T issue
    // S_partial(t) = Q_r · K_r(t)^T as soon as page t has landed and the
    // softmax has read S(t-1).  P·V is issued by its own warp, so a long
    // QK^T issue (the tensor pipe throttles it) never delays P·V, nor the
    // other way round; the two streams share only the tensor pipe.
    if (lane == 0) {
      TileCursor cq;
      cq.init(a.segs, s_begin, s_end);
      // Stage-0 descriptors: latent chunks (K-major) and the RoPE half,
      // advanced by adding the byte offset >> 4 to the start-address field
      // (no carry: shared addresses stay below 2^18).
      const uint64_t kdesc0 = sdesc_sw128(base + kOffKV, 16, 1024);
      const uint64_t rdesc0 = sdesc_sw64(base + kOffKV + 4 * kChunkBytes, 16, 512);
      for (uint32_t tq = 0; cq.valid(); ++tq) {
        const uint32_t st = tq % kStages;
        if (!wait_phase<false, kIssueSuspend>(BAR(B_KV_FULL + st), (tq / kStages) & 1u, err, abort_flag, a.wait_limit, a.wait_every)) break;
        // FP8: the RoPE half came with the codes (already complete; waited for its TMA visibility)
        if (kF8 && !wait_phase<false, kIssueSuspend>(BAR(B_F8_FULL + st), (tq / kStages) & 1u, err, abort_flag, a.wait_limit, a.wait_every))
          break;
        if (tq > 0 && !wait_phase<false, kIssueSuspend>(BAR(B_S_FREE), (tq - 1) & 1u, err, abort_flag, a.wait_limit, a.wait_every)) break;
        if (cq.first() &&
            !wait_phase<false, kIssueSuspend>(BAR(B_Q_READY), (uint32_t)(cq.s - s_begin) & 1u, err, abort_flag, a.wait_limit, a.wait_every))
          break;
        tc_fence_after();
        // [128 x 64] += Q_r[128 x 288] · K_r^T, K-major, 16 per step: 4 latent
        // chunks (128-byte swizzle) then the RoPE half (64-byte swizzle).
        const uint64_t dk = kdesc0 + (uint64_t)((st * kStageBytes) >> 4);
        const uint64_t dr = rdesc0 + (uint64_t)((st * kStageBytes) >> 4);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + kColS, tmem + kColQ + i * 32 + kk * 8, dk + (uint64_t)((i * kChunkBytes + kk * 32) >> 4),
                   kIdescQK, (i | kk) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          mma_ts(tmem + kColS, tmem + kColQ + 128 + kk * 8, dr + (uint64_t)((kk * 32) >> 4), kIdescQK, 1u);
        tc_commit(BAR(B_S_FULL0 + (tq & 1u)));
        if (kF8) *qk_issued = (int32_t)tq;
        cq.next();
      }
      // Every MMA of this thread must be finished before TMEM is released.
      tc_commit(BAR(B_DRAIN));
      wait_phase_drain(BAR(B_DRAIN), 0);
    }
    __syncwarp();
  };
  auto role_pv = [&]() {
    // ---------------------------------------------------------------- P·V issue
    if (lane == 0) {
      TileCursor cp;
      cp.init(a.segs, s_begin, s_end);
      // The latent chunks read MN-major for P·V, and the ones tile.
      const uint64_t vdesc0 = sdesc_sw128(base + kOffKV, 8192, 1024);
      const uint64_t odesc0 = sdesc_sw128(base + kOffOnes, 16, 1024);
      uint32_t G = 0;  // tiles of this cluster
      for (int s = s_begin; s < s_end; ++s) G += (uint32_t)(a.segs[8 * s + 3] - a.segs[8 * s + 2]);
      for (uint32_t tp = 0; cp.valid(); ++tp) {
        const bool first = cp.first();
        if (!wait_phase<false, kIssueSuspend>(BAR(B_P_FULL), tp & 1u, err, abort_flag, a.wait_limit, a.wait_every)) break;
        if (first && !wait_phase<false, kIssueSuspend>(BAR(B_O_FREE), (uint32_t)(cp.s - s_begin) & 1u, err, abort_flag, a.wait_limit, a.wait_every))
          break;
        // FP8: QK^T goes first in the tensor pipe, P·V(tp) being issued only
        // after every MMA of QK^T(tp+2) is (QK^T(tp+2) needs nothing P·V(tp)
        // produces); measured 2-4 % faster for FP8 and 10 % slower for bf16.
        if (kF8 && tp + 2 < G && *qk_issued < (int32_t)(tp + 2)) {
          const uint64_t t0 = cycles();
          bool gave_up = false;
          for (uint32_t it = 1; *qk_issued < (int32_t)(tp + 2); ++it) {
            if ((it & a.wait_every) == 0u && (*abort_flag || cycles() - t0 > a.wait_limit)) {
              if (!*abort_flag) atomicOr(err, (int32_t)MLA_DEVERR_TIMEOUT);
              *abort_flag = 1;
              gave_up = true;
              break;
            }
          }
          if (gave_up) break;
        }
        tc_fence_after();
        // O_r[128 x 256] += P[128 x 64] · V_r[64 x 256]; V_r is MN-major: 4 atoms
        // of 64 columns 8 KB apart (LBO), 8-token row groups 1 KB apart (SBO).
        // l[128 x 16] += P · 1 (every column holds the row sum of P), issued
        // interleaved so consecutive MMAs never share an accumulator.
        const uint64_t dv = vdesc0 + (uint64_t)(((tp % kStages) * kStageBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t acc = (first && kk == 0) ? 0u : 1u;
          mma_ts(tmem + kColO, tmem + kColP + kk * 8, dv + (uint64_t)((kk * 2048) >> 4), kIdescPV, acc);
          mma_ts(tmem + kColSum, tmem + kColP + kk * 8, odesc0 + (uint64_t)((kk * 32) >> 4), kIdescSum, acc);
        }
        // QK^T(tp) is complete (its scores were read before P(tp) existed), so
        // this commit frees the page stage once P·V(tp) has read it.
        tc_commit(BAR(B_KV_EMPTY + tp % kStages));
        tc_commit(BAR(B_O_DONE0 + (tp & 1u)));
        cp.next();
      }
      tc_commit(BAR(B_DRAIN_PV));
      wait_phase_drain(BAR(B_DRAIN_PV), 0);
    }
    __syncwarp();
  };
  auto role_convert = [&]() {
    // ---------------------------------------------------------------- FP8 converters
    // Tile t, stage t mod kStages.  Warp cw takes token rows cw, cw+4, ...;
    // lane l the row's output chunk l (latent dims 8l..8l+7 of this CTA's
    // half): 8 codes in, one 16-byte f16 chunk out, written in the 128-byte
    // swizzled layout the tensor core reads.  The f16 rows overwrite the
    // codes, so every converter thread reads all of its codes first and the
    // four warps meet at a named barrier before the first store.  A warp that
    // leaves the loop (a wait gave up, or the CTA's abort flag is up) first
    // arrives at that tile's barrier without waiting, so every warp counts
    // exactly once for every tile any warp syncs on: the barrier always
    // completes.  A warp leaves at its wait only after the abort flag was
    // raised (by its own timeout or another's), and a warp that passed an
    // earlier tile's barrier sees the flag at the next check.
    const int cw = warp - kConvWarp0;
    uint32_t G = 0;
    for (int s = s_begin; s < s_end; ++s) G += (uint32_t)(a.segs[8 * s + 3] - a.segs[8 * s + 2]);
    const uint32_t ct = (uint32_t)lane >> 3, cc = (uint32_t)lane & 7u;
    constexpr int kRows = kPage / kConvWarps;
    constexpr int kBatch = 4;
    for (uint32_t t = 0; t < G; ++t) {
      const uint32_t st = t % kStages;
      const bool w = wait_phase<false, true>(BAR(B_F8_FULL + st), (t / kStages) & 1u, err, abort_flag, a.wait_limit, a.wait_every);
      if (!__all_sync(0xffffffffu, w)) {
        named_bar_arrive(kConvBarrier, kConvWarps * 32);
        break;
      }
      const uint32_t stage = base + kOffKV + st * kStageBytes;
      // All loads first (codes and row scales into registers), so that the
      // store loop holds no shared-memory load behind a store and its rows'
      // arithmetic overlaps.
      // f16 operands: one conversion (exact) and one multiply by the row's
      // 2^k per pair, issued kBatch rows at a time so that one warp keeps
      // many in flight.  A scale outside [2^-15, 2^7] is clamped and flagged.
      // A row's factor is formed as soon as its scale is read, so the scales
      // themselves are never all live at once.
      uint2 code[kRows];
      uint32_t fac[kRows];
      bool in_range = true;
#pragma unroll
      for (int j = 0; j < kRows; ++j) {
        const uint32_t r = (uint32_t)(kConvWarps * j + cw);
        code[j] = ld_shared_v2(stage + r * 256u + (uint32_t)lane * 8u);
        bool ok_j;
        fac[j] = fp8_f16_factor(ld_shared_f32(stage + kF8ScaleOff + 4u * r), ok_j);
        in_range = in_range && ok_j;
      }
      if (!in_range && lane == 0) atomicOr(err, (int32_t)MLA_DEVERR_FP8_RANGE);  // warp-uniform
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        named_bar_arrive(kConvBarrier, kConvWarps * 32);
        break;
      }
      named_bar_sync(kConvBarrier, kConvWarps * 32);
#pragma unroll
      for (int j0 = 0; j0 < kRows; j0 += kBatch) {
        uint32_t h[kBatch][4];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          h[j][0] = e4m3x2_to_f16x2(code[j0 + j].x & 0xFFFFu);
          h[j][1] = e4m3x2_to_f16x2(code[j0 + j].x >> 16);
          h[j][2] = e4m3x2_to_f16x2(code[j0 + j].y & 0xFFFFu);
          h[j][3] = e4m3x2_to_f16x2(code[j0 + j].y >> 16);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) h[j][q] = mul_f16x2(h[j][q], fac[j0 + j]);
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const uint32_t r = (uint32_t)(kConvWarps * (j0 + j) + cw);
          st_shared_v4(stage + ct * kChunkBytes + r * 128u + ((cc ^ (r & 7u)) << 4), h[j][0], h[j][1], h[j][2],
                       h[j][3]);
        }
      }
      // the RoPE half (bf16 from the cache) becomes f16 in place: 256 16-byte
      // chunks, two per thread; an element keeps its place in the swizzled layout
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t at = stage + kF8RopeOff + (uint32_t)(k * 128 + cw * 32 + lane) * 16u;
        const float4 v = ld_shared_v4(at);
        st_shared_v4(at, bf16x2_to_f16x2(__float_as_uint(v.x)), bf16x2_to_f16x2(__float_as_uint(v.y)),
                     bf16x2_to_f16x2(__float_as_uint(v.z)), bf16x2_to_f16x2(__float_as_uint(v.w)));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_KV_FULL + st));
    }
    __syncwarp();
  };
  auto role_softmax = [&]() {
    // ---------------------------------------------------------------- softmax + epilogue
    // Warpgroup wg (warps 2-5 and 6-9; FP8: 4-7 and 8-11) takes the tiles g with g % 2 == wg, whole:
    // thread = head row = TMEM lane, all 64 tokens.  The only hand-off between
    // the warpgroups is the row's reference max, passed from tile g-1 to g.
    const int sw = warp - kSoftWarp0;        // 0 .. kSWarps-1
    const int wg = sw >> 2;
    const int q4 = warp & 3;                 // TMEM lane quarter this warp may access
    const int h = q4 * 32 + lane;            // head row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t swz = (uint32_t)(h & 7);  // 128-byte rows: 16-byte chunk k sits at k ^ (h & 7)
    const uint32_t row_off = (uint32_t)(h * kXRow);
    const uint32_t warp_off = (uint32_t)(q4 * kXWarp);
    const bool wg_leader = ((sw & 3) == 0 && lane == 0);
    // Scores cross the pair and are compared unscaled; the scale (times
    // log2 e) enters once, in the exponent.
    const float c2 = a.scale_log2;
    const float rescale_thr = 8.f / c2;  // lazy-rescale threshold: 8 in log2 units
    const __half2 c2h = __float2half2_rn(c2);
    __syncwarp();

    // Q_r of a segment's row into TMEM, this thread's row (144 columns), in
    // two rounds of loads so that at most 20 16-byte values are live.
    auto load_q = [&](int s) {
      const int row = a.segs[8 * s];
      const uint4* lat = reinterpret_cast<const uint4*>(a.q_abs + ((size_t)row * kH + h) * kDC + rank * 256);
      const uint4* rp = reinterpret_cast<const uint4*>(a.q_r + ((size_t)row * kH + h) * kDR + rank * kRopeHalf);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint4 v[20];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __ldg(lat + half * 16 + j);
        if (half == 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j) v[16 + j] = __ldg(rp + j);
        }
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) {
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            r[4 * j] = v[ci * 8 + j].x;
            r[4 * j + 1] = v[ci * 8 + j].y;
            r[4 * j + 2] = v[ci * 8 + j].z;
            r[4 * j + 3] = v[ci * 8 + j].w;
          }
          if constexpr (kF8) {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = bf16x2_to_f16x2(r[j]);
          }
          tmem_st32(tl + kColQ + half * 64 + ci * 32, r);
        }
        if (half == 0) {
          uint32_t r[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            r[4 * j] = v[16 + j].x;
            r[4 * j + 1] = v[16 + j].y;
            r[4 * j + 2] = v[16 + j].z;
            r[4 * j + 3] = v[16 + j].w;
          }
          if constexpr (kF8) {
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = bf16x2_to_f16x2(r[j]);
          }
          tmem_st16(tl + kColQ + 128, r);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(BAR(B_Q_READY));
    };

    // Read this row's 64 partial scores of tile t, free S, push the fp16
    // partial to the peer, and load the next segment's Q if tile
    // t ends a segment (its QK^T was the segment's last).  `own` keeps the
    // rounded values.
    auto fetch_push = [&](uint32_t t, const TileCursor& c, uint32_t (&own)[kWords]) -> bool {
      bool w = wait_phase<false, true>(BAR(B_S_FULL0 + (t & 1u)), (t >> 1) & 1u, err, abort_flag, a.wait_limit, a.wait_every);
      if (!__all_sync(0xffffffffu, w)) return false;
      tc_fence_after();
      {
        uint32_t r[64];
        tmem_ld64_sync(tl + kColS, r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_S_FREE));
#pragma unroll
        for (int j = 0; j < kWords; ++j)
          own[j] = cvt_f16x2_satfinite(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
      }
      // Stage in own buffer (t + kXLead) mod kXBufs and push into the peer's
      // buffer t mod kXBufs.  Both need the peer's tile t - kXLead to have
      // landed here; this warpgroup already waited for exactly that (with
      // cluster acquire) when it finished tile t - kXLead, its previous tile
      // but one, so no wait is needed here.
      static_assert(kXLead == 2, "tile t - kXLead must be this warpgroup's, already finished");
      const uint32_t stage = base + kOffX + ((t + kXLead) % kXBufs) * kXBytes;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        st_shared_v4(stage + row_off + (((uint32_t)k ^ swz) << 4), own[4 * k], own[4 * k + 1], own[4 * k + 2],
                     own[4 * k + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        bulk_copy_to_peer(mapa(base + kOffX + (t % kXBufs) * kXBytes + warp_off, peer), stage + warp_off,
                          (uint32_t)kXWarp, mapa(BAR(B_X_FULL0 + t % kXBufs), peer));
        push_cnt[sw] += 1u;  // copies this warp issued into the peer
      }
      if (c.last() && c.s + 1 < c.s_end) load_q(c.s + 1);
      return true;
    };

    // tile count of this cluster
    uint32_t G = 0;
    for (int s = s_begin; s < s_end; ++s) G += (uint32_t)(a.segs[8 * s + 3] - a.segs[8 * s + 2]);

    if (wg == 0) mbar_arrive(BAR(B_O_FREE));  // O is free for the first segment
    if (sw == 0 && lane == 0)                  // arm the ring: the first kXBufs tiles each expect one peer push
      for (uint32_t t = 0; t < G && t < (uint32_t)kXBufs; ++t) {
        mbar_arrive_expect_tx(BAR(B_X_FULL0 + t), (uint32_t)kXBytes);
        armed[t] = (int32_t)t;
      }
    TileCursor cf;  // this warpgroup's tile
    cf.init(a.segs, s_begin, s_end);
    if (wg == 1 && cf.valid()) cf.next();
    if (wg == 0 && G > 0) load_q(s_begin);
    uint32_t own[kWords];
    bool ok = true;
    for (uint32_t g = (uint32_t)wg; g < G && ok; g += 2) {
      if (!fetch_push(g, cf, own)) {
        ok = false;
        break;
      }
      // ---- add the peer's half (fp16, unscaled)
      const uint32_t xb = g % kXBufs;
      bool w = wait_phase<true, true>(BAR(B_X_FULL0 + xb), (g / kXBufs) & 1u, err, abort_flag, a.wait_limit, a.wait_every);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      // Re-arm this buffer's barrier for tile g + kXBufs (this warpgroup's
      // again).  That push cannot land before this warpgroup has pushed tile
      // g + kXBufs - kXLead, which it does only after finishing tile g.
      if (wg_leader && g + kXBufs < G) {
        mbar_arrive_expect_tx(BAR(B_X_FULL0 + xb), (uint32_t)kXBytes);
        armed[xb] = (int32_t)(g + kXBufs);
      }
      const uint32_t recv = base + kOffX + xb * kXBytes + row_off;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 v = ld_shared_v4(recv + (((uint32_t)k ^ swz) << 4));
        own[4 * k] = as_u32(__hadd2(as_h2(own[4 * k]), as_h2(__float_as_uint(v.x))));
        own[4 * k + 1] = as_u32(__hadd2(as_h2(own[4 * k + 1]), as_h2(__float_as_uint(v.y))));
        own[4 * k + 2] = as_u32(__hadd2(as_h2(own[4 * k + 2]), as_h2(__float_as_uint(v.z))));
        own[4 * k + 3] = as_u32(__hadd2(as_h2(own[4 * k + 3]), as_h2(__float_as_uint(v.w))));
      }

      // ---- causal/length mask and the row max of this tile
      const int valid = cf.vis - cf.pg * kPage;
      if (valid < kPage) {
#pragma unroll
        for (int j = 0; j < kWords; ++j) {
          if (2 * j >= valid) own[j] = (own[j] & 0xFFFF0000u) | 0xFC00u;          // low half -> -inf
          if (2 * j + 1 >= valid) own[j] = (own[j] & 0x0000FFFFu) | 0xFC000000u;  // high half -> -inf
        }
      }
      __half2 mx[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        mx[j] = __hmax2(__hmax2(as_h2(own[4 * j]), as_h2(own[4 * j + 1])), __hmax2(as_h2(own[4 * j + 2]), as_h2(own[4 * j + 3])));
      const __half2 mh = __hmax2(__hmax2(__hmax2(mx[0], mx[1]), __hmax2(mx[2], mx[3])),
                                 __hmax2(__hmax2(mx[4], mx[5]), __hmax2(mx[6], mx[7])));
      const float mt = fmaxf(__low2float(mh), __high2float(mh));

      // ---- reference max: tile g-1's (the other warpgroup's) unless this tile starts a segment
      const uint32_t gp = g - 1;  // the previous tile (the other warpgroup's)
      const bool od_ready = (g == 0) || mbar_test_wait(BAR(B_O_DONE0 + (gp & 1u)), (gp >> 1) & 1u);
      float m = mt, factor = 1.f;
      bool resc = false;
      if (!cf.first()) {
        const uint32_t slot = pair + 8u * (((g - 1) & 3u) * kH + h);
        uint2 v = ld_shared_v2_volatile(slot);
        if (v.y != g - 1) {
          const uint64_t t0 = cycles();
          for (uint32_t it = 1; (v = ld_shared_v2_volatile(slot)).y != g - 1; ++it) {
            if ((it & a.wait_every) == 0u && (*abort_flag || cycles() - t0 > a.wait_limit)) {
              if (!*abort_flag) atomicOr(err, (int32_t)MLA_DEVERR_TIMEOUT);
              *abort_flag = 1;
              break;
            }
          }
        }
        if (!__all_sync(0xffffffffu, v.y == g - 1)) {
          ok = false;
          break;
        }
        const float mp = __uint_as_float(v.x);
        if (mt > mp + rescale_thr) {  // lazy rescale: move the reference only on a large jump
          factor = exp2f((mp - mt) * c2);
          resc = true;
        } else {
          m = mp;
        }
      }
      // Hand m to tile g+1.  Four slots: the next writer of this one is tile
      // g+4, and the next writer of tile g-1's is tile g+3, which needs S
      // freed by tile g+2, fetched by this warpgroup only after this read;
      // two slots would not do, since a tile that starts a segment reads none
      // and may run ahead.
      st_shared_v2_volatile(pair + 8u * ((g & 3u) * kH + h), __float_as_uint(m), g);

      // ---- P = 2^(c2 (s - m)) in fp16 pairs (one fused multiply-add for the
      //      exponent), stored as bf16 for the tensor core (the FP8 cache's
      //      f16 operands take the fp16 P as it is)
      const __half2 mc2 = __float2half2_rn(-m * c2);
#pragma unroll
      for (int j = 0; j < kWords; ++j) {
        const uint32_t p16 = ex2_f16x2(as_u32(__hfma2(as_h2(own[j]), c2h, mc2)));
        if constexpr (kF8) {
          own[j] = p16;
        } else {
          const float2 p = __half22float2(as_h2(p16));
          own[j] = pack_bf16x2(p.x, p.y);
        }
      }
      // Writing P (single TMEM buffer) and a rescale both need P·V of tile g-1 done.
      if (g > 0) {
        w = od_ready || wait_phase<false, true>(BAR(B_O_DONE0 + (gp & 1u)), (gp >> 1) & 1u, err, abort_flag, a.wait_limit, a.wait_every);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          uint32_t o[32];
          tmem_ld32_sync(tl + kColO + c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * factor);
          tmem_st32(tl + kColO + c, o);
        }
        tmem_st1(tl + kColSum, __float_as_uint(__uint_as_float(tmem_ld1_sync(tl + kColSum)) * factor));
      }
      tmem_st32(tl + kColP, own);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_P_FULL));

      if (cf.last()) {
        // ---- epilogue of this segment: wait for its last P·V, normalise, store
        const int row = cf.row, slot = cf.slot;
        w = wait_phase(BAR(B_O_DONE0 + (g & 1u)), (g >> 1) & 1u, err, abort_flag, a.wait_limit, a.wait_every);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float lt = __uint_as_float(tmem_ld1_sync(tl + kColSum));
        const float inv = 1.f / lt;
        if (slot < 0) {
          uint4* dst = reinterpret_cast<uint4*>(a.o_lat + ((size_t)row * kH + h) * kDC + rank * 256);
#pragma unroll 1
          for (int c = 0; c < 256; c += 32) {
            uint32_t o[32];
            tmem_ld32_sync(tl + kColO + c, o);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c / 8 + v] = make_uint4(
                  pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv),
                  pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv),
                  pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv),
                  pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv));
          }
        } else {
          // Partials are read once, by the combine right after this kernel: kept
          // in L2 with evict-last priority through the rest of the KV stream.
          float4* dst = reinterpret_cast<float4*>(a.part_o + ((size_t)slot * kH + h) * kDC + rank * 256);
          const uint64_t keep = l2_policy_evict_last();
#pragma unroll 1
          for (int c = 0; c < 256; c += 32) {
            uint32_t o[32];
            tmem_ld32_sync(tl + kColO + c, o);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              st_global_v4_hint(dst + c / 4 + v,
                                make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                            __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv),
                                keep);
          }
        }
        tc_fence_before();
        mbar_arrive(BAR(B_O_FREE));
        if (rank == 0) {
          const float lse2 = m * c2 + log2f(lt);
          if (slot < 0) {
            if (a.lse) a.lse[(size_t)row * kH + h] = lse2 * 0.6931471805599453f;
          } else {
            a.part_lse[(size_t)slot * kH + h] = lse2;
          }
        }
      }
      cf.next();
      cf.next();
    }
  };
  if constexpr (kF8) {
    // 512 threads x 128 registers at launch: warpgroup 0 (producer, MMA
    // issue, an idle warp) drops to 64, warpgroup 3 (converters, which hold
    // a tile's codes and row factors in registers) to 112, the softmax
    // warpgroups 1-2 rise to 168; 128*64 + 128*112 + 256*168 = 65536, the
    // launch's total.  (96 for the converters spilled their codes.)
    if (warp < 4) {
      regs_dec<64>();
      if (warp == 0) role_producer();
      else if (warp == 1) role_qk();
      else if (warp == kPvWarp) role_pv();
    } else if (warp >= kConvWarp0) {
      regs_dec<112>();
      role_convert();
    } else {
      regs_inc<168>();
      role_softmax();
    }
  } else {
    if (warp == 0) role_producer();
    else if (warp == 1) role_qk();
    else if (warp == kPvWarp) role_pv();
    else role_softmax();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // Every role is done, so every score copy either CTA will ever issue has
  // been issued.  On the normal path each one was awaited by its receiver.
  // After an abort some may still be in flight: tell the peer how many copies
  // each softmax warp issued, and whether this CTA aborted.
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSWarps; ++i)
      st_cluster_u32(mapa(raw + kSmallMisc + kMiscPeerPush + 4u * i, peer), push_cnt[i]);
    const int32_t mine = *abort_flag;
    aborts[0] = mine;
    st_cluster_u32(mapa(raw + kSmallMisc + kMiscAborts + 4u, peer), (uint32_t)mine);
  }
  cluster_sync();  // neither CTA leaves while its peer may still address its shared memory
  if (aborts[0] != 0 || aborts[1] != 0) {
    // Drain: each exchange buffer has at most one armed phase this CTA did not
    // see complete.  The peer's counts say how many of that tile's four
    // per-warp copies it issued; the bytes of the copies never issued are
    // retired by hand, and the phase then completes once the issued ones land.
    if (threadIdx.x == 0) {
      for (int b = 0; b < kXBufs; ++b) {
        const int32_t t = armed[b];
        if (t < 0) continue;
        const uint32_t par = ((uint32_t)t / kXBufs) & 1u;
        if (mbar_test_wait_cluster(BAR(B_X_FULL0 + b), par)) continue;
        const uint32_t idx = (uint32_t)t >> 1, pg = (uint32_t)t & 1u;
        uint32_t issued = 0;
        for (int q = 0; q < 4; ++q) issued += peer_push[pg * 4 + q] > idx ? 1u : 0u;
        if (issued < 4) mbar_complete_tx(BAR(B_X_FULL0 + b), (4u - issued) * (uint32_t)kXWarp);
        const uint64_t t0 = cycles();
        while (!mbar_test_wait_cluster(BAR(B_X_FULL0 + b), par) && cycles() - t0 < kWaitLimitCycles) {
        }
      }
    }
    // and neither CTA leaves while a copy out of its shared memory may still be reading it
    cluster_sync();
  }
#undef BAR
}

// Merge split rows: lse = log2 Σ 2^{lse_s} (log2 domain), o = Σ 2^{lse_s - lse} o_s.
}  // namespace decode

int decode_smem_bytes() { return decode::Layout<false>::kSmemBytes; }
int decode_threads() { return decode::Layout<false>::kThreads; }

template <bool kF8>
static cudaError_t decode_prepare() {
  return cudaFuncSetAttribute(decode::decode_kernel<kF8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              decode::Layout<kF8>::kSmemBytes);
}

cudaError_t decode_max_clusters(int* out) {
  cudaError_t e = decode_prepare<false>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(decode::Layout<false>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = decode::Layout<false>::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, (const void*)decode::decode_kernel<false>, &cfg);
}

cudaError_t launch_decode(const CUtensorMap& kv_map, const CUtensorMap& rope_map, const DecodeArgs& args,
                          int num_clusters, bool fp8, cudaStream_t stream) {
  cudaError_t e = fp8 ? decode_prepare<true>() : decode_prepare<false>();
  if (e != cudaSuccess) return e;
  if (fp8)
    decode::decode_kernel<true><<<2 * num_clusters, decode::Layout<true>::kThreads, decode::Layout<true>::kSmemBytes,
                                  stream>>>(kv_map, rope_map, args);
  else
    decode::decode_kernel<false><<<2 * num_clusters, decode::Layout<false>::kThreads,
                                   decode::Layout<false>::kSmemBytes, stream>>>(kv_map, rope_map, args);
  return cudaGetLastError();
}

}  // namespace mla
