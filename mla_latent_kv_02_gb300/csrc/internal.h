// Internal interface between the C-ABI entry points (mla_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/mla.h"

namespace mla {

// Records `message` as this thread's mla_last_error() and returns `s`.
mla_status set_last_error(mla_status s, const char* message);

// Layout of the decode plan (int32 words).  Written by the host planner,
// read by the decode and combine kernels.
//   [0] magic  [1] T  [2] B  [3] num_clusters  [4] num_segments
//   [5] num_partials  [6] num_split_rows  [7] max_pages_needed
//   [8..15] reserved
//   seg_off   at kPlanHeader, num_clusters + 1 entries
//   segments  at seg_base, num_segments x 8: {row, b, page_begin, page_end,
//             visible, out_slot (-1 = final), 0, 0}
//   split rows at split_base, num_split_rows x 4: {row, slot_begin, n_slots, 0}
constexpr int kPlanHeader = 16;
constexpr int kSegWords = 8;
constexpr int kSplitWords = 4;

struct PlanLayout {
  int64_t seg_off;  // word offsets
  int64_t seg_base;
  int64_t split_base;
  int64_t words;
};
PlanLayout plan_layout(int64_t num_clusters, int64_t num_segments, int64_t num_split_rows);
// Upper bounds used to size the plan buffer.
inline int64_t plan_max_segments(int64_t T, int64_t num_clusters) { return T + num_clusters; }
inline int64_t plan_max_split_rows(int64_t T, int64_t num_clusters) {
  return T < num_clusters ? T : num_clusters;
}
inline int64_t plan_max_partials(int64_t num_clusters) { return 2 * num_clusters; }

struct DecodeArgs {
  const uint16_t* q_abs;  // bf16 [T, 128, 512]
  const uint16_t* q_r;    // bf16 [T, 128, 64]
  const int32_t* block_table;
  int32_t max_pages;
  int32_t pad_;
  int64_t num_pages;
  const int32_t* seg_off;
  const int32_t* segs;
  float scale_log2;  // scale * log2(e)
  int32_t pad2_;
  uint16_t* o_lat;     // bf16 [T, 128, 512]
  float* lse;          // [T, 128] or null
  float* part_o;       // fp32 [partials, 128, 512]
  float* part_lse;     // fp32 [partials, 128] (log2 domain)
  int32_t* dev_err;
  // plan summary, used to validate every segment before any access
  int32_t T;
  int32_t B;
  int32_t num_segments;
  int32_t num_partials;
  const float* kv_scales;  // FP8 cache: fp32 [num_pages * 64] token scales (null for bf16)
  // Bound, in SM cycles, of every wait in the decode loop (the drains before
  // exit keep the full default bound).
  uint64_t wait_limit;
  // The deadline is checked when a wait's probe count & wait_every is 0
  // (255 for the default bound; 0, every probe, for a short test bound).
  uint32_t wait_every;
  int32_t pad3_;
};

// Decompress branch over a batch of sequences: sequence i has M query rows
// at positions N - M .. N - 1; its query rows (q_c, q_r, out) start at row
// q_off, its cache rows (gathered rows, K_c, V_c) at token kv_off of the
// packed arrays.  The table rides in the launch parameters.
constexpr int kPrefillMaxSeqs = 64;
struct PrefillSeq {
  int32_t M;
  int32_t N;
  int32_t q_off;
  int32_t kv_off;
};
struct PrefillArgs {
  int32_t nb;           // sequences in seq[]
  float scale_log2;     // scale * log2(e)
  uint16_t* out;        // bf16 [rows, 128, 128]
  int32_t* dev_err;
  PrefillSeq seq[kPrefillMaxSeqs];
};

// Gather of the first n[i] cached tokens of sequence b[i] of the block
// table, for i < nb, to rows [off[i], off[i] + n[i]) of one packed output.
struct GatherBatch {
  int32_t nb;
  int32_t pad_;
  int64_t total;        // Σ n[i]
  int32_t b[kPrefillMaxSeqs];
  int32_t n[kPrefillMaxSeqs];
  int64_t off[kPrefillMaxSeqs];
};

struct CombineArgs {
  const int32_t* split_rows;
  const float* part_o;
  const float* part_lse;
  uint16_t* o_lat;
  float* lse;
  int32_t T;
  int32_t num_partials;
  int32_t* dev_err;
};

int decode_smem_bytes();
int decode_threads();
cudaError_t decode_max_clusters(int* out);
// bf16 cache: kv_map 128-byte swizzled boxes of 64 columns x 64 tokens x 4
// chunks (latent), rope_map 64-byte swizzled boxes of 32 columns x 64 tokens.
// FP8 cache (fp8 = true): kv_map uint8 boxes of 256 codes x 64 tokens (no
// swizzle), rope_map as above over the 640-byte rows; args.kv_scales set.
cudaError_t launch_decode(const CUtensorMap& kv_map, const CUtensorMap& rope_map, const DecodeArgs& args,
                          int num_clusters, bool fp8, cudaStream_t stream);
cudaError_t launch_combine(const CombineArgs& args, int num_split_rows, cudaStream_t stream);

cudaError_t launch_kv_append(const uint16_t* c_kv_new, const uint16_t* k_r_new, const int64_t* slots, int32_t n,
                             uint16_t* kv_cache, int64_t num_slots, int32_t* dev_err, cudaStream_t stream);
cudaError_t launch_rope_table(float* table, int32_t max_pos, double base, cudaStream_t stream);
cudaError_t launch_kv_append_rope(const uint16_t* c_kv_new, const uint16_t* k_pe_new, const int32_t* positions,
                                  const float* table, int32_t max_pos, const int64_t* slots, int32_t n,
                                  uint16_t* kv_cache, int64_t num_slots, int32_t* dev_err, cudaStream_t stream);
cudaError_t launch_rope_q(const uint16_t* q_pe, const int32_t* positions, const float* table, int32_t max_pos,
                          uint16_t* q_r, int32_t T, int32_t* dev_err, cudaStream_t stream);
cudaError_t launch_kv_append_fp8(const uint16_t* c_kv_new, const uint16_t* k_r_new, const int64_t* slots, int32_t n,
                                 uint8_t* rows, float* scales, int64_t num_slots, int32_t* dev_err,
                                 cudaStream_t stream);
cudaError_t launch_gather_fp8(const uint8_t* rows, const float* scales, int64_t num_pages,
                              const int32_t* block_table, int32_t max_pages, int32_t b, int32_t n_tokens,
                              uint16_t* out, int32_t* dev_err, cudaStream_t stream);
cudaError_t launch_kv_append_nvfp4(const uint16_t* c_kv_new, const uint16_t* k_r_new, const int64_t* slots,
                                   int32_t n, float tensor_scale, uint8_t* rows, int64_t num_slots,
                                   int32_t* dev_err, cudaStream_t stream);
cudaError_t launch_gather_nvfp4(const uint8_t* rows, float tensor_scale, int64_t num_pages,
                                const int32_t* block_table, int32_t max_pages, int32_t b, int32_t n_tokens,
                                uint16_t* out, int32_t* dev_err, cudaStream_t stream);
cudaError_t launch_gather_nvfp4_batch(const uint8_t* rows, float tensor_scale, int64_t num_pages,
                                      const int32_t* block_table, int32_t B, int32_t max_pages, const int32_t* seq_ids,
                                      const int64_t* out_offsets, int32_t nb, int64_t total_tokens, uint16_t* out,
                                      int32_t* dev_err, cudaStream_t stream);
cudaError_t launch_gather(const uint16_t* kv_cache, int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                          int32_t b, int32_t n_tokens, uint16_t* out, int32_t* dev_err, cudaStream_t stream);
cudaError_t launch_gather_batch(const uint16_t* kv_cache, int64_t num_pages, const int32_t* block_table,
                                int32_t max_pages, const GatherBatch& g, uint16_t* out, int32_t* dev_err,
                                cudaStream_t stream);

// Decompress-branch expansion: K_c and V_c in one pass (head-major outputs).
cudaError_t launch_expand_kv(const CUtensorMap& a_map, const CUtensorMap& k_map, const CUtensorMap& v_map,
                             const CUtensorMap& kc_map, const CUtensorMap& vc_map, int32_t n, int32_t* err,
                             cudaStream_t stream);
int prefill_smem_bytes();
cudaError_t launch_prefill_attn(const CUtensorMap& q_map, const CUtensorMap& r_map, const CUtensorMap& k_map,
                                const CUtensorMap& kr_map, const CUtensorMap& v_map, const PrefillArgs& args,
                                cudaStream_t stream);

// Per-head GEMM C[t, h, :] = A[t, h, :] · W[h] (bf16 in, fp32 accumulate, bf16 out).
enum class HeadGemm { kAbsorbQ, kUpV };
cudaError_t launch_head_gemm(HeadGemm kind, const CUtensorMap& a_map, const CUtensorMap& w_map,
                             const CUtensorMap& c_map, int32_t T, int32_t* err, cudaStream_t stream);

}  // namespace mla
