/*
 * mla.h — C ABI of the GB300 (sm_103a) absorbed paged MLA decode library.
 *
 * The operation is DeepSeek Multi-Head Latent Attention decode with matrix
 * absorption over a paged latent KV cache, as described by:
 *
 *   [P1] "撕开 DeepSeek MLA 源码：C++ 与 TensorRT-LLM 算子设计优化全景与 TaoToken 实践"
 *        (sheratonhq.com/news/189140): §1 the cached token (512-d latent c_KV
 *        plus 64-d decoupled RoPE key k_R, 576 bf16 elements), §3 the
 *        dimension constants and the plugin config (128 heads, content head
 *        dim 128, page_size 64, absorption on, bf16 cache), §4 the absorbed
 *        score (path B) and its scale, §5 the shared-memory and 16-byte
 *        alignment pitfalls.
 *   [P2] "DeepSeek的推理为什么比别人便宜一个数量级？——MLA、MoE、MTP技术拆解"
 *        (leslieaibin.github.io): the MLA section (K = c·W_UK, V = c·W_UV),
 *        the MTP section (two query tokens per decode step) and the closing
 *        inference-flow summary (the new latent is appended every step).
 *   [P3] bjbfmj.com/news/60700: the KV-byte formula and its calculator.
 *
 * Conventions
 *   - Every call returns an mla_status; on failure mla_last_error() gives a
 *     thread-local message.  Host-side validation runs before anything is
 *     enqueued: a failing call enqueues nothing.
 *   - Device buffers are owned by the caller.  Only the page pool (a host
 *     object) is allocated by the library; no entry point allocates or frees
 *     device memory.
 *   - bf16 tensors are passed as untyped pointers to IEEE bfloat16 values
 *     (uint16 bit patterns), row-major, contiguous, 16-byte aligned.
 *   - Device work is enqueued asynchronously on `stream` (a cudaStream_t;
 *     NULL is the legacy default stream) on the current CUDA device.
 *   - Anomalies seen on the device (a page id or slot outside the pool, an
 *     internal wait that exceeded its time limit) are OR-ed into the caller's
 *     int32 device error word `dev_err` as MLA_DEVERR_* bits; the kernel then
 *     skips or redirects the offending access instead of faulting.
 *     mla_check() reads that word.
 *   - Dimensions are fixed at the [P1] §3 constants: H = 128 heads, d_hc = 128,
 *     d_c = 512, d_r = 64, page_size = 64.  Anything else is
 *     MLA_ERR_UNSUPPORTED.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_NUM_HEADS 128
#define MLA_HEAD_DIM_C 128
#define MLA_LATENT_DIM 512
#define MLA_ROPE_DIM 64
#define MLA_PAGE_SIZE 64
#define MLA_TOKEN_ELEMS 576          /* d_c + d_r per cached token */
#define MLA_PAGE_BYTES (64 * 576 * 2) /* 73 728 B: one 64-token bf16 page */

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* null pointer, bad size or inconsistent arguments */
  MLA_ERR_MISALIGNED = 2,  /* a device pointer is not 16-byte aligned ([P1] §5) */
  MLA_ERR_UNSUPPORTED = 3, /* dimensions other than the [P1] §3 constants */
  MLA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  MLA_ERR_DEVICE = 5,      /* mla_check: the device error word is non-zero */
  MLA_ERR_TIMEOUT = 6,     /* mla_check: a kernel wait gave up (MLA_DEVERR_TIMEOUT) */
  MLA_ERR_NO_SPACE = 7     /* the page pool has fewer free pages than requested */
} mla_status;

/* Bits of the device error word. */
#define MLA_DEVERR_PAGE_OOB 1u /* block-table entry outside [0, num_pages): page 0 read instead */
#define MLA_DEVERR_SLOT_OOB 2u /* append/gather slot outside the pool: that token skipped */
#define MLA_DEVERR_TIMEOUT 4u  /* an mbarrier wait exceeded its limit; the kernel stopped early */
#define MLA_DEVERR_PLAN 8u     /* the plan buffer is not a valid decode plan */
#define MLA_DEVERR_POS_OOB 16u /* RoPE position outside [0, max_pos): that token / row skipped */
#define MLA_DEVERR_FP8_RANGE 32u /* FP8 decode: a token scale outside [2^-15, 2^7]; that row was clamped */
#define MLA_DEVERR_BATCH 64u   /* batched gather: a sequence id, offset or length out of range; those rows skipped */

/* Thread-local message of the last failing call (never NULL). */
const char* mla_last_error(void);
/* Static name of a status code. */
const char* mla_status_string(mla_status s);
/* Library ABI version (major * 100 + minor). */
int32_t mla_version(void);

/*
 * Model dimensions of [P1] §3 (mla_config.h constants and the plugin JSON),
 * plus the score scale 1/sqrt(d_hc + d_r) of [P1] §4.
 */
typedef struct mla_config {
  int32_t num_heads;  /* 128 */
  int32_t head_dim_c; /* 128 */
  int32_t latent_dim; /* 512 */
  int32_t rope_dim;   /* 64 */
  int32_t page_size;  /* 64 */
  float scale;        /* 1/sqrt(192) */
} mla_config;

mla_config mla_config_default(void);
/* MLA_OK if `cfg` holds the supported dimensions and a finite positive scale;
 * MLA_ERR_UNSUPPORTED for other dimensions; MLA_ERR_INVALID_ARG for NULL or a bad scale. */
mla_status mla_config_validate(const mla_config* cfg);

/*
 * [P3] KV-byte formula: *out = layers * (dc + dr) * elem_bytes * tokens * seqs.
 * MLA_ERR_INVALID_ARG if layers, dc, elem_bytes, tokens or seqs <= 0, dr < 0,
 * `out` is NULL, or the product overflows uint64.
 */
mla_status mla_kv_bytes(int64_t layers, int64_t dc, int64_t dr, int64_t elem_bytes,
                        int64_t tokens, int64_t seqs, uint64_t* out);

/* ---------------------------------------------------------------------------
 * Page pool and page tables (host objects).  Pages of 64 tokens, [P1] §3.
 * ------------------------------------------------------------------------- */
typedef struct mla_pool mla_pool;

/* Create a pool of page ids [0, num_pages).  num_pages >= 1. */
mla_status mla_pool_create(int32_t num_pages, mla_pool** out);
/* Take `n` free page ids (lowest first) into page_ids_out[n].  MLA_ERR_NO_SPACE
 * (nothing taken) if fewer than n are free. */
mla_status mla_pool_alloc(mla_pool* pool, int32_t n, int32_t* page_ids_out);
/* Return ids to the pool.  MLA_ERR_INVALID_ARG (nothing returned) if an id is
 * out of range, not allocated, or repeated. */
mla_status mla_pool_free(mla_pool* pool, const int32_t* ids, int32_t n);
mla_status mla_pool_available(const mla_pool* pool, int32_t* out);
void mla_pool_destroy(mla_pool* pool);

/*
 * Physical slot of token (seq_ids[i], positions[i]):
 *   slots_out[i] = block_table[b * max_pages + pos / 64] * 64 + pos % 64.
 * block_table is host int32 [batch, max_pages].  MLA_ERR_INVALID_ARG if a
 * sequence id or page index is out of range or the table entry is negative.
 */
mla_status mla_slot_mapping(const int32_t* block_table, int32_t batch, int32_t max_pages,
                            const int32_t* seq_ids, const int32_t* positions, int32_t n,
                            int64_t* slots_out);

/* ---------------------------------------------------------------------------
 * Device steps
 * ------------------------------------------------------------------------- */

/* Zero-fill the pool kv_cache [num_pages, 64, 576] bf16 (every slot must hold
 * finite values: a masked token still enters the P·V product with weight 0). */
mla_status mla_cache_init(void* kv_cache, int64_t num_pages, void* stream);

/*
 * Step A1 — append ([P2] inference-flow summary: each step's new latent joins
 * the cache; [P1] §3 page_size 64).  For i < n:
 *   kv_cache[slots[i]] = [c_kv_new[i, 0:512] | k_r_new[i, 0:64]]
 * c_kv_new bf16 [n, 512], k_r_new bf16 [n, 64], slots int64 [n] (device),
 * kv_cache bf16 [num_pages * 64, 576].  A slot outside [0, num_pages*64) sets
 * MLA_DEVERR_SLOT_OOB and that token is skipped.  n == 0 is a no-op.
 */
mla_status mla_kv_append(const void* c_kv_new, const void* k_r_new, const int64_t* slots,
                         int32_t n, void* kv_cache, int64_t num_pages, int32_t* dev_err,
                         void* stream);

/*
 * Copy the first n_tokens cached tokens of sequence b, in position order, to
 * out bf16 [n_tokens, 576] (device).  A bit-exact view of what the decode
 * kernel reads.  Bad page ids set MLA_DEVERR_PAGE_OOB and leave rows unwritten.
 */
mla_status mla_gather_paged(const void* kv_cache, int64_t num_pages, const int32_t* block_table,
                            int32_t max_pages, int32_t b, int32_t n_tokens, void* out,
                            int32_t* dev_err, void* stream);

/*
 * Step A2 — query absorption ([P1] §4 path B, einsum 'qhd,hdc->qhc'):
 *   q_abs[t, h, c] = sum_d q_c[t, h, d] * W_UK[h, d, c]
 * q_c bf16 [T, 128, 128], w_uk bf16 [128, 128, 512], q_abs bf16 [T, 128, 512];
 * fp32 accumulation, one bf16 rounding.  T == 0 is a no-op.  dev_err (device
 * int32, required) receives MLA_DEVERR_TIMEOUT if an internal wait gives up.
 */
mla_status mla_absorb_q(const void* q_c, const void* w_uk, void* q_abs, int32_t T, int32_t* dev_err,
                        void* stream);

/*
 * Step A5 — V up-projection ([P2] MLA section, V = c·W_UV, applied after the
 * attention by associativity):
 *   out[t, h, d] = sum_c o_lat[t, h, c] * W_UV[h, c, d]
 * o_lat bf16 [T, 128, 512], w_uv bf16 [128, 512, 128], out bf16 [T, 128, 128];
 * fp32 accumulation.  T == 0 is a no-op.  dev_err as for mla_absorb_q.
 */
mla_status mla_up_v(const void* o_lat, const void* w_uv, void* out, int32_t T, int32_t* dev_err,
                    void* stream);

/* ---------------------------------------------------------------------------
 * Step A3 + A4 — absorbed paged attention with split-KV and combine.
 *
 * Rows: query token i of sequence b is row t = sum_{b'<b} q_lens[b'] + i.  Its
 * sequence holds seq_lens[b] tokens (this step's q_lens[b] tokens already
 * appended), it sits at position seq_lens[b] - q_lens[b] + i and sees the
 * positions [0, that position] (causal within a multi-token query: the MTP
 * two-token decode of [P2] and chunked prefill of [P1]).
 *
 * Per row t and head h, over the visible tokens j ([P1] §4 path B):
 *   s_j   = (q_abs[t,h,:]·c_KV[j] + q_r[t,h,:]·k_R[j]) * scale
 *   o_lat[t,h,:] = sum_j softmax(s)_j c_KV[j]          (bf16 out)
 *   lse[t,h]     = ln sum_j exp(s_j)                    (fp32 out, optional)
 * ------------------------------------------------------------------------- */

/* Largest number of co-resident 2-CTA clusters the decode kernel can use on
 * the current device (the split plan's parallelism). */
mla_status mla_decode_max_clusters(int32_t* out);

/* Bytes of the plan buffer for T rows and num_clusters clusters. */
mla_status mla_decode_plan_bytes(int32_t T, int32_t num_clusters, size_t* bytes);

/* Bytes of the split-KV workspace for num_clusters clusters (fp32 partial
 * outputs and their log-sum-exp). */
mla_status mla_decode_workspace_size(int32_t num_clusters, size_t* bytes);

/* Summary of a plan, filled by the planner and passed back to mla_decode_paged. */
typedef struct mla_plan_info {
  uint32_t magic;         /* MLA_PLAN_MAGIC */
  int32_t T;              /* rows */
  int32_t B;              /* sequences */
  int32_t num_clusters;   /* clusters launched (<= requested) */
  int32_t num_segments;   /* (row, page range) work pieces */
  int32_t num_partials;   /* split pieces written to the workspace */
  int32_t num_split_rows; /* rows merged by the combine kernel */
  int32_t max_pages_needed; /* block-table columns the plan reads */
  int64_t total_tiles;    /* 64-token tiles over all rows */
  size_t plan_bytes;      /* bytes of plan data written */
} mla_plan_info;

#define MLA_PLAN_MAGIC 0x504C4D41u /* "AMLP" */

/*
 * Build the split-KV schedule on the host into plan_host (plan_bytes from
 * mla_decode_plan_bytes).  seq_lens/q_lens are host int32 [B] with
 * seq_lens[b] >= 1 and 0 <= q_lens[b] <= seq_lens[b].  Work (64-token tiles of
 * every row, in row order) is cut into equal contiguous ranges, one per
 * cluster; a row cut by a range boundary is computed in pieces and merged by
 * the combine step.
 */
mla_status mla_decode_plan_host(const int32_t* seq_lens, const int32_t* q_lens, int32_t B,
                                int32_t num_clusters, void* plan_host, size_t plan_bytes,
                                mla_plan_info* info);

/* As mla_decode_plan_host, then copies the plan to plan_dev on `stream`. */
mla_status mla_decode_plan(const int32_t* seq_lens_host, const int32_t* q_lens_host, int32_t B,
                           int32_t num_clusters, void* plan_dev, size_t plan_bytes,
                           mla_plan_info* info, void* stream);

/*
 * Run steps A3 and A4.
 *   q_abs bf16 [T, 128, 512]; q_r bf16 [T, 128, 64];
 *   kv_cache bf16 [num_pages, 64, 576]; block_table int32 [B, max_pages] (device);
 *   plan_dev / info from mla_decode_plan; workspace of ws_bytes >=
 *   mla_decode_workspace_size(info->num_clusters) (device, 16-B aligned);
 *   o_lat bf16 [T, 128, 512] out; lse fp32 [T, 128] out or NULL;
 *   dev_err int32 device word (required).
 * Every cache slot read must hold finite values (see mla_cache_init).
 */
mla_status mla_decode_paged(const void* q_abs, const void* q_r, const void* kv_cache,
                            int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                            const void* plan_dev, const mla_plan_info* info, float scale,
                            void* workspace, size_t ws_bytes, void* o_lat, float* lse,
                            int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------------------
 * Allocation-free decode (no counterpart in the source pages: it exists for
 * callers that cannot allocate device memory).
 * ------------------------------------------------------------------------- */

/* Size of the scratch that mla_decode_paged_noalloc keeps in a device array
 * of the library (plan area + split-KV workspace, 16.5 MiB in all). */
#define MLA_NOALLOC_PLAN_BYTES (512u * 1024u)
#define MLA_NOALLOC_WORKSPACE_BYTES (16u * 1024u * 1024u)

/*
 * mla_decode_paged for callers that cannot allocate device memory: a plugin
 * that its host framework hands only input and output tensors, an engine
 * whose memory pool already holds all free device memory, or a runtime that
 * forbids allocation after initialisation.  The caller passes only inputs and
 * outputs; the split plan and the split-KV workspace live in a file-scope
 * device array of the library (MLA_NOALLOC_PLAN_BYTES +
 * MLA_NOALLOC_WORKSPACE_BYTES, held on every device that loads the library
 * until the process exits).  No cudaMalloc, cudaFree or other allocating call
 * is made.
 *
 * Arguments as for mla_decode_paged, except that the sequence lengths are
 * given on the host (seq_lens_host / q_lens_host, int32 [B]) and the plan is
 * built internally.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) and the cluster count; make that first call
 * before capturing any stream.  The plan reaches the array inside the launch
 * parameters of a small copy kernel on `stream` (one launch per 7 936 plan
 * words, one for every usual batch), so the call reads no host memory after
 * it returns and never waits for the stream.
 *
 * When the plan for every cluster needs more split-KV workspace than the
 * array holds (MLA_NOALLOC_WORKSPACE_BYTES fits 63 split pieces; long
 * contexts split every row), the largest cluster count whose plan fits is
 * used, found by planning on the host from the most clusters down.  Fewer
 * clusters mean fewer SMs at work: on a GB300 (76 two-CTA clusters) a batch
 * of 16 sequences of 64K tokens runs on 48 clusters in about 1.6x the time of
 * mla_decode_paged, and a batch of 64 two-token MTP rows over 8K tokens on
 * 64 clusters (no split rows) in about 1.2x.  A batch whose plan exceeds
 * MLA_NOALLOC_PLAN_BYTES even on one cluster (about 16 000 query rows) is
 * rejected with MLA_ERR_INVALID_ARG.  Nothing in the array needs to start at
 * zero: every call writes the plan and every workspace slot before reading
 * them.  All calls share the one array, so calls that may overlap on the GPU
 * (different streams, or host threads racing on one device) race on it:
 * serialise them.
 */
mla_status mla_decode_paged_noalloc(const void* q_abs, const void* q_r, const void* kv_cache,
                                    int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                    const int32_t* seq_lens_host, const int32_t* q_lens_host, int32_t B,
                                    float scale, void* o_lat, float* lse, int32_t* dev_err, void* stream);

/* Test hook of mla_decode_paged_noalloc (no counterpart in the source pages):
 * the summary of the plan the last successful call on the current device
 * ran (its cluster count and split pieces).  MLA_ERR_INVALID_ARG before the
 * first call on this device or when out is NULL. */
mla_status mla_debug_noalloc_last_plan(mla_plan_info* out);

/* ---------------------------------------------------------------------------
 * Decoupled RoPE in fp32 ([P1] §1: the 64-d RoPE key carries the position
 * apart from the latent; §3: the plugin's RoPE compute dtype is fp32; §4:
 * the RoPE table is generated in fp32 and applied with fp32 multiply-adds).
 * Rotation: consecutive pairs (x[2i], x[2i+1]), i < 32, turned by the angle
 * p * base^(-2i/64) (the pages print no formula; the standard rotary
 * embedding, base 10000 by convention).
 * Shared rules: table is 16-byte aligned, positions and dev_err 4-byte
 * aligned (else MLA_ERR_MISALIGNED); NULL pointers, negative counts and
 * max_pos < 1 are MLA_ERR_INVALID_ARG and enqueue nothing.
 * ------------------------------------------------------------------------- */

/*
 * Fill table fp32 [max_pos, 32, 2] (device, caller-owned, 256 B per
 * position) with (cos, sin) of every position's angles, each computed in
 * double precision and rounded once to fp32.  base must be finite and > 1;
 * max_pos in [1, 2^24].  max_pos == 0 is a no-op.
 */
mla_status mla_rope_table(int32_t max_pos, float base, float* table, void* stream);

/*
 * Step A1 with the RoPE key rotated on the way in.  For i < n:
 *   kv_cache[slots[i]] = [c_kv_new[i, 0:512] | rope(k_pe_new[i, 0:64], positions[i])]
 * c_kv_new bf16 [n, 512] (copied bit for bit), k_pe_new bf16 [n, 64] (the
 * unrotated key), positions int32 [n] (each token's position in its sequence),
 * table from mla_rope_table with max_pos rows, slots int64 [n]; all device.
 * The rotation is fp32 (fused multiply-add) rounded to bf16.  A slot outside
 * the pool sets MLA_DEVERR_SLOT_OOB, a position outside [0, max_pos) sets
 * MLA_DEVERR_POS_OOB; either way that token is skipped.  n == 0 is a no-op.
 */
mla_status mla_kv_append_rope(const void* c_kv_new, const void* k_pe_new, const int32_t* positions,
                              const float* table, int32_t max_pos, const int64_t* slots, int32_t n,
                              void* kv_cache, int64_t num_pages, int32_t* dev_err, void* stream);

/*
 * Rotate the queries' RoPE part: q_r[t, h, :] = rope(q_pe[t, h, :], positions[t]),
 * q_pe and q_r bf16 [T, 128, 64] (may not overlap), positions int32 [T], table
 * as above; fp32 rotation rounded to bf16.  A position outside [0, max_pos)
 * sets MLA_DEVERR_POS_OOB and leaves that token's rows unwritten.  T == 0
 * is a no-op; overlapping q_pe and q_r is MLA_ERR_INVALID_ARG.
 */
mla_status mla_rope_q(const void* q_pe, const int32_t* positions, const float* table, int32_t max_pos,
                      void* q_r, int32_t T, int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------------------
 * Decompress branch ([P1] §3: kPrefillThresh = 256, the plugin's
 * prefill_absorption_threshold; §4 path A: K = c_KV·W_UK per head; [P2] MLA
 * section: V = c_KV·W_UV).  A chunk of at least MLA_PREFILL_THRESHOLD query
 * tokens of one sequence is not absorbed: its cached latent is expanded once
 * into per-head K_c and V_c, and standard causal attention runs per head,
 *   s = (q_c[t,h]·K_c[j,h] + q_R[t,h]·k_R[j]) * scale,  out[t,h] = softmax(s)·V_c[.,h],
 * query t of the chunk (M rows) sitting at position N - M + t of its
 * sequence (N tokens cached, the chunk included) and seeing [0, N - M + t].
 * The result equals steps A2-A5 of the absorbed path (the same out).
 * ------------------------------------------------------------------------- */
#define MLA_PREFILL_THRESHOLD 256
#define MLA_BRANCH_ABSORB 0
#define MLA_BRANCH_DECOMPRESS 1

/* The threshold (256) and the branch a sequence's q_len takes. */
int32_t mla_prefill_threshold(void);
int32_t mla_branch_for(int32_t q_len);

/*
 * Expand n cached rows: rows bf16 [n, 576] (e.g. from mla_gather_paged; only
 * columns 0..511 are read), W_UK bf16 [128, 128, 512], W_UV bf16 [128, 512, 128];
 * k_c[h, t, :] = rows[t, 0:512]·W_UK[h]^T and v_c[h, t, :] = rows[t, 0:512]·W_UV[h],
 * bf16 [128, n, 128], head-major (fp32 accumulation, one rounding).  All
 * pointers device, 16-byte aligned.  n == 0 is a no-op.
 */
mla_status mla_expand_kv(const void* rows, int32_t n, const void* w_uk, const void* w_uv, void* k_c, void* v_c,
                         int32_t* dev_err, void* stream);

/*
 * Causal attention of the decompress branch for one sequence: q_c bf16
 * [M, 128, 128] and q_r bf16 [M, 128, 64] (the chunk's rows), rows bf16
 * [N, 576] (k_R read from columns 512..575), k_c / v_c from mla_expand_kv,
 * out bf16 [M, 128, 128].  1 <= M <= N (M == 0 is a no-op); scale finite > 0.
 */
mla_status mla_prefill_attention(const void* q_c, const void* q_r, int32_t M, const void* rows, const void* k_c,
                                 const void* v_c, int32_t N, float scale, void* out, int32_t* dev_err,
                                 void* stream);

/* Workspace bytes mla_prefill_decompress needs for N cached tokens:
 * gathered rows [N, 576] (16-byte rounded) + K_c + V_c (2 * N * 32 KiB). */
mla_status mla_prefill_workspace_size(int32_t N, size_t* bytes);

/*
 * The whole branch for sequence b of a paged cache: gather its N cached
 * tokens, expand them (mla_expand_kv) and attend into out bf16
 * [M, 128, 128] (mla_prefill_decompress_batch with one sequence whose rows
 * start at row 0).  workspace is
 * device memory of at least mla_prefill_workspace_size(N) bytes, 16-byte
 * aligned; the same validation and device error bits as the three calls.
 */
mla_status mla_prefill_decompress(const void* q_c, const void* q_r, int32_t M, const void* kv_cache, int64_t num_pages,
                                  const int32_t* block_table, int32_t max_pages, int32_t b, int32_t N,
                                  const void* w_uk, const void* w_uv, float scale, void* workspace, size_t ws_bytes,
                                  void* out, int32_t* dev_err, void* stream);

/* Workspace bytes mla_prefill_decompress_batch needs for nb sequences of
 * n_tokens[i] cached tokens (host int32 [nb], nb <= 64): the packed rows
 * [Σ n, 576] (16-byte rounded) + K_c + V_c (2 * Σ n * 32 KiB).
 * MLA_ERR_INVALID_ARG for nb outside [0, 64] or a negative length. */
mla_status mla_prefill_batch_workspace_size(const int32_t* n_tokens, int32_t nb, size_t* bytes);

/*
 * The decompress branch for every qualifying sequence of a batch in three
 * launches: one gather of all nb sequences' cached rows into one packed
 * array, one expansion of all of them (mla_expand_kv over Σ n_tokens rows)
 * and one attention launch over every (sequence, head, 128-row query tile).
 * Host int32 arrays of nb entries (nb <= 64): seq_ids (block-table rows,
 * each in [0, batch)), q_starts (first row of the sequence's chunk in q_c,
 * q_r and out), q_lens (1 <= q_len <= n_tokens) and n_tokens (cached tokens
 * of the sequence, its chunk included).  q_c bf16 [rows, 128, 128], q_r
 * bf16 [rows, 128, 64], out bf16 [rows, 128, 128] on the device, rows the
 * largest q_starts[i] + q_lens[i]; only the chunks' rows of out are
 * written.  block_table int32 [batch, max_pages].  workspace: device, at
 * least mla_prefill_batch_workspace_size bytes, 16-byte aligned.  The same
 * validation and device error bits as the single-sequence calls (a
 * block-table entry outside the pool sets MLA_DEVERR_PAGE_OOB); nothing is
 * launched when validation fails.  nb == 0 is a no-op.
 */
mla_status mla_prefill_decompress_batch(const void* q_c, const void* q_r, const int32_t* seq_ids,
                                        const int32_t* q_starts, const int32_t* q_lens, const int32_t* n_tokens,
                                        int32_t nb, const void* kv_cache, int64_t num_pages,
                                        const int32_t* block_table, int32_t batch, int32_t max_pages,
                                        const void* w_uk, const void* w_uv, float scale, void* workspace,
                                        size_t ws_bytes, void* out, int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------------------
 * FP8 (E4M3) latent cache ([P3] bjbfmj.com/news/60700: quantisation scale
 * factors are stored beside the cached elements; [P1] opening section and
 * §5: a quantised gather with 16-byte vector loads).  E4M3 is the OCP 8-bit
 * floating point format (bias 7, 3 mantissa bits, subnormals, max 448).
 * Each token's 512 latent values share a power-of-two scale 2^k, k the
 * smallest integer with max|c| <= 448 * 2^k (k = 0 for an all-zero row);
 * codes are c * 2^-k rounded to the nearest E4M3 value, ties to even.  The
 * 64 RoPE values stay bf16.
 *
 * Layout (caller-owned device memory):
 *   rows   uint8 [num_pages][64][MLA_FP8_ROW_BYTES]: codes 0..511, then the
 *          64 bf16 RoPE values (bytes 512..639); 16-byte aligned;
 *   scales fp32 [num_pages][64]: 2^k per token; 16-byte aligned.
 * 644 bytes per token against 1152 for the bf16 cache.
 * ------------------------------------------------------------------------- */
#define MLA_FP8_ROW_BYTES 640

/*
 * Quantise and store: for i < n, rows[slots[i]] = [codes(c_kv_new[i]) | k_r_new[i]]
 * and scales[slots[i]] = 2^k.  c_kv_new bf16 [n, 512], k_r_new bf16 [n, 64],
 * slots int64 [n] (8-byte aligned).  A slot outside the pool sets
 * MLA_DEVERR_SLOT_OOB and that token is skipped.  n == 0 is a no-op.
 */
mla_status mla_kv_append_fp8(const void* c_kv_new, const void* k_r_new, const int64_t* slots, int32_t n,
                             void* rows, float* scales, int64_t num_pages, int32_t* dev_err, void* stream);

/*
 * Dequantising gather: out bf16 [n_tokens, 576] = the first n_tokens cached
 * tokens of sequence b, latent as code * 2^k (exact in bf16), then the RoPE
 * values bit for bit.  Errors as for mla_gather_paged.
 */
mla_status mla_gather_paged_fp8(const void* rows, const float* scales, int64_t num_pages,
                                const int32_t* block_table, int32_t max_pages, int32_t b, int32_t n_tokens,
                                void* out, int32_t* dev_err, void* stream);

/*
 * Steps A3 and A4 over the FP8 cache: as mla_decode_paged with kv_cache
 * replaced by (rows, scales) above.  The tensor-core operands are f16: the
 * latent is dequantised exactly on chip (code * 2^k is an exact f16 while
 * 2^-15 <= 2^k <= 2^7, i.e. max|c| of a token in [448 * 2^-16, 448 * 2^7];
 * all-zero tokens have k = 0), q_abs, q_R and the RoPE key are rounded from
 * bf16 to f16, and P is f16.  A token whose scale is outside that range is
 * clamped to it and sets MLA_DEVERR_FP8_RANGE.  The same plan and workspace
 * serve both formats.  Every slot read must hold finite codes (E4M3 NaN
 * codes are never written by mla_kv_append_fp8) and a power-of-two scale.
 */
mla_status mla_decode_paged_fp8(const void* q_abs, const void* q_r, const void* rows, const float* scales,
                                int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                const void* plan_dev, const mla_plan_info* info, float scale, void* workspace,
                                size_t ws_bytes, void* o_lat, float* lse, int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------------------
 * NVFP4 latent cache ([P1] opening section and §5: the latent is gathered in
 * NVFP4 with 16-byte vector loads, which fault on a base that is not 16-byte
 * aligned; here the host rejects such bases with MLA_ERR_MISALIGNED before
 * any launch).  NVFP4 as NVIDIA defines it: E2M1 elements (magnitudes 0, 0.5,
 * 1, 1.5, 2, 3, 4, 6), one E4M3 scale per block of 16 elements, one fp32
 * tensor scale s_t (here a caller constant, finite and > 0).
 *   block scale s_b = E4M3(fp32(amax_block / fp32(6 * s_t))), nearest even,
 *                     saturating at 448;
 *   code            = E2M1(fp32(x / fp32(s_b * s_t))), nearest even,
 *                     saturating at 6 (all zero when s_b * s_t is zero);
 *   value           = bf16(fp32(fp32(e2m1 * s_b) * s_t)).
 * Row layout, rows uint8 [num_pages][64][MLA_NVFP4_ROW_BYTES], 16-byte
 * aligned: bytes 0..255 the codes (element 2i in the low nibble of byte i),
 * 256..287 the 32 block scales, 288..415 the 64 bf16 RoPE values.
 * ------------------------------------------------------------------------- */
#define MLA_NVFP4_ROW_BYTES 416

/* Quantise and store rows[slots[i]] for i < n (as mla_kv_append_fp8). */
mla_status mla_kv_append_nvfp4(const void* c_kv_new, const void* k_r_new, const int64_t* slots, int32_t n,
                               float tensor_scale, void* rows, int64_t num_pages, int32_t* dev_err,
                               void* stream);

/* Dequantising gather into out bf16 [n_tokens, 576] (errors as mla_gather_paged). */
mla_status mla_gather_paged_nvfp4(const void* rows, float tensor_scale, int64_t num_pages,
                                  const int32_t* block_table, int32_t max_pages, int32_t b, int32_t n_tokens,
                                  void* out, int32_t* dev_err, void* stream);

/*
 * Batched dequantising gather, one launch for many sequences: for i < nb,
 * the first n_i = out_offsets[i+1] - out_offsets[i] cached tokens of
 * sequence seq_ids[i], in position order, go to rows [out_offsets[i],
 * out_offsets[i+1]) of out bf16 [total_tokens, 576] (the values of
 * mla_gather_paged_nvfp4).  seq_ids int32 [nb] and out_offsets int64 [nb+1]
 * are device arrays (out_offsets[0] = 0, non-decreasing, out_offsets[nb] =
 * total_tokens); block_table int32 [B, max_pages].  A row whose sequence id is
 * outside [0, B), whose position needs more than max_pages pages, or whose
 * offsets are inconsistent sets MLA_DEVERR_BATCH and is left unwritten; bad
 * page ids set MLA_DEVERR_PAGE_OOB.  nb == 0 or total_tokens == 0 is a no-op.
 * Host errors: MLA_ERR_INVALID_ARG (a null pointer, negative sizes, B or
 * max_pages < 1, tensor_scale not finite and > 0), MLA_ERR_MISALIGNED (rows
 * and out 16-byte, out_offsets 8-byte, the other pointers 4-byte aligned).
 */
mla_status mla_gather_paged_nvfp4_batch(const void* rows, float tensor_scale, int64_t num_pages,
                                        const int32_t* block_table, int32_t B, int32_t max_pages,
                                        const int32_t* seq_ids, const int64_t* out_offsets, int32_t nb,
                                        int64_t total_tokens, void* out, int32_t* dev_err, void* stream);

/*
 * Synchronise `stream`, read the device error word into *word_out (may be
 * NULL) and map it: 0 -> MLA_OK, MLA_DEVERR_TIMEOUT set -> MLA_ERR_TIMEOUT,
 * other bits -> MLA_ERR_DEVICE.  The word is not cleared.
 */
mla_status mla_check(void* stream, const int32_t* dev_err, int32_t* word_out);

/*
 * Test hook for the decode kernel's failure path (no counterpart on the
 * source pages; they describe no failure handling).  Every wait inside the
 * decode loop (mla_decode_paged, mla_decode_paged_fp8 and the entry points
 * built on them) gives up after `cycles` SM clock cycles, sets
 * MLA_DEVERR_TIMEOUT in the call's dev_err, and the kernel stops: it waits
 * for its own loads, MMAs and the score copies already in flight, frees its
 * tensor memory and returns, so the context stays usable.  0 restores the
 * default, 2^31 cycles (about a second at the maximum SM clock).  The
 * setting is process-wide and applies to launches made after the call.
 * Errors: MLA_ERR_INVALID_ARG if cycles exceeds the default.
 */
mla_status mla_debug_set_decode_wait_limit(uint64_t cycles);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
