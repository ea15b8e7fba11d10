// C-ABI entry points of libmla (declared in include/mla.h): argument
// validation, the page pool, slot mapping, the split-KV planner, TMA tensor
// maps and kernel launches.  No entry point allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/mla.h"
#include "internal.h"

namespace {

thread_local std::string g_last_error = "no error";

// Bound of the decode kernel's waits, in SM cycles (about a second at the
// maximum clock); mla_debug_set_decode_wait_limit changes it for tests.
constexpr uint64_t kDefaultDecodeWaitLimit = 1ull << 31;
std::atomic<uint64_t> g_decode_wait_limit{kDefaultDecodeWaitLimit};

mla_status fail(mla_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

mla_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MLA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

#define CHECK_PTR(p)                                                     \
  do {                                                                   \
    if ((p) == nullptr) return fail(MLA_ERR_INVALID_ARG, "%s is NULL", #p); \
  } while (0)
#define CHECK_ALIGN16(p)                                                                          \
  do {                                                                                            \
    if (!aligned16(p)) return fail(MLA_ERR_MISALIGNED, "%s is not 16-byte aligned", #p);          \
  } while (0)

constexpr int64_t kRowBytes = MLA_TOKEN_ELEMS * 2;  // 1152

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 tensor map (128-byte swizzle unless told otherwise); dims innermost
// first, strides in bytes for dims 1..rank-1.
mla_status make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                    const uint32_t* box, const char* what,
                    CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
                    CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, dtype, (cuuint32_t)rank, const_cast<void*>(base),
                  reinterpret_cast<const cuuint64_t*>(dims), reinterpret_cast<const cuuint64_t*>(strides),
                  reinterpret_cast<const cuuint32_t*>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
  return MLA_OK;
}

// ------------------------------------------------------------------ planner
struct PlanRow {
  int32_t b;
  int32_t visible;
  int32_t npages;
};

// Minimum 64-token tiles per cluster: below it, the per-range fixed costs
// (query load, epilogue, a combine partial) outweigh the added parallelism.
constexpr int64_t kMinTilesPerCluster = 2;

mla_status build_plan(const int32_t* seq_lens, const int32_t* q_lens, int32_t B, int32_t num_clusters,
                      int32_t* out, size_t out_words, mla_plan_info* info) {
  if (B < 0) return fail(MLA_ERR_INVALID_ARG, "B = %d is negative", B);
  if (B > 0) {
    CHECK_PTR(seq_lens);
    CHECK_PTR(q_lens);
  }
  if (num_clusters < 1) return fail(MLA_ERR_INVALID_ARG, "num_clusters = %d < 1", num_clusters);
  std::vector<PlanRow> rows;
  int64_t total = 0;
  int32_t max_pages = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t n = seq_lens[b], q = q_lens[b];
    if (n < 1) return fail(MLA_ERR_INVALID_ARG, "seq_lens[%d] = %d < 1", b, n);
    if (q < 0 || q > n) return fail(MLA_ERR_INVALID_ARG, "q_lens[%d] = %d outside [0, seq_len = %d]", b, q, n);
    max_pages = std::max<int32_t>(max_pages, (n + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE);
    for (int32_t i = 0; i < q; ++i) {
      const int32_t vis = n - q + i + 1;
      const int32_t np = (vis + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;
      rows.push_back({b, vis, np});
      total += np;
    }
    if ((int64_t)rows.size() > (int64_t)INT32_MAX / MLA_NUM_HEADS)
      return fail(MLA_ERR_INVALID_ARG, "too many query rows");
  }
  const int64_t T = (int64_t)rows.size();
  // Lanes: when every sequence has the same number Q >= 2 of query rows
  // (multi-token decode), the clusters are split into Q lanes and lane j takes
  // row j of every sequence, cut into equal contiguous tile ranges the same
  // way in every lane.  Cluster c of each lane then reads the same pages at
  // nearly the same time, so the rows of a sequence share one DRAM read of
  // each page through L2.  Otherwise there is one lane over all rows.
  int32_t lanes = 1;
  {
    int32_t q0 = -1;
    bool uniform = true;
    for (int32_t b = 0; b < B; ++b) {
      if (q_lens[b] == 0) continue;
      if (q0 < 0) q0 = q_lens[b];
      uniform = uniform && q_lens[b] == q0;
    }
    if (uniform && q0 >= 2 && num_clusters / q0 >= 1) lanes = q0;
  }
  std::vector<std::vector<int32_t>> lane_rows(lanes);
  {
    int32_t r = 0;
    for (int32_t b = 0; b < B; ++b)
      for (int32_t i = 0; i < q_lens[b]; ++i, ++r) lane_rows[lanes == 1 ? 0 : i].push_back(r);
  }
  const int32_t clusters_per_lane = num_clusters / lanes;
  // segments
  struct Seg {
    int32_t row, b, pb, pe, vis, slot;
  };
  std::vector<Seg> segs;
  std::vector<int32_t> seg_off;
  std::vector<int32_t> row_pieces(T, 0);
  for (int32_t lane = 0; lane < lanes; ++lane) {
    const std::vector<int32_t>& lr = lane_rows[lane];
    int64_t lane_total = 0;
    for (int32_t r : lr) lane_total += rows[r].npages;
    if (lane_total == 0) continue;
    const int64_t tiles_per =
        std::max<int64_t>((lane_total + clusters_per_lane - 1) / clusters_per_lane, kMinTilesPerCluster);
    const int64_t used = (lane_total + tiles_per - 1) / tiles_per;
    int64_t row_start = 0;
    size_t k = 0;  // index into lr
    for (int64_t c = 0; c < used; ++c) {
      const int64_t lo = c * tiles_per, hi = std::min(lane_total, lo + tiles_per);
      seg_off.push_back((int32_t)segs.size());
      while (k < lr.size() && row_start + rows[lr[k]].npages <= lo) row_start += rows[lr[k++]].npages;
      int64_t rs = row_start;
      for (size_t kk = k; kk < lr.size() && rs < hi; rs += rows[lr[kk++]].npages) {
        const int32_t rr = lr[kk];
        const int64_t pb = std::max<int64_t>(lo - rs, 0), pe = std::min<int64_t>(hi - rs, rows[rr].npages);
        if (pe <= pb) continue;
        segs.push_back({rr, rows[rr].b, (int32_t)pb, (int32_t)pe, rows[rr].visible, -1});
        ++row_pieces[rr];
      }
    }
  }
  const int64_t used = (int64_t)seg_off.size();
  seg_off.push_back((int32_t)segs.size());
  // partial slots for rows cut into several pieces, contiguous per row
  std::vector<int32_t> split;  // {row, slot_begin, n, 0}
  int32_t nslots = 0;
  {
    int32_t last_row = -1;
    for (auto& s : segs) {
      if (row_pieces[s.row] < 2) continue;
      if (s.row != last_row) {
        split.insert(split.end(), {s.row, nslots, row_pieces[s.row], 0});
        last_row = s.row;
      }
      s.slot = nslots++;
    }
  }
  const int64_t nsplit = (int64_t)split.size() / mla::kSplitWords;
  const mla::PlanLayout L = mla::plan_layout(used, (int64_t)segs.size(), nsplit);
  if ((size_t)L.words > out_words)
    return fail(MLA_ERR_INVALID_ARG, "plan buffer holds %zu bytes, %lld needed", out_words * 4,
                (long long)L.words * 4);
  std::fill(out, out + L.words, 0);
  out[0] = (int32_t)MLA_PLAN_MAGIC;
  out[1] = (int32_t)T;
  out[2] = B;
  out[3] = (int32_t)used;
  out[4] = (int32_t)segs.size();
  out[5] = nslots;
  out[6] = (int32_t)nsplit;
  out[7] = max_pages;
  std::copy(seg_off.begin(), seg_off.end(), out + L.seg_off);
  for (size_t i = 0; i < segs.size(); ++i) {
    int32_t* w = out + L.seg_base + mla::kSegWords * i;
    w[0] = segs[i].row;
    w[1] = segs[i].b;
    w[2] = segs[i].pb;
    w[3] = segs[i].pe;
    w[4] = segs[i].vis;
    w[5] = segs[i].slot;
  }
  std::copy(split.begin(), split.end(), out + L.split_base);
  if (info) {
    info->magic = MLA_PLAN_MAGIC;
    info->T = (int32_t)T;
    info->B = B;
    info->num_clusters = (int32_t)used;
    info->num_segments = (int32_t)segs.size();
    info->num_partials = nslots;
    info->num_split_rows = (int32_t)nsplit;
    info->max_pages_needed = max_pages;
    info->total_tiles = total;
    info->plan_bytes = (size_t)L.words * 4;
  }
  return MLA_OK;
}

size_t workspace_bytes_for(int64_t partials) {
  return (size_t)partials * (MLA_NUM_HEADS * MLA_LATENT_DIM * 4 + MLA_NUM_HEADS * 4);
}

}  // namespace

namespace mla {
mla_status set_last_error(mla_status s, const char* message) { return fail(s, "%s", message); }

PlanLayout plan_layout(int64_t num_clusters, int64_t num_segments, int64_t num_split_rows) {
  PlanLayout L;
  L.seg_off = kPlanHeader;
  L.seg_base = (L.seg_off + num_clusters + 1 + 7) / 8 * 8;
  L.split_base = L.seg_base + kSegWords * num_segments;
  L.words = L.split_base + kSplitWords * num_split_rows;
  return L;
}
}  // namespace mla

struct mla_pool {
  std::vector<uint8_t> used;
  int32_t free_count = 0;
};

extern "C" {

const char* mla_last_error(void) { return g_last_error.c_str(); }

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_MISALIGNED: return "MLA_ERR_MISALIGNED";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_DEVICE: return "MLA_ERR_DEVICE";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_NO_SPACE: return "MLA_ERR_NO_SPACE";
  }
  return "MLA_ERR_UNKNOWN";
}

int32_t mla_version(void) { return 100; }

mla_config mla_config_default(void) {
  mla_config c;
  c.num_heads = MLA_NUM_HEADS;
  c.head_dim_c = MLA_HEAD_DIM_C;
  c.latent_dim = MLA_LATENT_DIM;
  c.rope_dim = MLA_ROPE_DIM;
  c.page_size = MLA_PAGE_SIZE;
  c.scale = (float)(1.0 / std::sqrt((double)(MLA_HEAD_DIM_C + MLA_ROPE_DIM)));
  return c;
}

mla_status mla_config_validate(const mla_config* cfg) {
  CHECK_PTR(cfg);
  if (cfg->num_heads != MLA_NUM_HEADS || cfg->head_dim_c != MLA_HEAD_DIM_C || cfg->latent_dim != MLA_LATENT_DIM ||
      cfg->rope_dim != MLA_ROPE_DIM || cfg->page_size != MLA_PAGE_SIZE)
    return fail(MLA_ERR_UNSUPPORTED, "only heads=128, d_hc=128, d_c=512, d_r=64, page_size=64 are supported");
  if (!(cfg->scale > 0.f) || !std::isfinite(cfg->scale))
    return fail(MLA_ERR_INVALID_ARG, "scale must be finite and positive");
  return MLA_OK;
}

mla_status mla_kv_bytes(int64_t layers, int64_t dc, int64_t dr, int64_t elem_bytes, int64_t tokens, int64_t seqs,
                        uint64_t* out) {
  CHECK_PTR(out);
  if (layers <= 0 || dc <= 0 || elem_bytes <= 0 || tokens <= 0 || seqs <= 0 || dr < 0)
    return fail(MLA_ERR_INVALID_ARG, "invalid dimension");
  uint64_t acc = (uint64_t)layers, t;
  if (__builtin_add_overflow((uint64_t)dc, (uint64_t)dr, &t) || __builtin_mul_overflow(acc, t, &acc) ||
      __builtin_mul_overflow(acc, (uint64_t)elem_bytes, &acc) || __builtin_mul_overflow(acc, (uint64_t)tokens, &acc) ||
      __builtin_mul_overflow(acc, (uint64_t)seqs, &acc))
    return fail(MLA_ERR_INVALID_ARG, "byte count overflows uint64");
  *out = acc;
  return MLA_OK;
}

// ------------------------------------------------------------------ pool
mla_status mla_pool_create(int32_t num_pages, mla_pool** out) {
  CHECK_PTR(out);
  if (num_pages < 1) return fail(MLA_ERR_INVALID_ARG, "num_pages = %d < 1", num_pages);
  auto* p = new (std::nothrow) mla_pool();
  if (!p) return fail(MLA_ERR_NO_SPACE, "out of host memory");
  p->used.assign((size_t)num_pages, 0);
  p->free_count = num_pages;
  *out = p;
  return MLA_OK;
}

mla_status mla_pool_alloc(mla_pool* pool, int32_t n, int32_t* ids) {
  CHECK_PTR(pool);
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "n = %d < 0", n);
  if (n == 0) return MLA_OK;
  CHECK_PTR(ids);
  if (n > pool->free_count)
    return fail(MLA_ERR_NO_SPACE, "%d pages requested, %d free", n, pool->free_count);
  int32_t k = 0;
  for (size_t i = 0; i < pool->used.size() && k < n; ++i)
    if (!pool->used[i]) {
      pool->used[i] = 1;
      ids[k++] = (int32_t)i;
    }
  pool->free_count -= n;
  return MLA_OK;
}

mla_status mla_pool_free(mla_pool* pool, const int32_t* ids, int32_t n) {
  CHECK_PTR(pool);
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "n = %d < 0", n);
  if (n == 0) return MLA_OK;
  CHECK_PTR(ids);
  std::vector<uint8_t> seen(pool->used.size(), 0);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || (size_t)id >= pool->used.size()) return fail(MLA_ERR_INVALID_ARG, "page id %d out of range", id);
    if (!pool->used[id]) return fail(MLA_ERR_INVALID_ARG, "page id %d is not allocated", id);
    if (seen[id]) return fail(MLA_ERR_INVALID_ARG, "page id %d repeated", id);
    seen[id] = 1;
  }
  for (int32_t i = 0; i < n; ++i) pool->used[ids[i]] = 0;
  pool->free_count += n;
  return MLA_OK;
}

mla_status mla_pool_available(const mla_pool* pool, int32_t* out) {
  CHECK_PTR(pool);
  CHECK_PTR(out);
  *out = pool->free_count;
  return MLA_OK;
}

void mla_pool_destroy(mla_pool* pool) { delete pool; }

mla_status mla_slot_mapping(const int32_t* block_table, int32_t batch, int32_t max_pages, const int32_t* seq_ids,
                            const int32_t* positions, int32_t n, int64_t* slots_out) {
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "n = %d < 0", n);
  if (n == 0) return MLA_OK;
  CHECK_PTR(block_table);
  CHECK_PTR(seq_ids);
  CHECK_PTR(positions);
  CHECK_PTR(slots_out);
  if (batch < 1 || max_pages < 1) return fail(MLA_ERR_INVALID_ARG, "batch and max_pages must be >= 1");
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = seq_ids[i], pos = positions[i];
    if (b < 0 || b >= batch) return fail(MLA_ERR_INVALID_ARG, "seq_ids[%d] = %d out of range", i, b);
    if (pos < 0 || pos / MLA_PAGE_SIZE >= max_pages)
      return fail(MLA_ERR_INVALID_ARG, "positions[%d] = %d beyond the block table", i, pos);
    const int32_t page = block_table[(int64_t)b * max_pages + pos / MLA_PAGE_SIZE];
    if (page < 0) return fail(MLA_ERR_INVALID_ARG, "no page mapped for sequence %d position %d", b, pos);
    slots_out[i] = (int64_t)page * MLA_PAGE_SIZE + pos % MLA_PAGE_SIZE;
  }
  return MLA_OK;
}

// ------------------------------------------------------------------ device steps
mla_status mla_cache_init(void* kv_cache, int64_t num_pages, void* stream) {
  CHECK_PTR(kv_cache);
  CHECK_ALIGN16(kv_cache);
  if (num_pages < 1) return fail(MLA_ERR_INVALID_ARG, "num_pages = %lld < 1", (long long)num_pages);
  cudaError_t e = cudaMemsetAsync(kv_cache, 0, (size_t)num_pages * MLA_PAGE_BYTES, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return MLA_OK;
}

mla_status mla_kv_append(const void* c_kv_new, const void* k_r_new, const int64_t* slots, int32_t n, void* kv_cache,
                         int64_t num_pages, int32_t* dev_err, void* stream) {
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "n = %d < 0", n);
  if (n == 0) return MLA_OK;
  CHECK_PTR(c_kv_new);
  CHECK_PTR(k_r_new);
  CHECK_PTR(slots);
  CHECK_PTR(kv_cache);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(c_kv_new);
  CHECK_ALIGN16(k_r_new);
  CHECK_ALIGN16(kv_cache);
  if (!aligned(slots, 8)) return fail(MLA_ERR_MISALIGNED, "slots is not 8-byte aligned");
  if (!aligned(dev_err, 4)) return fail(MLA_ERR_MISALIGNED, "dev_err is not 4-byte aligned");
  if (num_pages < 1) return fail(MLA_ERR_INVALID_ARG, "num_pages = %lld < 1", (long long)num_pages);
  cudaError_t e = mla::launch_kv_append((const uint16_t*)c_kv_new, (const uint16_t*)k_r_new, slots, n,
                                        (uint16_t*)kv_cache, num_pages * MLA_PAGE_SIZE, dev_err, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return MLA_OK;
}

mla_status mla_rope_table(int32_t max_pos, float base, float* table, void* stream) {
  if (max_pos < 0 || max_pos > (1 << 24)) return fail(MLA_ERR_INVALID_ARG, "max_pos = %d outside [0, 2^24]", max_pos);
  if (!(base > 1.f) || !std::isfinite(base)) return fail(MLA_ERR_INVALID_ARG, "base must be finite and > 1");
  if (max_pos == 0) return MLA_OK;
  CHECK_PTR(table);
  CHECK_ALIGN16(table);
  cudaError_t e = mla::launch_rope_table(table, max_pos, (double)base, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope_table launch");
  return MLA_OK;
}

mla_status mla_kv_append_rope(const void* c_kv_new, const void* k_pe_new, const int32_t* positions, const float* table,
                              int32_t max_pos, const int64_t* slots, int32_t n, void* kv_cache, int64_t num_pages,
                              int32_t* dev_err, void* stream) {
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "n = %d < 0", n);
  if (n == 0) return MLA_OK;
  CHECK_PTR(c_kv_new);
  CHECK_PTR(k_pe_new);
  CHECK_PTR(positions);
  CHECK_PTR(table);
  CHECK_PTR(slots);
  CHECK_PTR(kv_cache);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(c_kv_new);
  CHECK_ALIGN16(k_pe_new);
  CHECK_ALIGN16(kv_cache);
  CHECK_ALIGN16(table);
  if (!aligned(slots, 8)) return fail(MLA_ERR_MISALIGNED, "slots is not 8-byte aligned");
  if (!aligned(positions, 4) || !aligned(dev_err, 4))
    return fail(MLA_ERR_MISALIGNED, "positions and dev_err must be 4-byte aligned");
  if (max_pos < 1) return fail(MLA_ERR_INVALID_ARG, "max_pos = %d < 1", max_pos);
  if (num_pages < 1) return fail(MLA_ERR_INVALID_ARG, "num_pages = %lld < 1", (long long)num_pages);
  cudaError_t e = mla::launch_kv_append_rope((const uint16_t*)c_kv_new, (const uint16_t*)k_pe_new, positions, table,
                                             max_pos, slots, n, (uint16_t*)kv_cache, num_pages * MLA_PAGE_SIZE,
                                             dev_err, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kv_append_rope launch");
  return MLA_OK;
}

mla_status mla_rope_q(const void* q_pe, const int32_t* positions, const float* table, int32_t max_pos, void* q_r,
                      int32_t T, int32_t* dev_err, void* stream) {
  if (T < 0) return fail(MLA_ERR_INVALID_ARG, "T = %d < 0", T);
  if (T == 0) return MLA_OK;
  CHECK_PTR(q_pe);
  CHECK_PTR(positions);
  CHECK_PTR(table);
  CHECK_PTR(q_r);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(q_pe);
  CHECK_ALIGN16(q_r);
  if (!aligned(positions, 4) || !aligned(dev_err, 4))
    return fail(MLA_ERR_MISALIGNED, "positions and dev_err must be 4-byte aligned");
  CHECK_ALIGN16(table);
  if (max_pos < 1) return fail(MLA_ERR_INVALID_ARG, "max_pos = %d < 1", max_pos);
  const uintptr_t a0 = (uintptr_t)q_pe, b0 = (uintptr_t)q_r, len = (uintptr_t)T * MLA_NUM_HEADS * MLA_ROPE_DIM * 2;
  if (a0 < b0 + len && b0 < a0 + len) return fail(MLA_ERR_INVALID_ARG, "q_pe and q_r overlap");
  cudaError_t e = mla::launch_rope_q((const uint16_t*)q_pe, positions, table, max_pos, (uint16_t*)q_r, T, dev_err,
                                     (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope_q launch");
  return MLA_OK;
}

mla_status mla_gather_paged(const void* kv_cache, int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                            int32_t b, int32_t n_tokens, void* out, int32_t* dev_err, void* stream) {
  if (n_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "n_tokens = %d < 0", n_tokens);
  if (n_tokens == 0) return MLA_OK;
  CHECK_PTR(kv_cache);
  CHECK_PTR(block_table);
  CHECK_PTR(out);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(kv_cache);
  CHECK_ALIGN16(out);
  if (num_pages < 1 || max_pages < 1 || b < 0) return fail(MLA_ERR_INVALID_ARG, "bad pool/table sizes");
  if ((n_tokens + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE > max_pages)
    return fail(MLA_ERR_INVALID_ARG, "n_tokens = %d needs more than max_pages = %d pages", n_tokens, max_pages);
  cudaError_t e = mla::launch_gather((const uint16_t*)kv_cache, num_pages, block_table, max_pages, b, n_tokens,
                                     (uint16_t*)out, dev_err, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  return MLA_OK;
}

mla_status mla_kv_append_fp8(const void* c_kv_new, const void* k_r_new, const int64_t* slots, int32_t n,
                             void* rows, float* scales, int64_t num_pages, int32_t* dev_err, void* stream) {
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "n = %d < 0", n);
  if (n == 0) return MLA_OK;
  CHECK_PTR(c_kv_new);
  CHECK_PTR(k_r_new);
  CHECK_PTR(slots);
  CHECK_PTR(rows);
  CHECK_PTR(scales);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(c_kv_new);
  CHECK_ALIGN16(k_r_new);
  CHECK_ALIGN16(rows);
  CHECK_ALIGN16(scales);
  if (!aligned(slots, 8)) return fail(MLA_ERR_MISALIGNED, "slots is not 8-byte aligned");
  if (!aligned(dev_err, 4)) return fail(MLA_ERR_MISALIGNED, "dev_err is not 4-byte aligned");
  if (num_pages < 1) return fail(MLA_ERR_INVALID_ARG, "num_pages = %lld < 1", (long long)num_pages);
  cudaError_t e = mla::launch_kv_append_fp8((const uint16_t*)c_kv_new, (const uint16_t*)k_r_new, slots, n,
                                            (uint8_t*)rows, scales, num_pages * MLA_PAGE_SIZE, dev_err,
                                            (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kv_append_fp8 launch");
  return MLA_OK;
}

mla_status mla_gather_paged_fp8(const void* rows, const float* scales, int64_t num_pages,
                                const int32_t* block_table, int32_t max_pages, int32_t b, int32_t n_tokens,
                                void* out, int32_t* dev_err, void* stream) {
  if (n_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "n_tokens = %d < 0", n_tokens);
  if (n_tokens == 0) return MLA_OK;
  CHECK_PTR(rows);
  CHECK_PTR(scales);
  CHECK_PTR(block_table);
  CHECK_PTR(out);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(rows);
  CHECK_ALIGN16(scales);
  CHECK_ALIGN16(out);
  if (!aligned(block_table, 4) || !aligned(dev_err, 4))
    return fail(MLA_ERR_MISALIGNED, "block_table and dev_err must be 4-byte aligned");
  if (num_pages < 1 || max_pages < 1 || b < 0) return fail(MLA_ERR_INVALID_ARG, "bad pool/table sizes");
  if ((n_tokens + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE > max_pages)
    return fail(MLA_ERR_INVALID_ARG, "n_tokens = %d needs more than max_pages = %d pages", n_tokens, max_pages);
  cudaError_t e = mla::launch_gather_fp8((const uint8_t*)rows, scales, num_pages, block_table, max_pages, b,
                                         n_tokens, (uint16_t*)out, dev_err, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "gather_fp8 launch");
  return MLA_OK;
}

mla_status mla_kv_append_nvfp4(const void* c_kv_new, const void* k_r_new, const int64_t* slots, int32_t n,
                               float tensor_scale, void* rows, int64_t num_pages, int32_t* dev_err,
                               void* stream) {
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "n = %d < 0", n);
  if (n == 0) return MLA_OK;
  if (!(tensor_scale > 0.f) || !std::isfinite(tensor_scale))
    return fail(MLA_ERR_INVALID_ARG, "tensor_scale must be finite and > 0");
  CHECK_PTR(c_kv_new);
  CHECK_PTR(k_r_new);
  CHECK_PTR(slots);
  CHECK_PTR(rows);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(c_kv_new);
  CHECK_ALIGN16(k_r_new);
  CHECK_ALIGN16(rows);
  if (!aligned(slots, 8)) return fail(MLA_ERR_MISALIGNED, "slots is not 8-byte aligned");
  if (!aligned(dev_err, 4)) return fail(MLA_ERR_MISALIGNED, "dev_err is not 4-byte aligned");
  if (num_pages < 1) return fail(MLA_ERR_INVALID_ARG, "num_pages = %lld < 1", (long long)num_pages);
  cudaError_t e = mla::launch_kv_append_nvfp4((const uint16_t*)c_kv_new, (const uint16_t*)k_r_new, slots, n,
                                              tensor_scale, (uint8_t*)rows, num_pages * MLA_PAGE_SIZE, dev_err,
                                              (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kv_append_nvfp4 launch");
  return MLA_OK;
}

mla_status mla_gather_paged_nvfp4(const void* rows, float tensor_scale, int64_t num_pages,
                                  const int32_t* block_table, int32_t max_pages, int32_t b, int32_t n_tokens,
                                  void* out, int32_t* dev_err, void* stream) {
  if (n_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "n_tokens = %d < 0", n_tokens);
  if (n_tokens == 0) return MLA_OK;
  if (!(tensor_scale > 0.f) || !std::isfinite(tensor_scale))
    return fail(MLA_ERR_INVALID_ARG, "tensor_scale must be finite and > 0");
  CHECK_PTR(rows);
  CHECK_PTR(block_table);
  CHECK_PTR(out);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(rows);
  CHECK_ALIGN16(out);
  if (!aligned(block_table, 4) || !aligned(dev_err, 4))
    return fail(MLA_ERR_MISALIGNED, "block_table and dev_err must be 4-byte aligned");
  if (num_pages < 1 || max_pages < 1 || b < 0) return fail(MLA_ERR_INVALID_ARG, "bad pool/table sizes");
  if ((n_tokens + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE > max_pages)
    return fail(MLA_ERR_INVALID_ARG, "n_tokens = %d needs more than max_pages = %d pages", n_tokens, max_pages);
  cudaError_t e = mla::launch_gather_nvfp4((const uint8_t*)rows, tensor_scale, num_pages, block_table, max_pages, b,
                                           n_tokens, (uint16_t*)out, dev_err, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "gather_nvfp4 launch");
  return MLA_OK;
}

mla_status mla_gather_paged_nvfp4_batch(const void* rows, float tensor_scale, int64_t num_pages,
                                        const int32_t* block_table, int32_t B, int32_t max_pages,
                                        const int32_t* seq_ids, const int64_t* out_offsets, int32_t nb,
                                        int64_t total_tokens, void* out, int32_t* dev_err, void* stream) {
  if (nb < 0 || total_tokens < 0)
    return fail(MLA_ERR_INVALID_ARG, "nb = %d, total_tokens = %lld: negative", nb, (long long)total_tokens);
  if (nb == 0 || total_tokens == 0) return MLA_OK;
  if (!(tensor_scale > 0.f) || !std::isfinite(tensor_scale))
    return fail(MLA_ERR_INVALID_ARG, "tensor_scale must be finite and > 0");
  CHECK_PTR(rows);
  CHECK_PTR(block_table);
  CHECK_PTR(seq_ids);
  CHECK_PTR(out_offsets);
  CHECK_PTR(out);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(rows);
  CHECK_ALIGN16(out);
  if (!aligned(out_offsets, 8)) return fail(MLA_ERR_MISALIGNED, "out_offsets is not 8-byte aligned");
  if (!aligned(block_table, 4) || !aligned(seq_ids, 4) || !aligned(dev_err, 4))
    return fail(MLA_ERR_MISALIGNED, "block_table, seq_ids and dev_err must be 4-byte aligned");
  if (num_pages < 1 || B < 1 || max_pages < 1) return fail(MLA_ERR_INVALID_ARG, "bad pool/table sizes");
  if (total_tokens > ((int64_t)1 << 40)) return fail(MLA_ERR_INVALID_ARG, "total_tokens too large");
  cudaError_t e = mla::launch_gather_nvfp4_batch((const uint8_t*)rows, tensor_scale, num_pages, block_table, B,
                                                 max_pages, seq_ids, out_offsets, nb, total_tokens, (uint16_t*)out,
                                                 dev_err, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "gather_nvfp4_batch launch");
  return MLA_OK;
}

// Decompress-branch workspace: gathered rows [N, 576] (rounded up to 16 B),
// then K_c and V_c [N, 128, 128] bf16.
static size_t prefill_rows_bytes(int64_t N) { return ((size_t)N * kRowBytes + 15) / 16 * 16; }
static size_t prefill_ws_bytes(int64_t N) {
  return prefill_rows_bytes(N) + 2 * (size_t)N * MLA_NUM_HEADS * MLA_HEAD_DIM_C * 2;
}

static mla_status head_gemm(mla::HeadGemm kind, const void* a, const void* w, void* c, int32_t T, int32_t* dev_err,
                            void* stream) {
  if (T < 0) return fail(MLA_ERR_INVALID_ARG, "T = %d < 0", T);
  if (T == 0) return MLA_OK;
  CHECK_PTR(a);
  CHECK_PTR(w);
  CHECK_PTR(c);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(a);
  CHECK_ALIGN16(w);
  CHECK_ALIGN16(c);
  if (T > (1 << 24)) return fail(MLA_ERR_INVALID_ARG, "T = %d too large", T);
  const bool absorb = kind == mla::HeadGemm::kAbsorbQ;
  const uint64_t K = absorb ? MLA_HEAD_DIM_C : MLA_LATENT_DIM;
  const uint64_t N = absorb ? MLA_LATENT_DIM : MLA_HEAD_DIM_C;
  CUtensorMap amap, wmap;
  // activations [T, 128, K]; box = 64 of K x 1 head x 128 tokens
  const uint64_t adims[3] = {K, MLA_NUM_HEADS, (uint64_t)T};
  const uint64_t astr[2] = {K * 2, K * 2 * MLA_NUM_HEADS};
  const uint32_t abox[3] = {64, 1, 128};
  // weights [128, K, N]; box = 64 of N x 64 of K x 1 head
  const uint64_t wdims[3] = {N, K, MLA_NUM_HEADS};
  const uint64_t wstr[2] = {N * 2, N * 2 * K};
  const uint32_t wbox[3] = {64, 64, 1};
  // outputs [T, 128, N]; box = 64 of N x 1 head x 128 tokens (TMA store)
  const uint64_t cdims[3] = {N, MLA_NUM_HEADS, (uint64_t)T};
  const uint64_t cstr[2] = {N * 2, N * 2 * MLA_NUM_HEADS};
  CUtensorMap cmap;
  mla_status s = make_map(&amap, a, 3, adims, astr, abox, "activations");
  if (s != MLA_OK) return s;
  s = make_map(&wmap, w, 3, wdims, wstr, wbox, "weights");
  if (s != MLA_OK) return s;
  s = make_map(&cmap, c, 3, cdims, cstr, abox, "outputs");
  if (s != MLA_OK) return s;
  cudaError_t e = mla::launch_head_gemm(kind, amap, wmap, cmap, T, dev_err, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, absorb ? "absorb_q launch" : "up_v launch");
  return MLA_OK;
}

// ------------------------------------------------------------------ decompress branch
int32_t mla_prefill_threshold(void) { return MLA_PREFILL_THRESHOLD; }

int32_t mla_branch_for(int32_t q_len) { return q_len >= MLA_PREFILL_THRESHOLD ? MLA_BRANCH_DECOMPRESS : MLA_BRANCH_ABSORB; }

mla_status mla_expand_kv(const void* rows, int32_t n, const void* w_uk, const void* w_uv, void* k_c, void* v_c,
                         int32_t* dev_err, void* stream) {
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "n = %d < 0", n);
  if (n == 0) return MLA_OK;
  CHECK_PTR(rows);
  CHECK_PTR(w_uk);
  CHECK_PTR(w_uv);
  CHECK_PTR(k_c);
  CHECK_PTR(v_c);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(rows);
  CHECK_ALIGN16(w_uk);
  CHECK_ALIGN16(w_uv);
  CHECK_ALIGN16(k_c);
  CHECK_ALIGN16(v_c);
  if (!aligned(dev_err, 4)) return fail(MLA_ERR_MISALIGNED, "dev_err is not 4-byte aligned");
  if (n > (1 << 24)) return fail(MLA_ERR_INVALID_ARG, "n = %d too large", n);
  CUtensorMap amap, kmap, vmap;
  // latent part of the rows [n, 576] as {512, 1 (shared by every head), n}
  const uint64_t adims[3] = {MLA_LATENT_DIM, 1, (uint64_t)n};
  const uint64_t astr[2] = {(uint64_t)kRowBytes, (uint64_t)kRowBytes};
  const uint32_t abox[3] = {64, 1, 128};
  mla_status s = make_map(&amap, rows, 3, adims, astr, abox, "latent rows");
  if (s != MLA_OK) return s;
  // W_UK [128, 128 (d_hc), 512 (d_c)] read K-major: box 64 of d_c x 64 of d_hc (one CTA's half) x 1 head
  const uint64_t kdims[3] = {MLA_LATENT_DIM, MLA_HEAD_DIM_C, MLA_NUM_HEADS};
  const uint64_t kstr[2] = {MLA_LATENT_DIM * 2, (uint64_t)MLA_LATENT_DIM * 2 * MLA_HEAD_DIM_C};
  const uint32_t kbox[3] = {64, 64, 1};
  s = make_map(&kmap, w_uk, 3, kdims, kstr, kbox, "W_UK (K-major)");
  if (s != MLA_OK) return s;
  // W_UV [128, 512 (d_c), 128 (d_hc)] as in step A5
  const uint64_t vdims[3] = {MLA_HEAD_DIM_C, MLA_LATENT_DIM, MLA_NUM_HEADS};
  const uint64_t vstr[2] = {MLA_HEAD_DIM_C * 2, (uint64_t)MLA_HEAD_DIM_C * 2 * MLA_LATENT_DIM};
  const uint32_t vbox[3] = {64, 64, 1};
  s = make_map(&vmap, w_uv, 3, vdims, vstr, vbox, "W_UV");
  if (s != MLA_OK) return s;
  // K_c, V_c [128 heads, n, 128] as {128, n, 128 heads}: box 64 x 128 tokens x 1 head (TMA stores)
  const uint64_t odims[3] = {MLA_HEAD_DIM_C, (uint64_t)n, MLA_NUM_HEADS};
  const uint64_t ostr[2] = {MLA_HEAD_DIM_C * 2, (uint64_t)n * MLA_HEAD_DIM_C * 2};
  const uint32_t obox[3] = {64, 128, 1};
  CUtensorMap kcmap, vcmap;
  s = make_map(&kcmap, k_c, 3, odims, ostr, obox, "K_c");
  if (s != MLA_OK) return s;
  s = make_map(&vcmap, v_c, 3, odims, ostr, obox, "V_c");
  if (s != MLA_OK) return s;
  cudaError_t e = mla::launch_expand_kv(amap, kmap, vmap, kcmap, vcmap, n, dev_err, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "expand_kv launch");
  return MLA_OK;
}

// Tensor maps over the packed arrays of a batch (T rows of queries, N cached
// tokens in all) and the attention launch.
static mla_status prefill_attention_launch(const void* q_c, const void* q_r, int64_t T, const void* rows,
                                           const void* k_c, const void* v_c, int64_t N, const mla::PrefillArgs& a,
                                           void* stream) {
  CUtensorMap qm, rm, km, krm, vm;
  const uint32_t box3[3] = {64, 1, 128};
  const uint64_t qd[3] = {MLA_HEAD_DIM_C, MLA_NUM_HEADS, (uint64_t)T};
  const uint64_t qs[2] = {MLA_HEAD_DIM_C * 2, (uint64_t)MLA_HEAD_DIM_C * 2 * MLA_NUM_HEADS};
  const uint64_t rd[3] = {MLA_ROPE_DIM, MLA_NUM_HEADS, (uint64_t)T};
  const uint64_t rs[2] = {MLA_ROPE_DIM * 2, (uint64_t)MLA_ROPE_DIM * 2 * MLA_NUM_HEADS};
  const uint64_t kd[3] = {MLA_HEAD_DIM_C, (uint64_t)N, MLA_NUM_HEADS};   // head-major K_c / V_c
  const uint64_t ks[2] = {MLA_HEAD_DIM_C * 2, (uint64_t)MLA_HEAD_DIM_C * 2 * (uint64_t)N};
  const uint32_t kbox[3] = {64, 128, 1};
  const uint64_t krd[2] = {MLA_TOKEN_ELEMS, (uint64_t)N};
  const uint64_t krs[1] = {(uint64_t)kRowBytes};
  const uint32_t box2[2] = {64, 128};
  mla_status s = make_map(&qm, q_c, 3, qd, qs, box3, "q_c");
  if (s == MLA_OK) s = make_map(&rm, q_r, 3, rd, rs, box3, "q_r");
  if (s == MLA_OK) s = make_map(&km, k_c, 3, kd, ks, kbox, "K_c");
  if (s == MLA_OK) s = make_map(&vm, v_c, 3, kd, ks, kbox, "V_c");
  if (s == MLA_OK) s = make_map(&krm, rows, 2, krd, krs, box2, "k_R rows");
  if (s != MLA_OK) return s;
  cudaError_t e = mla::launch_prefill_attn(qm, rm, km, krm, vm, a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "prefill attention launch");
  return MLA_OK;
}

mla_status mla_prefill_attention(const void* q_c, const void* q_r, int32_t M, const void* rows, const void* k_c,
                                 const void* v_c, int32_t N, float scale, void* out, int32_t* dev_err,
                                 void* stream) {
  if (M < 0 || N < 0) return fail(MLA_ERR_INVALID_ARG, "M = %d, N = %d: negative", M, N);
  if (M == 0) return MLA_OK;
  if (M > N) return fail(MLA_ERR_INVALID_ARG, "M = %d query rows exceed the N = %d cached tokens", M, N);
  if (N > (1 << 24)) return fail(MLA_ERR_INVALID_ARG, "N = %d too large", N);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(MLA_ERR_INVALID_ARG, "scale must be finite and positive");
  CHECK_PTR(q_c);
  CHECK_PTR(q_r);
  CHECK_PTR(rows);
  CHECK_PTR(k_c);
  CHECK_PTR(v_c);
  CHECK_PTR(out);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(q_c);
  CHECK_ALIGN16(q_r);
  CHECK_ALIGN16(rows);
  CHECK_ALIGN16(k_c);
  CHECK_ALIGN16(v_c);
  CHECK_ALIGN16(out);
  if (!aligned(dev_err, 4)) return fail(MLA_ERR_MISALIGNED, "dev_err is not 4-byte aligned");
  mla::PrefillArgs a = {};
  a.nb = 1;
  a.seq[0] = {M, N, 0, 0};
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  a.out = (uint16_t*)out;
  a.dev_err = dev_err;
  return prefill_attention_launch(q_c, q_r, M, rows, k_c, v_c, N, a, stream);
}

mla_status mla_prefill_workspace_size(int32_t N, size_t* bytes) {
  CHECK_PTR(bytes);
  if (N < 0) return fail(MLA_ERR_INVALID_ARG, "N = %d < 0", N);
  *bytes = prefill_ws_bytes(N);
  return MLA_OK;
}

mla_status mla_prefill_batch_workspace_size(const int32_t* n_tokens, int32_t nb, size_t* bytes) {
  CHECK_PTR(bytes);
  if (nb < 0 || nb > mla::kPrefillMaxSeqs)
    return fail(MLA_ERR_INVALID_ARG, "nb = %d outside [0, %d]", nb, mla::kPrefillMaxSeqs);
  if (nb > 0) CHECK_PTR(n_tokens);
  int64_t total = 0;
  for (int32_t i = 0; i < nb; ++i) {
    if (n_tokens[i] < 0) return fail(MLA_ERR_INVALID_ARG, "n_tokens[%d] = %d < 0", i, n_tokens[i]);
    total += n_tokens[i];
  }
  if (total > (1 << 24)) return fail(MLA_ERR_INVALID_ARG, "%lld cached tokens in all: too many", (long long)total);
  *bytes = prefill_ws_bytes(total);
  return MLA_OK;
}

mla_status mla_prefill_decompress_batch(const void* q_c, const void* q_r, const int32_t* seq_ids,
                                        const int32_t* q_starts, const int32_t* q_lens, const int32_t* n_tokens,
                                        int32_t nb, const void* kv_cache, int64_t num_pages,
                                        const int32_t* block_table, int32_t batch, int32_t max_pages,
                                        const void* w_uk, const void* w_uv, float scale, void* workspace,
                                        size_t ws_bytes, void* out, int32_t* dev_err, void* stream) {
  if (nb < 0 || nb > mla::kPrefillMaxSeqs)
    return fail(MLA_ERR_INVALID_ARG, "nb = %d outside [0, %d]", nb, mla::kPrefillMaxSeqs);
  if (nb == 0) return MLA_OK;
  CHECK_PTR(seq_ids);
  CHECK_PTR(q_starts);
  CHECK_PTR(q_lens);
  CHECK_PTR(n_tokens);
  CHECK_PTR(q_c);
  CHECK_PTR(q_r);
  CHECK_PTR(kv_cache);
  CHECK_PTR(block_table);
  CHECK_PTR(w_uk);
  CHECK_PTR(w_uv);
  CHECK_PTR(workspace);
  CHECK_PTR(out);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(q_c);
  CHECK_ALIGN16(q_r);
  CHECK_ALIGN16(kv_cache);
  CHECK_ALIGN16(w_uk);
  CHECK_ALIGN16(w_uv);
  CHECK_ALIGN16(workspace);
  CHECK_ALIGN16(out);
  if (!aligned(block_table, 4) || !aligned(dev_err, 4))
    return fail(MLA_ERR_MISALIGNED, "block_table and dev_err must be 4-byte aligned");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(MLA_ERR_INVALID_ARG, "scale must be finite and positive");
  if (num_pages < 1 || batch < 1 || max_pages < 1) return fail(MLA_ERR_INVALID_ARG, "bad pool/table sizes");
  mla::GatherBatch g = {};
  mla::PrefillArgs a = {};
  int64_t total = 0, rows_end = 0;
  for (int32_t i = 0; i < nb; ++i) {
    const int32_t b = seq_ids[i], M = q_lens[i], N = n_tokens[i], q0 = q_starts[i];
    if (b < 0 || b >= batch) return fail(MLA_ERR_INVALID_ARG, "seq_ids[%d] = %d outside [0, %d)", i, b, batch);
    if (M < 1 || N < M)
      return fail(MLA_ERR_INVALID_ARG, "sequence %d: q_len %d must be in [1, n_tokens = %d]", i, M, N);
    if ((N + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE > max_pages)
      return fail(MLA_ERR_INVALID_ARG, "sequence %d: %d tokens need more than max_pages = %d pages", i, N, max_pages);
    if (q0 < 0) return fail(MLA_ERR_INVALID_ARG, "q_starts[%d] = %d < 0", i, q0);
    g.b[i] = b;
    g.n[i] = N;
    g.off[i] = total;
    a.seq[i] = {M, N, q0, (int32_t)total};
    total += N;
    rows_end = std::max<int64_t>(rows_end, (int64_t)q0 + M);
  }
  if (total > (1 << 24)) return fail(MLA_ERR_INVALID_ARG, "%lld cached tokens in all: too many", (long long)total);
  if (rows_end > (1 << 24)) return fail(MLA_ERR_INVALID_ARG, "query rows past 2^24");
  if (ws_bytes < prefill_ws_bytes(total))
    return fail(MLA_ERR_INVALID_ARG, "workspace holds %zu bytes, %lld cached tokens need %zu", ws_bytes,
                (long long)total, prefill_ws_bytes(total));
  g.nb = nb;
  g.total = total;
  a.nb = nb;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  a.out = (uint16_t*)out;
  a.dev_err = dev_err;
  uint8_t* ws = (uint8_t*)workspace;
  void* rows = ws;
  void* k_c = ws + prefill_rows_bytes(total);
  void* v_c = (uint8_t*)k_c + (size_t)total * MLA_NUM_HEADS * MLA_HEAD_DIM_C * 2;
  cudaError_t e = mla::launch_gather_batch((const uint16_t*)kv_cache, num_pages, block_table, max_pages, g,
                                           (uint16_t*)rows, dev_err, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "batched gather launch");
  mla_status s = mla_expand_kv(rows, (int32_t)total, w_uk, w_uv, k_c, v_c, dev_err, stream);
  if (s != MLA_OK) return s;
  return prefill_attention_launch(q_c, q_r, rows_end, rows, k_c, v_c, total, a, stream);
}

mla_status mla_prefill_decompress(const void* q_c, const void* q_r, int32_t M, const void* kv_cache, int64_t num_pages,
                                  const int32_t* block_table, int32_t max_pages, int32_t b, int32_t N,
                                  const void* w_uk, const void* w_uv, float scale, void* workspace, size_t ws_bytes,
                                  void* out, int32_t* dev_err, void* stream) {
  if (M < 0 || N < 0) return fail(MLA_ERR_INVALID_ARG, "M = %d, N = %d: negative", M, N);
  if (M == 0) return MLA_OK;
  if (M > N) return fail(MLA_ERR_INVALID_ARG, "M = %d query rows exceed the N = %d cached tokens", M, N);
  if (b < 0) return fail(MLA_ERR_INVALID_ARG, "b = %d < 0", b);
  const int32_t zero = 0;
  // one sequence: its block-table row b, its query rows at the start of q_c / q_r / out
  return mla_prefill_decompress_batch(q_c, q_r, &b, &zero, &M, &N, 1, kv_cache, num_pages, block_table, b + 1,
                                      max_pages, w_uk, w_uv, scale, workspace, ws_bytes, out, dev_err, stream);
}

mla_status mla_absorb_q(const void* q_c, const void* w_uk, void* q_abs, int32_t T, int32_t* dev_err, void* stream) {
  return head_gemm(mla::HeadGemm::kAbsorbQ, q_c, w_uk, q_abs, T, dev_err, stream);
}

mla_status mla_up_v(const void* o_lat, const void* w_uv, void* out, int32_t T, int32_t* dev_err, void* stream) {
  return head_gemm(mla::HeadGemm::kUpV, o_lat, w_uv, out, T, dev_err, stream);
}

// ------------------------------------------------------------------ decode
mla_status mla_decode_max_clusters(int32_t* out) {
  CHECK_PTR(out);
  int n = 0;
  cudaError_t e = mla::decode_max_clusters(&n);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
  if (n < 1) return fail(MLA_ERR_CUDA, "the decode kernel cannot be resident on this device");
  *out = n;
  return MLA_OK;
}

mla_status mla_decode_plan_bytes(int32_t T, int32_t num_clusters, size_t* bytes) {
  CHECK_PTR(bytes);
  if (T < 0 || num_clusters < 1) return fail(MLA_ERR_INVALID_ARG, "need T >= 0 and num_clusters >= 1");
  const mla::PlanLayout L = mla::plan_layout(num_clusters, mla::plan_max_segments(T, num_clusters),
                                             mla::plan_max_split_rows(T, num_clusters));
  *bytes = (size_t)L.words * 4;
  return MLA_OK;
}

mla_status mla_decode_workspace_size(int32_t num_clusters, size_t* bytes) {
  CHECK_PTR(bytes);
  if (num_clusters < 1) return fail(MLA_ERR_INVALID_ARG, "num_clusters = %d < 1", num_clusters);
  *bytes = workspace_bytes_for(mla::plan_max_partials(num_clusters));
  return MLA_OK;
}

mla_status mla_decode_plan_host(const int32_t* seq_lens, const int32_t* q_lens, int32_t B, int32_t num_clusters,
                                void* plan_host, size_t plan_bytes, mla_plan_info* info) {
  CHECK_PTR(plan_host);
  CHECK_PTR(info);
  if (!aligned(plan_host, 4)) return fail(MLA_ERR_MISALIGNED, "plan_host is not 4-byte aligned");
  return build_plan(seq_lens, q_lens, B, num_clusters, (int32_t*)plan_host, plan_bytes / 4, info);
}

mla_status mla_decode_plan(const int32_t* seq_lens_host, const int32_t* q_lens_host, int32_t B, int32_t num_clusters,
                           void* plan_dev, size_t plan_bytes, mla_plan_info* info, void* stream) {
  CHECK_PTR(plan_dev);
  CHECK_PTR(info);
  CHECK_ALIGN16(plan_dev);
  std::vector<int32_t> host(plan_bytes / 4);
  mla_status s = build_plan(seq_lens_host, q_lens_host, B, num_clusters, host.data(), host.size(), info);
  if (s != MLA_OK) return s;
  // Pageable source: the call returns once the data is staged, so `host` may go.
  cudaError_t e = cudaMemcpyAsync(plan_dev, host.data(), info->plan_bytes, cudaMemcpyHostToDevice,
                                  (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "plan copy");
  return MLA_OK;
}

static mla_status decode_common(const void* q_abs, const void* q_r, const void* kv_cache, const float* kv_scales,
                                int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                const void* plan_dev, const mla_plan_info* info, float scale, void* workspace,
                                size_t ws_bytes, void* o_lat, float* lse, int32_t* dev_err, void* stream,
                                bool fp8) {
  CHECK_PTR(info);
  if (info->magic != MLA_PLAN_MAGIC) return fail(MLA_ERR_INVALID_ARG, "info is not a decode plan summary");
  if (info->T == 0 || info->num_clusters == 0) return MLA_OK;
  CHECK_PTR(q_abs);
  CHECK_PTR(q_r);
  CHECK_PTR(kv_cache);
  CHECK_PTR(block_table);
  CHECK_PTR(plan_dev);
  CHECK_PTR(o_lat);
  CHECK_PTR(dev_err);
  CHECK_ALIGN16(q_abs);
  CHECK_ALIGN16(q_r);
  CHECK_ALIGN16(kv_cache);
  CHECK_ALIGN16(plan_dev);
  CHECK_ALIGN16(o_lat);
  if (fp8) {
    CHECK_PTR(kv_scales);
    CHECK_ALIGN16(kv_scales);
  }
  if (!aligned(block_table, 4) || !aligned(dev_err, 4) || (lse && !aligned(lse, 4)))
    return fail(MLA_ERR_MISALIGNED, "block_table, dev_err and lse must be 4-byte aligned");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(MLA_ERR_INVALID_ARG, "scale must be finite and positive");
  if (num_pages < 1 || num_pages * MLA_PAGE_SIZE > (int64_t)INT32_MAX)
    return fail(MLA_ERR_INVALID_ARG, "num_pages = %lld outside [1, 2^31/64)", (long long)num_pages);
  if (max_pages < info->max_pages_needed)
    return fail(MLA_ERR_INVALID_ARG, "block table has %d columns, the plan reads %d", max_pages,
                info->max_pages_needed);
  const size_t need_ws = workspace_bytes_for(info->num_partials);
  if (info->num_partials > 0) {
    CHECK_PTR(workspace);
    CHECK_ALIGN16(workspace);
    if (ws_bytes < need_ws)
      return fail(MLA_ERR_INVALID_ARG, "workspace holds %zu bytes, the plan needs %zu", ws_bytes, need_ws);
  }

  CUtensorMap kv_map, rope_map;
  mla_status s;
  if (fp8) {
    // Codes: a CTA's 256 of each token row, 64 rows per box (no swizzle: the
    // converters read them); RoPE halves as bf16 columns 256.. of the rows.
    const uint64_t cdims[2] = {MLA_FP8_ROW_BYTES, (uint64_t)num_pages * MLA_PAGE_SIZE};
    const uint64_t cstr[1] = {MLA_FP8_ROW_BYTES};
    const uint32_t cbox[2] = {256, 64};
    s = make_map(&kv_map, kv_cache, 2, cdims, cstr, cbox, "fp8 codes", CU_TENSOR_MAP_SWIZZLE_NONE,
                 CU_TENSOR_MAP_DATA_TYPE_UINT8);
    if (s != MLA_OK) return s;
    const uint64_t rdims[2] = {MLA_FP8_ROW_BYTES / 2, (uint64_t)num_pages * MLA_PAGE_SIZE};
    const uint32_t rope_box[2] = {32, 64};
    s = make_map(&rope_map, kv_cache, 2, rdims, cstr, rope_box, "fp8 RoPE halves", CU_TENSOR_MAP_SWIZZLE_64B);
    if (s != MLA_OK) return s;
  } else {
    // Latent part as a 3D view {64 elements, token, 64-element chunk}: one box
    // of 4 chunks x 64 tokens lands as 4 consecutive 128-byte-swizzled 8 KB
    // tiles, one TMA instruction per page for a CTA's latent half.
    const uint64_t ldims[3] = {64, (uint64_t)num_pages * MLA_PAGE_SIZE, MLA_LATENT_DIM / 64};
    const uint64_t lstr[2] = {(uint64_t)kRowBytes, 128};
    const uint32_t lbox[3] = {64, 64, 4};
    s = make_map(&kv_map, kv_cache, 3, ldims, lstr, lbox, "kv_cache latent chunks");
    if (s != MLA_OK) return s;
    const uint64_t dims[2] = {MLA_TOKEN_ELEMS, (uint64_t)num_pages * MLA_PAGE_SIZE};
    const uint64_t str[1] = {(uint64_t)kRowBytes};
    const uint32_t rope_box[2] = {32, 64};
    s = make_map(&rope_map, kv_cache, 2, dims, str, rope_box, "kv_cache RoPE halves", CU_TENSOR_MAP_SWIZZLE_64B);
    if (s != MLA_OK) return s;
  }

  const mla::PlanLayout L = mla::plan_layout(info->num_clusters, info->num_segments, info->num_split_rows);
  const int32_t* plan = (const int32_t*)plan_dev;
  float* part_o = (float*)workspace;
  float* part_lse = part_o ? part_o + (size_t)info->num_partials * MLA_NUM_HEADS * MLA_LATENT_DIM : nullptr;

  mla::DecodeArgs a = {};
  a.q_abs = (const uint16_t*)q_abs;
  a.q_r = (const uint16_t*)q_r;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.seg_off = plan + L.seg_off;
  a.segs = plan + L.seg_base;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  a.o_lat = (uint16_t*)o_lat;
  a.lse = lse;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.dev_err = dev_err;
  a.T = info->T;
  a.B = info->B;
  a.num_segments = info->num_segments;
  a.num_partials = info->num_partials;
  a.kv_scales = fp8 ? kv_scales : nullptr;
  a.wait_limit = g_decode_wait_limit.load(std::memory_order_relaxed);
  a.wait_every = a.wait_limit < (1ull << 20) ? 0u : 255u;
  cudaError_t e = mla::launch_decode(kv_map, rope_map, a, info->num_clusters, fp8, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  if (info->num_split_rows > 0) {
    mla::CombineArgs c = {};
    c.split_rows = plan + L.split_base;
    c.part_o = part_o;
    c.part_lse = part_lse;
    c.o_lat = (uint16_t*)o_lat;
    c.lse = lse;
    c.T = info->T;
    c.num_partials = info->num_partials;
    c.dev_err = dev_err;
    e = mla::launch_combine(c, info->num_split_rows, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  }
  return MLA_OK;
}

mla_status mla_decode_paged(const void* q_abs, const void* q_r, const void* kv_cache, int64_t num_pages,
                            const int32_t* block_table, int32_t max_pages, const void* plan_dev,
                            const mla_plan_info* info, float scale, void* workspace, size_t ws_bytes, void* o_lat,
                            float* lse, int32_t* dev_err, void* stream) {
  return decode_common(q_abs, q_r, kv_cache, nullptr, num_pages, block_table, max_pages, plan_dev, info, scale,
                       workspace, ws_bytes, o_lat, lse, dev_err, stream, false);
}

mla_status mla_decode_paged_fp8(const void* q_abs, const void* q_r, const void* rows, const float* scales,
                                int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                const void* plan_dev, const mla_plan_info* info, float scale, void* workspace,
                                size_t ws_bytes, void* o_lat, float* lse, int32_t* dev_err, void* stream) {
  return decode_common(q_abs, q_r, rows, scales, num_pages, block_table, max_pages, plan_dev, info, scale,
                       workspace, ws_bytes, o_lat, lse, dev_err, stream, true);
}

mla_status mla_debug_set_decode_wait_limit(uint64_t cycles) {
  if (cycles > kDefaultDecodeWaitLimit)
    return fail(MLA_ERR_INVALID_ARG, "wait limit %llu above the default %llu", (unsigned long long)cycles,
                (unsigned long long)kDefaultDecodeWaitLimit);
  g_decode_wait_limit.store(cycles == 0 ? kDefaultDecodeWaitLimit : cycles, std::memory_order_relaxed);
  return MLA_OK;
}

mla_status mla_check(void* stream, const int32_t* dev_err, int32_t* word_out) {
  CHECK_PTR(dev_err);
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int32_t w = 0;
  e = cudaMemcpy(&w, dev_err, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (word_out) *word_out = w;
  if (w == 0) return MLA_OK;
  if (w & MLA_DEVERR_TIMEOUT) return fail(MLA_ERR_TIMEOUT, "a kernel wait timed out (device error word 0x%x)", w);
  return fail(MLA_ERR_DEVICE, "device error word 0x%x", w);
}

}  // extern "C"
