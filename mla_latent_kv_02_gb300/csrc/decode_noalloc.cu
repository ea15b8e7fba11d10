// mla_decode_paged_noalloc: the decode step (A3 + A4) for callers that cannot
// allocate device memory.
//
// The regular entry point needs two caller-owned device buffers besides the
// inputs and outputs: the split plan and the split-KV workspace.  Some
// callers cannot provide them: a plugin that a host framework hands only its
// input and output tensors, an engine whose memory pool has reserved all free
// device memory at start-up (a cudaMalloc would fail, or fragment the pool
// and break its accounting), or a runtime that forbids allocation after
// initialisation.  This variant keeps both buffers in one file-scope device
// array, reserved when the library is loaded and held by every GPU that loads
// it until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/mla.h"
#include "internal.h"

namespace {

constexpr size_t kPlanArea = MLA_NOALLOC_PLAN_BYTES;
constexpr size_t kWorkArea = MLA_NOALLOC_WORKSPACE_BYTES;

// Plan words first, then fp32 partial outputs and their log-sum-exp.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kPlanArea + kWorkArea];

constexpr int kMaxDevices = 64;
struct DeviceScratch {
  bool ready = false;
  unsigned char* ptr = nullptr;  // device address of g_noalloc_scratch on that device
  int32_t max_clusters = 0;
};
std::mutex g_mutex;  // guards the per-device table and the host plan buffer
DeviceScratch g_devices[kMaxDevices];
int32_t g_host_plan[kPlanArea / sizeof(int32_t)];  // host staging of the plan

}  // namespace

extern "C" mla_status mla_decode_paged_noalloc(const void* q_abs, const void* q_r, const void* kv_cache,
                                               int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                               const int32_t* seq_lens_host, const int32_t* q_lens_host, int32_t B,
                                               float scale, void* o_lat, float* lse, int32_t* dev_err,
                                               void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mla::set_last_error(MLA_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return mla::set_last_error(MLA_ERR_UNSUPPORTED, "device ordinal above 63");
  if (B < 0) return mla::set_last_error(MLA_ERR_INVALID_ARG, "B is negative");
  if (B > 0 && (seq_lens_host == nullptr || q_lens_host == nullptr))
    return mla::set_last_error(MLA_ERR_INVALID_ARG, "seq_lens_host and q_lens_host are required");

  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceScratch& ds = g_devices[dev];
  if (!ds.ready) {
    // Set-up, once per device, with that device current: the host-side name
    // of the array is not a device address, so ask the runtime for it.
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return mla::set_last_error(MLA_ERR_CUDA, "cudaGetSymbolAddress of the no-alloc scratch failed");
    int32_t nc = 0;
    mla_status s = mla_decode_max_clusters(&nc);
    if (s != MLA_OK) return s;
    ds.ptr = static_cast<unsigned char*>(p);
    ds.max_clusters = nc;
    ds.ready = true;
  }

  int64_t T = 0;
  for (int32_t b = 0; b < B; ++b) T += q_lens_host[b] > 0 ? q_lens_host[b] : 0;
  if (T > INT32_MAX) return mla::set_last_error(MLA_ERR_INVALID_ARG, "too many query rows");

  // Fewest clusters that still fit: halve the cluster count until the plan's
  // split partials fit the workspace area (one cluster never splits a row).
  mla_plan_info info;
  for (int32_t nc = ds.max_clusters;; nc = nc > 1 ? nc / 2 : 0) {
    if (nc == 0) return mla::set_last_error(MLA_ERR_INVALID_ARG, "no plan fits the no-alloc scratch");
    size_t plan_bytes = 0;
    mla_status s = mla_decode_plan_bytes((int32_t)T, nc, &plan_bytes);
    if (s != MLA_OK) return s;
    if (plan_bytes > kPlanArea) {
      if (nc > 1) continue;
      char msg[200];
      snprintf(msg, sizeof(msg), "%lld query rows need a %zu-byte plan; the no-alloc scratch holds %zu",
               (long long)T, plan_bytes, kPlanArea);
      return mla::set_last_error(MLA_ERR_INVALID_ARG, msg);
    }
    s = mla_decode_plan_host(seq_lens_host, q_lens_host, B, nc, g_host_plan, sizeof(g_host_plan), &info);
    if (s != MLA_OK) return s;
    size_t ws = 0;
    if (info.num_partials > 0) {
      ws = (size_t)info.num_partials * (MLA_NUM_HEADS * MLA_LATENT_DIM * 4 + MLA_NUM_HEADS * 4);
      if (ws > kWorkArea) continue;
    }
    break;
  }
  if (info.T == 0 || info.num_clusters == 0) return MLA_OK;
  // Pageable source: the copy is staged before the call returns.
  e = cudaMemcpyAsync(ds.ptr, g_host_plan, info.plan_bytes, cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e != cudaSuccess) return mla::set_last_error(MLA_ERR_CUDA, "copying the plan into the no-alloc scratch failed");
  return mla_decode_paged(q_abs, q_r, kv_cache, num_pages, block_table, max_pages, ds.ptr, &info, scale,
                          ds.ptr + kPlanArea, kWorkArea, o_lat, lse, dev_err, stream);
}
