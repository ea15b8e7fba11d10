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
//
// The plan is built on the host and handed to the device inside the launch
// parameters of a small copy kernel (at most kChunkWords words per launch),
// so no host memory is read after the call returns and the host never waits
// for the stream.
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

// One launch's share of the plan, passed by value (the parameter space of a
// launch holds up to 32 764 bytes).
constexpr int kChunkWords = 7936;
struct PlanChunk {
  int32_t offset;  // first word of the plan this chunk carries
  int32_t count;   // words in this chunk
  int32_t words[kChunkWords];
};
static_assert(sizeof(PlanChunk) + sizeof(void*) <= 32764, "plan chunk exceeds the launch parameter space");

__global__ void __launch_bounds__(256) plan_copy_kernel(const __grid_constant__ PlanChunk c, int32_t* dst) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < c.count; i += gridDim.x * blockDim.x)
    dst[c.offset + i] = c.words[i];
}

constexpr int kMaxDevices = 64;
struct DeviceScratch {
  bool ready = false;
  unsigned char* ptr = nullptr;  // device address of g_noalloc_scratch on that device
  int32_t max_clusters = 0;
  mla_plan_info last = {};       // summary of the last plan this device ran
};
std::mutex g_mutex;  // guards the per-device table, the host plan buffer and the chunk
DeviceScratch g_devices[kMaxDevices];
int32_t g_host_plan[kPlanArea / sizeof(int32_t)];  // the plan as built on the host
PlanChunk g_chunk;                                  // staging of one launch's parameters

size_t workspace_for(int32_t partials) {
  return (size_t)partials * (MLA_NUM_HEADS * MLA_LATENT_DIM * 4 + MLA_NUM_HEADS * 4);
}

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

  // The most clusters whose plan fits: the plan area, and the split partials
  // in the workspace area.  Counts are tried from the most down (a host plan
  // is cheap: linear in rows + clusters); one cluster never splits a row, so
  // the descent ends whenever the plan area holds the rows at all.
  mla_plan_info info;
  bool found = false;
  for (int32_t nc = ds.max_clusters; nc >= 1 && !found; --nc) {
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
    found = workspace_for(info.num_partials) <= kWorkArea;
  }
  if (!found) return mla::set_last_error(MLA_ERR_INVALID_ARG, "no plan fits the no-alloc scratch");
  if (info.T == 0 || info.num_clusters == 0) {
    ds.last = info;
    return MLA_OK;
  }
  // The plan into the array: its words ride in the launch parameters.
  const int32_t words = (int32_t)(info.plan_bytes / sizeof(int32_t));
  for (int32_t off = 0; off < words; off += kChunkWords) {
    g_chunk.offset = off;
    g_chunk.count = words - off < kChunkWords ? words - off : kChunkWords;
    for (int32_t i = 0; i < g_chunk.count; ++i) g_chunk.words[i] = g_host_plan[off + i];
    plan_copy_kernel<<<(g_chunk.count + 255) / 256, 256, 0, (cudaStream_t)stream>>>(
        g_chunk, reinterpret_cast<int32_t*>(ds.ptr));
    e = cudaGetLastError();
    if (e != cudaSuccess)
      return mla::set_last_error(MLA_ERR_CUDA, "copying the plan into the no-alloc scratch failed");
  }
  mla_status s = mla_decode_paged(q_abs, q_r, kv_cache, num_pages, block_table, max_pages, ds.ptr, &info, scale,
                                  ds.ptr + kPlanArea, kWorkArea, o_lat, lse, dev_err, stream);
  if (s == MLA_OK) ds.last = info;
  return s;
}

extern "C" mla_status mla_debug_noalloc_last_plan(mla_plan_info* out) {
  if (out == nullptr) return mla::set_last_error(MLA_ERR_INVALID_ARG, "out is NULL");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return mla::set_last_error(MLA_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return mla::set_last_error(MLA_ERR_UNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_devices[dev].ready) return mla::set_last_error(MLA_ERR_INVALID_ARG, "no no-alloc call on this device yet");
  *out = g_devices[dev].last;
  return MLA_OK;
}
