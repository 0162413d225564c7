// mla_decode_noalloc: plan + decode for callers that cannot allocate device memory.
//
// Some callers have no way to provide a workspace: a serving loop that has handed every free byte
// of the GPU to a pre-sized KV pool, or a latency-critical decode step that must not risk the
// device-wide synchronisation a cudaMalloc can bring. For them the split-KV scratch (work table
// plus FP32 partials) lives in one fixed file-scope device array. Every GPU that loads the library
// holds this array until the process exits. The call allocates nothing: no cudaMalloc or cudaFree,
// no allocating library routine, no host heap (the host-side table is staged in static storage
// under a mutex). It then hands the array to the ordinary mla_decode_run as its workspace.
//
// The array keeps whatever the last call left in it. Nothing in it has to start at zero: each call
// uploads its own table and every partial is written before it is read. Calls whose GPU work
// overlaps (two streams, two host threads) share the one array and race on it.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/qkvp.h"
#include "qkvp_internal.h"

using namespace qkvp;

namespace {

constexpr uint64_t kScratchBytes = QKVP_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxBatch = QKVP_NOALLOC_MAX_BATCH;
constexpr int kMaxWorkers = 1024;
constexpr int kMaxSegments = QKVP_NOALLOC_MAX_SEGMENTS;
constexpr int kMaxDevices = 64;

// The scratch. In host code `g_scratch` is only a stand-in for the symbol, never a device address:
// host code passes the address that cudaGetSymbolAddress returned for the current device.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mutex;                     // guards the static host staging and the address cache
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_scratch, per device
uint8_t g_table[kMaxSegments * sizeof(Segment) + (kMaxWorkers + 1) * 4 + (kMaxBatch + 1) * 4 + kMaxBatch * 4 +
                4 * 256];

}  // namespace

extern "C" int mla_decode_noalloc(const int32_t* kv_indptr_host, const int32_t* kv_len_host, int32_t batch,
                                  int32_t num_heads, int32_t kv_dtype, int32_t num_sms, int32_t min_splits,
                                  const void* q, const void* kv_data, const uint8_t* kv_scale,
                                  int64_t num_pages, const int32_t* kv_indices, float sm_scale,
                                  float global_scale, void* out, float* lse, qkvp_stream_t stream) {
  // the argument checks of mla_decode_plan, plus the fixed capacity of the scratch
  if (batch > kMaxBatch) return QKVP_E_WORKSPACE;
  int st = check_plan_args(kv_indptr_host, kv_len_host, batch, num_heads, kPage, kv_dtype, min_splits);
  if (st != QKVP_OK) return st;
  int dev = 0;
  if (num_sms <= 0) {
    if (cudaGetDevice(&dev) != cudaSuccess) return QKVP_E_CUDA;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return QKVP_E_CUDA;
  }
  const int hc = mma_heads_per_cta(num_heads);
  if (hc == 0) return QKVP_E_UNSUPPORTED;
  const int cpw = num_heads / hc;
  // the same worker count as mla_decode_plan for this kernel family (capped by the static arrays)
  const int workers = std::max(1, num_sms / cpw);
  if (workers > kMaxWorkers) return QKVP_E_WORKSPACE;

  std::lock_guard<std::mutex> lock(g_mutex);
  // The planner of mla_decode_plan, writing into static storage: the same segments, in the same order.
  static Segment segs[kMaxSegments];
  static int32_t wptr[kMaxWorkers + 1];
  static int32_t rptr[kMaxBatch + 1];
  static int32_t wide[kMaxBatch];
  const SplitOut table{segs, kMaxSegments, wptr, rptr, wide};
  SplitInfo info;
  if (!split_pages(kv_indptr_host, kv_len_host, batch, workers, min_splits, table, info)) return QKVP_E_WORKSPACE;
  qkvp_plan plan;
  std::memset(&plan, 0, sizeof(plan));
  fill_plan(&plan, info, batch, num_heads, kv_dtype, QKVP_ALGO_MMA_SYNC, workers, cpw);
  if (plan.workspace_bytes > kScratchBytes || plan.table_bytes > sizeof(g_table)) return QKVP_E_WORKSPACE;
  plan.magic = kPlanMagic;
  write_table(g_table, table, info, workers, batch);
  // The table upload below reads g_table, which the next call overwrites: a captured graph would
  // replay whatever the last call left there. The call is refused during capture.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cap) != cudaSuccess) return QKVP_E_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return QKVP_E_UNSUPPORTED;

  // Set-up, once per device, with that device current: the device address of the scratch.
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QKVP_E_CUDA;
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return QKVP_E_CUDA;
    g_scratch_addr[dev] = p;
  }
  void* scratch = g_scratch_addr[dev];
  // g_table is pageable: the runtime stages it before this call returns (after the stream's earlier
  // work has drained), so the next caller may overwrite it as soon as the lock is released.
  if (cudaMemcpyAsync(scratch, g_table, plan.table_bytes, cudaMemcpyHostToDevice,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return QKVP_E_CUDA;
  return mla_decode_run(&plan, q, kv_data, kv_scale, num_pages, kv_indices, sm_scale, global_scale, out,
                        lse, scratch, kScratchBytes, stream);
}
