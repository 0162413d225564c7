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

// The same split as mla_decode_plan (requests end to end in page units, worker w takes pages
// [w * quota, (w + 1) * quota), pieces cut at request boundaries and at `cap` pages), written
// straight into static arrays. Returns the segment count, or -1 if it exceeds kMaxSegments.
int64_t split_static(const int32_t* indptr, const int32_t* len, int batch, int workers, int min_splits,
                     Segment* segs, int32_t* wptr, int32_t* rptr, int32_t* wide, qkvp_plan* plan) {
  int64_t total = 0, tokens = 0;
  for (int r = 0; r < batch; ++r) {
    total += (static_cast<int64_t>(len[r]) + kPage - 1) / kPage;
    tokens += len[r];
  }
  const int64_t quota = total > 0 ? (total + workers - 1) / workers : 0;
  int64_t cap = quota;
  if (min_splits > 0 && total > 0) cap = std::max<int64_t>(1, std::min<int64_t>(quota, total / min_splits));
  int64_t n = 0, start_r = 0;
  int r = 0;
  int32_t max_pages = 0, min_pages = total > 0 ? INT32_MAX : 0;
  for (int w = 0; w < workers; ++w) {
    wptr[w] = static_cast<int32_t>(n);
    const int64_t a = std::min(total, w * quota), b = std::min(total, (w + 1) * quota);
    max_pages = std::max<int32_t>(max_pages, static_cast<int32_t>(b - a));
    if (total > 0) min_pages = std::min<int32_t>(min_pages, static_cast<int32_t>(b - a));
    int64_t x = a;
    while (x < b) {
      while (r < batch && start_r + (static_cast<int64_t>(len[r]) + kPage - 1) / kPage <= x) {
        start_r += (static_cast<int64_t>(len[r]) + kPage - 1) / kPage;
        ++r;
      }
      const int64_t end_r = start_r + (static_cast<int64_t>(len[r]) + kPage - 1) / kPage;
      const int64_t y = std::min(b, end_r);
      for (int64_t c = x; c < y; c += cap) {
        if (n >= kMaxSegments) return -1;
        const int64_t e = std::min(y, c + cap);
        Segment g{};
        g.req = r;
        g.page_begin = static_cast<int32_t>(indptr[r] + (c - start_r));
        g.num_pages = static_cast<int32_t>(e - c);
        g.num_tokens = static_cast<int32_t>(std::min<int64_t>(len[r], (e - start_r) * kPage) - (c - start_r) * kPage);
        segs[n++] = g;
      }
      x = y;
    }
  }
  wptr[workers] = static_cast<int32_t>(n);
  int64_t k = 0;
  int32_t part = 0, split = 0, empty = 0, most = 0, nwide = 0;
  for (int q = 0; q < batch; ++q) {
    rptr[q] = static_cast<int32_t>(k);
    const int64_t k0 = k;
    while (k < n && segs[k].req == q) ++k;
    if (k == k0) ++empty;
    if (k - k0 >= 2) ++split;
    most = std::max<int32_t>(most, static_cast<int32_t>(k - k0));
    if (k - k0 > kCombineWideSegs) wide[nwide++] = q;
    for (int64_t i = k0; i < k; ++i) segs[i].partial = (k - k0 == 1) ? -1 : part++;
  }
  rptr[batch] = static_cast<int32_t>(k);
  plan->num_segments = static_cast<int32_t>(n);
  plan->num_split_requests = split;
  plan->num_empty_requests = empty;
  plan->num_partials = part;
  plan->max_request_segments = most;
  plan->num_wide_requests = nwide;
  plan->max_worker_pages = max_pages;
  plan->min_worker_pages = min_pages;
  plan->total_pages = total;
  plan->total_tokens = tokens;
  return n;
}

}  // namespace

extern "C" int mla_decode_noalloc(const int32_t* kv_indptr_host, const int32_t* kv_len_host, int32_t batch,
                                  int32_t num_heads, int32_t kv_dtype, int32_t num_sms, int32_t min_splits,
                                  const void* q, const void* kv_data, const uint8_t* kv_scale,
                                  int64_t num_pages, const int32_t* kv_indices, float sm_scale,
                                  float global_scale, void* out, float* lse, qkvp_stream_t stream) {
  // the same argument checks as mla_decode_plan, plus the fixed capacity of the scratch
  if (batch < 0 || min_splits < 0) return QKVP_E_INVALID;
  if (batch > 0 && (!kv_indptr_host || !kv_len_host)) return QKVP_E_INVALID;
  if (num_heads < 16 || num_heads > 128 || num_heads % 16) return QKVP_E_UNSUPPORTED;
  if (kv_dtype != QKVP_KV_FP8_E4M3 && kv_dtype != QKVP_KV_NVFP4 && kv_dtype != QKVP_KV_BF16 &&
      kv_dtype != QKVP_KV_FP8_PER_TOKEN)
    return QKVP_E_UNSUPPORTED;
  if (batch > kMaxBatch) return QKVP_E_WORKSPACE;
  if (batch > 0 && kv_indptr_host[0] != 0) return QKVP_E_INVALID;
  for (int r = 0; r < batch; ++r) {
    const int64_t np = static_cast<int64_t>(kv_indptr_host[r + 1]) - kv_indptr_host[r];
    if (np < 0 || kv_len_host[r] < 0) return QKVP_E_INVALID;
    if ((static_cast<int64_t>(kv_len_host[r]) + kPage - 1) / kPage > np) return QKVP_E_INVALID;
  }
  int dev = 0;
  if (num_sms <= 0) {
    if (cudaGetDevice(&dev) != cudaSuccess) return QKVP_E_CUDA;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return QKVP_E_CUDA;
  }
  const int hc = mma_heads_per_cta(num_heads);
  if (hc == 0) return QKVP_E_UNSUPPORTED;
  const int cpw = num_heads / hc;
  const int workers = std::min(kMaxWorkers, std::max(1, num_sms / cpw));

  std::lock_guard<std::mutex> lock(g_mutex);
  // Lay the table out in static host storage exactly as mla_decode_run reads it. The segment count
  // is bounded by kMaxSegments before the layout is known, so stage segments first, then place the
  // worker and request ranges behind them.
  static Segment segs[kMaxSegments];
  static int32_t wptr[kMaxWorkers + 1];
  static int32_t rptr[kMaxBatch + 1];
  static int32_t wide[kMaxBatch];
  qkvp_plan plan;
  std::memset(&plan, 0, sizeof(plan));
  const int64_t nseg = split_static(kv_indptr_host, kv_len_host, batch, workers, min_splits, segs, wptr, rptr, wide,
                                    &plan);
  if (nseg < 0) return QKVP_E_WORKSPACE;
  const TableLayout t = table_layout(nseg, workers, batch);
  plan.batch = batch;
  plan.num_heads = num_heads;
  plan.page_size = kPage;
  plan.kv_dtype = kv_dtype;
  plan.algo = QKVP_ALGO_MMA_SYNC;
  plan.num_workers = workers;
  plan.ctas_per_worker = cpw;
  plan.table_bytes = t.bytes;
  plan.status_offset = t.status;
  plan.partial_o_offset = t.bytes;
  plan.partial_lse_offset = t.bytes + align_up(static_cast<uint64_t>(plan.num_partials) * num_heads * kDv * 4);
  plan.workspace_bytes = plan.partial_lse_offset + align_up(static_cast<uint64_t>(plan.num_partials) * num_heads * 4);
  if (plan.workspace_bytes > kScratchBytes || t.bytes > sizeof(g_table)) return QKVP_E_WORKSPACE;
  plan.magic = kPlanMagic;
  std::memset(g_table, 0, t.bytes);
  if (nseg > 0) std::memcpy(g_table + t.segs, segs, nseg * sizeof(Segment));
  std::memcpy(g_table + t.wptr, wptr, (workers + 1) * 4);
  std::memcpy(g_table + t.rptr, rptr, (batch + 1) * 4);
  if (plan.num_wide_requests > 0) std::memcpy(g_table + t.wide, wide, plan.num_wide_requests * 4);

  // Set-up, once per device, with that device current: the device address of the scratch.
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QKVP_E_CUDA;
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return QKVP_E_CUDA;
    g_scratch_addr[dev] = p;
  }
  void* scratch = g_scratch_addr[dev];
  // g_table is pageable: the runtime stages it before this call returns, so the next caller may
  // overwrite it as soon as the lock is released.
  if (cudaMemcpyAsync(scratch, g_table, t.bytes, cudaMemcpyHostToDevice,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return QKVP_E_CUDA;
  return mla_decode_run(&plan, q, kv_data, kv_scale, num_pages, kv_indices, sm_scale, global_scale, out,
                        lse, scratch, kScratchBytes, stream);
}
