// libqkvp C ABI: argument checks, the split-KV planner and kernel dispatch.
//
// Nothing here allocates device memory. mla_decode_plan builds its work table on the host (the
// split itself is in split.cu) and copies it into the caller's workspace with one asynchronous copy
// on the caller's stream, staged through library-owned pinned buffers.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/qkvp.h"
#include "qkvp_internal.h"

using namespace qkvp;

namespace {

constexpr uint64_t kAlign = kTableAlign;
constexpr int kTcSegmentCost = 14;  // pages of work one request start costs the tcgen05 kernel
// ... and the token-major tcgen05 kernel (its pipeline drains at a request's Q load and segment end;
// measured on the 64-request mixed batch at 16 / 32 / 64 heads, one box: 8 pages 97 / 131 / 206 us,
// 11 pages 97 / 120 / 185, 14 pages 98 / 121 / 177, 20 pages 102 / 124 / 182, 26 pages 104 / 126 /
// 186; 44 x 32K at 32 heads 292 / 289 / 287 / 291 / 294 us; with no charge, before the batched Q load
// and the one-pass softmax, 119 / 163 / 265 us)
constexpr int kTmSegmentCost = 14;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Pinned host staging for work-table uploads, per device: a small ring of buffers, each with an
// event recorded after its copy. A copy from pageable memory can hold the calling thread until the
// stream's earlier work has drained, which serialises a host loop of plan + decode with the GPU;
// from pinned memory the copy is queued and the call returns. A slot is reused only after its
// previous copy has completed (its event). The buffers live until the process exits.
constexpr int kStageDevices = 64, kStageSlots = 4;
constexpr size_t kStageMinBytes = 64 << 10;
struct StageSlot {
  void* host = nullptr;
  size_t cap = 0;
  cudaEvent_t done = nullptr;
};
std::mutex g_stage_mutex;
StageSlot g_stage[kStageDevices][kStageSlots];
int g_stage_next[kStageDevices] = {};

// Copies n bytes to the device buffer dst in stream order (never called during stream capture).
// Pinned staging where it can; a pageable copy if pinned memory is refused (the runtime stages a
// pageable source before the call returns, so `src` may be freed afterwards).
cudaError_t upload_table(void* dst, const void* src, size_t n, cudaStream_t st) {
  int dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kStageDevices) {
    std::lock_guard<std::mutex> lock(g_stage_mutex);
    StageSlot& slot = g_stage[dev][g_stage_next[dev]];
    bool ok = true;
    if (slot.done && cudaEventSynchronize(slot.done) != cudaSuccess) ok = false;
    if (ok && slot.cap < n) {
      if (slot.host) cudaFreeHost(slot.host);
      slot.host = nullptr;
      slot.cap = 0;
      const size_t want = n > kStageMinBytes ? n : kStageMinBytes;
      if (cudaHostAlloc(&slot.host, want, cudaHostAllocPortable) == cudaSuccess) slot.cap = want;
      else { slot.host = nullptr; ok = false; }
    }
    if (ok && !slot.done && cudaEventCreateWithFlags(&slot.done, cudaEventDisableTiming) != cudaSuccess) {
      slot.done = nullptr;
      ok = false;
    }
    if (ok) {
      std::memcpy(slot.host, src, n);
      cudaError_t e = cudaMemcpyAsync(dst, slot.host, n, cudaMemcpyHostToDevice, st);
      if (e == cudaSuccess) e = cudaEventRecord(slot.done, st);
      g_stage_next[dev] = (g_stage_next[dev] + 1) % kStageSlots;
      return e;
    }
    cudaGetLastError();   // a refused pinned allocation is not an error of this call
  }
  return cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, st);
}

int query_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return sms;
}

bool finite_float(float x) { return std::isfinite(x); }

// The kernel family AUTO picks, from decode-kernel times measured on one GB300 (44 x 32K FP8 and
// per-token FP8, 10 x 160K and 1 x 1M NVFP4, the 64-request mixed batch; decode kernel only):
// - 32 to 64 heads on quantized pools: the token-major tcgen05 kernel. FP8 at 32 / 48 / 64 heads
//   287 / 390 / 405 us against 311 (mma.sync) / 494 / 495 us (CTA pair); per-token FP8 296 / 459 /
//   474 against 322 / 539 / 542 us (mma.sync); NVFP4 10 x 160K at 32 / 64 heads 350 / 484 against 542
//   (mma.sync) / 544 us, 1M 236 / 333 against 347 / 361 us; mixed batch at 32 / 48 / 64 heads
//   121 / 173 / 177 against 123 / 183 / 185 us.
// - 16 heads: the mma.sync kernel (FP8 200 against 255 us, NVFP4 279 against 313 us, mixed batch 91
//   against 98 us).
// - More heads (and BF16 pools from 64): the tcgen05 CTA-pair kernel, whose 128 head rows cost the
//   same at any head count; BF16 pools below 64 heads take mma.sync.
int auto_algo(int num_heads, int kv_dtype) {
  if (kv_dtype != QKVP_KV_BF16 && num_heads >= 32 && num_heads <= 64) return QKVP_ALGO_TCGEN05_TOKENS;
  if (num_heads >= 64) return QKVP_ALGO_TCGEN05;
  return QKVP_ALGO_MMA_SYNC;
}

}  // namespace

extern "C" {

int qkvp_version(void) { return 100; }

const char* qkvp_status_string(int status) {
  switch (status) {
    case QKVP_OK: return "ok";
    case QKVP_E_INVALID: return "invalid argument";
    case QKVP_E_UNSUPPORTED: return "unsupported configuration";
    case QKVP_E_WORKSPACE: return "workspace missing or too small";
    case QKVP_E_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int kv_append_quant(const void* src, int32_t src_dtype, int64_t n_tokens, const int64_t* slot_mapping,
                    void* kv_data, uint8_t* kv_scale, int32_t kv_dtype, float global_scale,
                    int32_t page_size, int64_t num_pages, qkvp_stream_t stream) {
  if (n_tokens < 0 || num_pages < 0) return QKVP_E_INVALID;
  if (src_dtype != QKVP_SRC_FP8_E4M3 && src_dtype != QKVP_SRC_BF16) return QKVP_E_UNSUPPORTED;
  if (kv_dtype != QKVP_KV_FP8_E4M3 && kv_dtype != QKVP_KV_NVFP4 && kv_dtype != QKVP_KV_FP8_PER_TOKEN)
    return QKVP_E_UNSUPPORTED;
  if (page_size != QKVP_PAGE_SIZE) return QKVP_E_UNSUPPORTED;
  if (kv_dtype != QKVP_KV_NVFP4) {
    if (kv_scale != nullptr || global_scale != 1.0f) return QKVP_E_INVALID;
  } else {
    if (kv_scale == nullptr || !finite_float(global_scale) || !(global_scale > 0.0f)) return QKVP_E_INVALID;
    if (!aligned(kv_scale, 16)) return QKVP_E_INVALID;
  }
  if (n_tokens == 0) return QKVP_OK;
  if (!src || !slot_mapping || !kv_data) return QKVP_E_INVALID;
  if (!aligned(src, 16) || !aligned(kv_data, 16) || !aligned(slot_mapping, 8)) return QKVP_E_INVALID;
  if (num_pages > (INT64_MAX / page_size)) return QKVP_E_INVALID;
  cudaError_t e = launch_append(src, src_dtype, n_tokens, slot_mapping, kv_data, kv_scale, kv_dtype,
                                global_scale, num_pages * page_size, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QKVP_OK : QKVP_E_CUDA;
}

int mla_decode_plan(const int32_t* kv_indptr_host, const int32_t* kv_len_host, int32_t batch,
                    int32_t num_heads, int32_t page_size, int32_t kv_dtype, int32_t num_sms,
                    int32_t min_splits, int32_t algo, void* workspace, uint64_t workspace_bytes,
                    qkvp_stream_t stream, qkvp_plan* plan) {
  if (!plan) return QKVP_E_INVALID;
  std::memset(plan, 0, sizeof(*plan));
  int st = check_plan_args(kv_indptr_host, kv_len_host, batch, num_heads, page_size, kv_dtype, min_splits);
  if (st != QKVP_OK) return st;
  if (algo == QKVP_ALGO_AUTO) algo = auto_algo(num_heads, kv_dtype);
  if (algo != QKVP_ALGO_MMA_SYNC && algo != QKVP_ALGO_TCGEN05 && algo != QKVP_ALGO_MMA_FP8 &&
      algo != QKVP_ALGO_TCGEN05_TOKENS)
    return QKVP_E_UNSUPPORTED;
  if (algo == QKVP_ALGO_MMA_FP8 && kv_dtype != QKVP_KV_FP8_E4M3 && kv_dtype != QKVP_KV_FP8_PER_TOKEN)
    return QKVP_E_UNSUPPORTED;
  if (algo == QKVP_ALGO_TCGEN05_TOKENS && (kv_dtype == QKVP_KV_BF16 || tm_heads_padded(num_heads) == 0))
    return QKVP_E_UNSUPPORTED;
  int cpw, workers;
  if (algo == QKVP_ALGO_TCGEN05_TOKENS) {
    // one worker = one CTA, one CTA per SM
    cpw = 1;
    if (num_sms <= 0) {
      num_sms = query_sms();
      if (num_sms <= 0) return QKVP_E_CUDA;
    }
    workers = num_sms;
  } else if (algo == QKVP_ALGO_TCGEN05) {
    // one worker = one CTA pair; by default as many pairs as the device runs at once
    cpw = 2;
    if (num_sms <= 0) {
      workers = tc_max_active_clusters();
      if (workers <= 0) return QKVP_E_CUDA;
    } else {
      workers = std::max(1, num_sms / 2);
    }
  } else {
    if (num_sms <= 0) {
      num_sms = query_sms();
      if (num_sms <= 0) return QKVP_E_CUDA;
    }
    const int hc = algo == QKVP_ALGO_MMA_FP8 ? mma_fp8_heads_per_cta(num_heads) : mma_heads_per_cta(num_heads);
    if (hc == 0) return QKVP_E_UNSUPPORTED;
    cpw = num_heads / hc;
    workers = std::max(1, num_sms / cpw);
  }

  // The tcgen05 kernel pays for every request a CTA pair starts: the request's Q is loaded (about
  // 11 us) and the pipeline drains and refills around it (measured with a segment timeline of the
  // kernel on one GB300, at ~1.6 us per page in steady state). Its split balances pages plus this
  // many pages per request started (14 measured best among 0, 8, 14, 20, 28: mixed batch 234 ->
  // 192 us, 44 x 32K 515 -> 509 us, NVFP4 10 x 160K 568 -> 550 us). BF16 pools (the cast-then-attend
  // baseline) take about three times longer per page, so a request start costs them little and equal
  // quotas balance better (mixed batch 500 us against 522 us with the charge); the mma.sync kernel's
  // split gives equal page quotas too.
  const int seg_cost = algo == QKVP_ALGO_TCGEN05 && kv_dtype != QKVP_KV_BF16 ? kTcSegmentCost
                       : algo == QKVP_ALGO_TCGEN05_TOKENS                     ? kTmSegmentCost
                                                                              : 0;
  // count the segments, then fill the table arrays
  SplitInfo info;
  split_pages(kv_indptr_host, kv_len_host, batch, workers, min_splits, SplitOut{}, info, seg_cost);
  // at least one element, so that the fill pass gets a non-null array even without segments
  std::vector<Segment> segs(static_cast<size_t>(std::max<int64_t>(1, info.num_segments)));
  std::vector<int32_t> wptr(workers + 1), rptr(batch + 1), wide(batch > 0 ? batch : 1);
  const SplitOut out{segs.data(), info.num_segments, wptr.data(), rptr.data(), wide.data()};
  if (!split_pages(kv_indptr_host, kv_len_host, batch, workers, min_splits, out, info, seg_cost)) return QKVP_E_INVALID;
  fill_plan(plan, info, batch, num_heads, kv_dtype, algo, workers, cpw);
  if (workspace == nullptr) return QKVP_OK;  // size query: no device work
  if (workspace_bytes < plan->workspace_bytes || !aligned(workspace, kAlign)) {
    const uint64_t need = plan->workspace_bytes;
    std::memset(plan, 0, sizeof(*plan));
    plan->workspace_bytes = need;
    return QKVP_E_WORKSPACE;
  }
  // The table upload is a copy from host memory that this call owns only until it returns; a graph
  // captured around it would read that memory again at every replay. Plans are made outside capture.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cap) != cudaSuccess) return QKVP_E_CUDA;
  if (cap != cudaStreamCaptureStatusNone) {
    std::memset(plan, 0, sizeof(*plan));
    return QKVP_E_UNSUPPORTED;
  }
  std::vector<uint8_t> blob(plan->table_bytes);
  write_table(blob.data(), out, info, workers, batch);
  cudaError_t e = upload_table(workspace, blob.data(), blob.size(), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return QKVP_E_CUDA;
  plan->magic = kPlanMagic;
  return QKVP_OK;
}

namespace {

int check_run_args(const qkvp_plan* plan, int64_t num_pages, float sm_scale, float global_scale,
                   void* workspace, uint64_t workspace_bytes) {
  if (!plan || plan->magic != kPlanMagic) return QKVP_E_INVALID;
  if (!workspace || workspace_bytes < plan->workspace_bytes || !aligned(workspace, kAlign)) return QKVP_E_WORKSPACE;
  if (num_pages < 0 || !finite_float(sm_scale)) return QKVP_E_INVALID;
  if (plan->kv_dtype == QKVP_KV_NVFP4) {
    if (!finite_float(global_scale) || !(global_scale > 0.0f)) return QKVP_E_INVALID;
  } else if (global_scale != 1.0f) {
    return QKVP_E_INVALID;
  }
  return QKVP_OK;
}

DecodeArgs make_args(const qkvp_plan* plan, const void* q, const void* kv_data, const uint8_t* kv_scale,
                     int64_t num_pages, const int32_t* kv_indices, float sm_scale, float global_scale,
                     void* out, float* lse, void* workspace) {
  const TableLayout t = table_layout(plan->num_segments, plan->num_workers, plan->batch);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.kv = static_cast<const uint8_t*>(kv_data);
  a.kv_scale = kv_scale;
  a.num_pages = num_pages;
  a.kv_indices = kv_indices;
  a.segs = reinterpret_cast<const Segment*>(ws + t.segs);
  a.worker_ptr = reinterpret_cast<const int32_t*>(ws + t.wptr);
  a.req_seg_ptr = reinterpret_cast<const int32_t*>(ws + t.rptr);
  a.wide_req = reinterpret_cast<const int32_t*>(ws + t.wide);
  a.part_o = reinterpret_cast<float*>(ws + plan->partial_o_offset);
  a.part_lse = reinterpret_cast<float*>(ws + plan->partial_lse_offset);
  a.status = reinterpret_cast<int*>(ws + t.status);
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.batch = plan->batch;
  a.heads = plan->num_heads;
  a.num_workers = plan->num_workers;
  a.ctas_per_worker = plan->ctas_per_worker;
  a.num_segments = plan->num_segments;
  a.kv_dtype = plan->kv_dtype;
  a.fp8_qk = plan->algo == QKVP_ALGO_MMA_FP8 ? 1 : 0;
  a.scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * global_scale * 1.4426950408889634);
  a.out_scale = global_scale;
  return a;
}

}  // namespace

int mla_decode_attend(const qkvp_plan* plan, const void* q, const void* kv_data, const uint8_t* kv_scale,
                      int64_t num_pages, const int32_t* kv_indices, float sm_scale, float global_scale,
                      void* out, float* lse, void* workspace, uint64_t workspace_bytes,
                      qkvp_stream_t stream) {
  int st = check_run_args(plan, num_pages, sm_scale, global_scale, workspace, workspace_bytes);
  if (st != QKVP_OK) return st;
  if (plan->batch == 0 || plan->num_segments == 0) return QKVP_OK;
  if (!q || !out || !aligned(q, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4))) return QKVP_E_INVALID;
  if (!kv_data || !kv_indices || !aligned(kv_data, 32) || !aligned(kv_indices, 4)) return QKVP_E_INVALID;
  if (plan->kv_dtype == QKVP_KV_NVFP4 && (!kv_scale || !aligned(kv_scale, 16))) return QKVP_E_INVALID;
  const DecodeArgs a = make_args(plan, q, kv_data, kv_scale, num_pages, kv_indices, sm_scale,
                                 global_scale, out, lse, workspace);
  cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = plan->algo == QKVP_ALGO_TCGEN05          ? launch_decode_tc(a, st_)
                  : plan->algo == QKVP_ALGO_TCGEN05_TOKENS ? launch_decode_tm(a, st_)
                                                           : launch_decode_mma(a, st_);
  return e == cudaSuccess ? QKVP_OK : QKVP_E_CUDA;
}

int mla_decode_combine(const qkvp_plan* plan, float global_scale, void* out, float* lse,
                       void* workspace, uint64_t workspace_bytes, qkvp_stream_t stream) {
  int st = check_run_args(plan, 0, 0.0f, global_scale, workspace, workspace_bytes);
  if (st != QKVP_OK) return st;
  if (plan->batch == 0 || (plan->num_split_requests == 0 && plan->num_empty_requests == 0)) return QKVP_OK;
  if (!out || !aligned(out, 16) || (lse && !aligned(lse, 4))) return QKVP_E_INVALID;
  if (plan->num_wide_requests < 0 || plan->num_wide_requests > plan->batch) return QKVP_E_INVALID;
  const DecodeArgs a = make_args(plan, nullptr, nullptr, nullptr, 0, nullptr, 0.0f, global_scale,
                                 out, lse, workspace);
  cudaError_t e = launch_combine(a, plan->num_wide_requests, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QKVP_OK : QKVP_E_CUDA;
}

int mla_decode_run(const qkvp_plan* plan, const void* q, const void* kv_data, const uint8_t* kv_scale,
                   int64_t num_pages, const int32_t* kv_indices, float sm_scale, float global_scale,
                   void* out, float* lse, void* workspace, uint64_t workspace_bytes,
                   qkvp_stream_t stream) {
  int st = mla_decode_attend(plan, q, kv_data, kv_scale, num_pages, kv_indices, sm_scale, global_scale,
                             out, lse, workspace, workspace_bytes, stream);
  if (st != QKVP_OK) return st;
  return mla_decode_combine(plan, global_scale, out, lse, workspace, workspace_bytes, stream);
}

int kv_gather_fp8(const void* kv_data, const uint8_t* kv_scale, int32_t kv_dtype, float global_scale,
                  int32_t page_size, int64_t num_pages, const int32_t* kv_indptr, const int32_t* kv_indices,
                  int64_t nnz, const int64_t* tok_indptr, int32_t batch, int64_t total_tokens, uint8_t* out,
                  qkvp_stream_t stream) {
  if (page_size != kPage) return QKVP_E_UNSUPPORTED;
  if (kv_dtype == QKVP_KV_BF16 || kv_dtype == QKVP_KV_FP8_PER_TOKEN) return QKVP_E_UNSUPPORTED;
  if (kv_dtype != QKVP_KV_FP8_E4M3 && kv_dtype != QKVP_KV_NVFP4) return QKVP_E_INVALID;
  if (batch < 0 || total_tokens < 0 || nnz < 0 || num_pages < 0) return QKVP_E_INVALID;
  if (kv_dtype == QKVP_KV_NVFP4) {
    if (!finite_float(global_scale) || !(global_scale > 0.0f)) return QKVP_E_INVALID;
  } else if (global_scale != 1.0f || kv_scale) {
    return QKVP_E_INVALID;
  }
  if (batch == 0 || total_tokens == 0) return QKVP_OK;
  if (!kv_data || !kv_indptr || !kv_indices || !tok_indptr || !out) return QKVP_E_INVALID;
  if (!aligned(kv_data, 16) || !aligned(out, 16) || !aligned(tok_indptr, 8) || !aligned(kv_indptr, 4) ||
      !aligned(kv_indices, 4))
    return QKVP_E_INVALID;
  if (kv_dtype == QKVP_KV_NVFP4 && !kv_scale) return QKVP_E_INVALID;
  GatherArgs a{};
  a.kv = static_cast<const uint8_t*>(kv_data);
  a.kv_scale = kv_scale;
  a.num_pages = num_pages;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.nnz = nnz;
  a.tok_indptr = tok_indptr;
  a.out = out;
  a.total_tokens = total_tokens;
  a.batch = batch;
  a.kv_dtype = kv_dtype == QKVP_KV_NVFP4 ? KV_NVFP4 : KV_FP8;
  a.g = global_scale;
  cudaError_t e = launch_gather_fp8(a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QKVP_OK : QKVP_E_CUDA;
}

int kv_gather_pages_bf16(const uint8_t* kv_data, int32_t page_size, int64_t num_pages, const int32_t* page_ids,
                         int64_t n_pages, void* out, qkvp_stream_t stream) {
  if (page_size != kPage) return QKVP_E_UNSUPPORTED;
  if (n_pages < 0 || num_pages < 0) return QKVP_E_INVALID;
  if (n_pages == 0) return QKVP_OK;
  if (!kv_data || !page_ids || !out || !aligned(kv_data, 16) || !aligned(out, 16) || !aligned(page_ids, 4))
    return QKVP_E_INVALID;
  cudaError_t e = launch_gather_pages_bf16(kv_data, num_pages, page_ids, n_pages, out,
                                           reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QKVP_OK : QKVP_E_CUDA;
}

int kv_pool_cast_bf16(const uint8_t* in, int64_t n_elems, void* out, qkvp_stream_t stream) {
  if (n_elems < 0 || n_elems % 16) return QKVP_E_INVALID;
  if (n_elems == 0) return QKVP_OK;
  if (!in || !out || !aligned(in, 16) || !aligned(out, 16)) return QKVP_E_INVALID;
  cudaError_t e = launch_cast(in, n_elems, static_cast<uint16_t*>(out), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QKVP_OK : QKVP_E_CUDA;
}

int qkvp_encode_f32(const float* x, int64_t n, int32_t fmt, uint8_t* codes, qkvp_stream_t stream) {
  if (n < 0 || (fmt != 1 && fmt != 2)) return QKVP_E_INVALID;
  if (n == 0) return QKVP_OK;
  if (!x || !codes || !aligned(x, 4)) return QKVP_E_INVALID;
  cudaError_t e = launch_encode(x, n, fmt, codes, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QKVP_OK : QKVP_E_CUDA;
}

}  // extern "C"
