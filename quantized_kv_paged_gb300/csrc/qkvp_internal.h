// Internal declarations shared by the translation units of libqkvp (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/qkvp.h"

namespace qkvp {

constexpr int kLatent = 576;            // 512 nope + 64 rope
constexpr int kDv = 512;                // V = the first 512 latent dims
constexpr int kPage = 64;               // tokens per page
constexpr int kPacked = kLatent / 2;    // NVFP4 data bytes per token (two E2M1 codes per byte)
constexpr int kScales = kLatent / 16;   // NVFP4 E4M3 block scales per token
constexpr uint64_t kPlanMagic = 0x716b76702d706c31ull;

enum : int { KV_FP8 = 1, KV_NVFP4 = 2, KV_BF16 = 3, KV_FP8PT = 4 };
// Per-token-scaled FP8 page: 64 rows of 576 E4M3 codes, then 64 FP32 token scales.
constexpr int kPtScaleOff = kPage * kLatent;              // 36,864
constexpr int kPtPageBytes = kPage * (kLatent + 4);       // 37,120
enum : int { SRC_FP8 = 1, SRC_BF16 = 2 };
enum : int { ALGO_AUTO = 0, ALGO_MMA = 1, ALGO_TC = 2 };

// One piece of one request's page list, processed by one worker from start to end. Segments are
// stored in request order; a request whose pages form a single segment is written straight to the
// output (partial < 0), otherwise each segment writes a normalised FP32 partial and its
// log2-sum-exp, merged by the combine kernel.
struct Segment {
  int32_t req;
  int32_t page_begin;   // index into kv_indices of the first page
  int32_t num_pages;
  int32_t num_tokens;   // tokens covered (the last page may be partial)
  int32_t partial;      // partial slot, or -1 for a direct write
  int32_t pad[3];
};
static_assert(sizeof(Segment) == 32, "segment layout");

struct DecodeArgs {
  const uint16_t* q;          // bf16 [B][H][576]
  const uint8_t* kv;          // pool (fp8 / nvfp4 data / bf16)
  const uint8_t* kv_scale;    // nvfp4 block scales
  int64_t num_pages;
  const int32_t* kv_indices;
  const Segment* segs;
  const int32_t* worker_ptr;  // [num_workers + 1]
  const int32_t* req_seg_ptr; // [batch + 1]
  const int32_t* wide_req;    // [num_wide] requests with more than kCombineWideSegs segments
  float* part_o;              // [num_segments][H][512]
  float* part_lse;            // [num_segments][H], log2 domain
  uint16_t* out;              // bf16 [B][H][512]
  float* lse;                 // [B][H] natural log, may be null
  int* status;                // device status word (timeouts), inside the workspace
  int batch, heads, num_workers, ctas_per_worker, num_segments, kv_dtype;
  int fp8_qk;                 // mma.sync kernel: FP8 Q.K^T (two-term E4M3 Q) instead of FP16
  float scale_log2;           // sm_scale * g * log2(e)
  float out_scale;            // g
};

// Workspace layout of a plan: the segment table, the per-worker segment ranges, the per-request
// segment ranges and the list of wide requests, each 256-byte aligned, followed by the FP32 partials.
constexpr uint64_t kTableAlign = 256;
inline uint64_t align_up(uint64_t x) { return (x + kTableAlign - 1) / kTableAlign * kTableAlign; }

// The status word is zero after planning; a kernel that gives up waiting sets bits in it.
struct TableLayout {
  uint64_t segs, wptr, rptr, wide, status, bytes;
};

// A request cut into more segments than this is merged by the combine's wide CTAs (eight segment
// groups per quarter head) instead of one thread per 8 output dims walking every segment; the
// planner lists such requests in the table.
constexpr int kCombineWideSegs = 8;

inline TableLayout table_layout(int64_t segments, int64_t workers, int64_t batch) {
  TableLayout t;
  t.segs = 0;
  t.wptr = align_up(static_cast<uint64_t>(segments) * sizeof(Segment));
  t.rptr = t.wptr + align_up(static_cast<uint64_t>(workers + 1) * 4);
  t.wide = t.rptr + align_up(static_cast<uint64_t>(batch + 1) * 4);
  t.status = t.wide + align_up(static_cast<uint64_t>(batch) * 4);
  t.bytes = t.status + kTableAlign;
  return t;
}

// The split-KV planner (split.cu), shared by mla_decode_plan and mla_decode_noalloc. It writes into
// the caller's arrays: segs [max_segs], wptr [workers + 1], rptr [batch + 1], wide [batch]. With
// segs == nullptr it only counts (num_segments, page totals and per-worker page counts); the
// per-request fields of SplitInfo need the segments. Returns false when more than max_segs
// segments would be written.
struct SplitOut {
  Segment* segs = nullptr;
  int64_t max_segs = 0;
  int32_t* wptr = nullptr;
  int32_t* rptr = nullptr;
  int32_t* wide = nullptr;
};
struct SplitInfo {
  int64_t num_segments = 0;
  int32_t split_reqs = 0, empty_reqs = 0, max_pages = 0, min_pages = 0, partials = 0, max_req_segs = 0,
          num_wide = 0;
  int64_t total_pages = 0, total_tokens = 0;
};
// seg_cost > 0 balances pages + seg_cost per request each worker starts (the tcgen05 kernel loads a
// new request's Q and refills its pipeline at each); 0 gives every worker an equal page quota.
bool split_pages(const int32_t* indptr, const int32_t* len, int batch, int workers, int min_splits,
                 const SplitOut& out, SplitInfo& info, int seg_cost = 0);
// The argument checks of mla_decode_plan that need no device (status code, QKVP_OK if they pass).
int check_plan_args(const int32_t* indptr, const int32_t* len, int batch, int num_heads, int page_size,
                    int kv_dtype, int min_splits);
// Sets every field of *plan except magic from a split (table layout, offsets and workspace size).
void fill_plan(qkvp_plan* plan, const SplitInfo& info, int batch, int num_heads, int kv_dtype, int algo,
               int workers, int ctas_per_worker);
// Writes the work table of a filled split into blob [table_layout(...).bytes], zeros elsewhere.
void write_table(uint8_t* blob, const SplitOut& s, const SplitInfo& info, int workers, int batch);

// Arguments of the extend-path gather (kv_gather_fp8).
struct GatherArgs {
  const uint8_t* kv;
  const uint8_t* kv_scale;
  int64_t num_pages;
  const int32_t* kv_indptr;   // [batch + 1], pages
  const int32_t* kv_indices;  // [nnz] page ids
  int64_t nnz;
  const int64_t* tok_indptr;  // [batch + 1], workspace rows
  uint8_t* out;               // [total_tokens][576] E4M3
  int64_t total_tokens;
  int batch, kv_dtype;
  float g;
};

cudaError_t launch_gather_fp8(const GatherArgs& a, cudaStream_t s);
cudaError_t launch_gather_pages_bf16(const uint8_t* pool, int64_t num_pages, const int32_t* ids, int64_t n,
                                     void* out, cudaStream_t s);
cudaError_t launch_append(const void* src, int src_dtype, int64_t n, const int64_t* slots,
                          void* kv_data, uint8_t* kv_scale, int kv_dtype, float g,
                          int64_t num_slots, cudaStream_t s);
cudaError_t launch_encode(const float* x, int64_t n, int fmt, uint8_t* codes, cudaStream_t s);
cudaError_t launch_cast(const uint8_t* in, int64_t n, uint16_t* out, cudaStream_t s);
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_tm(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_combine(const DecodeArgs& a, int num_wide, cudaStream_t s);

// Heads per CTA of the mma.sync kernel for a head count (0 if unsupported), and of its FP8 Q.K^T
// variant (16 or 32).
int mma_heads_per_cta(int heads);
int mma_fp8_heads_per_cta(int heads);
// Head columns of the token-major tcgen05 kernel for a head count (16, 32 or 64; 0 if unsupported).
int tm_heads_padded(int heads);
// CTA pairs of the tcgen05 kernel that the current device runs at once (-1 on error).
int tc_max_active_clusters();

}  // namespace qkvp
