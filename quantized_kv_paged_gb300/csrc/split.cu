// The split-KV planner shared by mla_decode_plan and mla_decode_noalloc (host code).
//
// Requests are laid end to end in request order, one unit per page (ceil(len / 64) pages each),
// and worker w takes the contiguous run of pages [w * quota, (w + 1) * quota), quota =
// ceil(total / workers), so no worker holds more than one page above the mean. Each worker's run is
// cut at request boundaries and into pieces of at most `cap` pages, cap = total / min_splits when a
// minimum number of splits is asked for; each piece is one segment. Segments therefore come in
// request order, and the segments of one request are contiguous. The routine uses no heap: it
// writes into the caller's arrays, so the no-allocation entry point can hand it static storage.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>

#include "../../include/qkvp.h"
#include "qkvp_internal.h"

namespace qkvp {

int check_plan_args(const int32_t* indptr, const int32_t* len, int batch, int num_heads, int page_size,
                    int kv_dtype, int min_splits) {
  if (batch < 0 || min_splits < 0) return QKVP_E_INVALID;
  if (batch > 0 && (!indptr || !len)) return QKVP_E_INVALID;
  if (page_size != QKVP_PAGE_SIZE) return QKVP_E_UNSUPPORTED;
  if (num_heads < 16 || num_heads > 128 || num_heads % 16) return QKVP_E_UNSUPPORTED;
  if (kv_dtype != QKVP_KV_FP8_E4M3 && kv_dtype != QKVP_KV_NVFP4 && kv_dtype != QKVP_KV_BF16 &&
      kv_dtype != QKVP_KV_FP8_PER_TOKEN)
    return QKVP_E_UNSUPPORTED;
  if (batch > 0 && indptr[0] != 0) return QKVP_E_INVALID;
  for (int r = 0; r < batch; ++r) {
    const int64_t np = static_cast<int64_t>(indptr[r + 1]) - indptr[r];
    if (np < 0 || len[r] < 0) return QKVP_E_INVALID;
    if ((static_cast<int64_t>(len[r]) + page_size - 1) / page_size > np) return QKVP_E_INVALID;
  }
  return QKVP_OK;
}

void fill_plan(qkvp_plan* plan, const SplitInfo& info, int batch, int num_heads, int kv_dtype, int algo,
               int workers, int ctas_per_worker) {
  const TableLayout t = table_layout(info.num_segments, workers, batch);
  plan->batch = batch;
  plan->num_heads = num_heads;
  plan->page_size = kPage;
  plan->kv_dtype = kv_dtype;
  plan->algo = algo;
  plan->num_workers = workers;
  plan->ctas_per_worker = ctas_per_worker;
  plan->num_segments = static_cast<int32_t>(info.num_segments);
  plan->num_split_requests = info.split_reqs;
  plan->num_empty_requests = info.empty_reqs;
  plan->max_worker_pages = info.max_pages;
  plan->min_worker_pages = info.min_pages;
  plan->num_partials = info.partials;
  plan->max_request_segments = info.max_req_segs;
  plan->num_wide_requests = info.num_wide;
  plan->total_pages = info.total_pages;
  plan->total_tokens = info.total_tokens;
  plan->table_bytes = t.bytes;
  plan->status_offset = t.status;
  plan->partial_o_offset = t.bytes;
  plan->partial_lse_offset = t.bytes + align_up(static_cast<uint64_t>(info.partials) * num_heads * kDv * 4);
  plan->workspace_bytes = plan->partial_lse_offset + align_up(static_cast<uint64_t>(info.partials) * num_heads * 4);
}

void write_table(uint8_t* blob, const SplitOut& s, const SplitInfo& info, int workers, int batch) {
  const TableLayout t = table_layout(info.num_segments, workers, batch);
  std::memset(blob, 0, t.bytes);
  if (info.num_segments > 0) std::memcpy(blob + t.segs, s.segs, info.num_segments * sizeof(Segment));
  std::memcpy(blob + t.wptr, s.wptr, (workers + 1) * sizeof(int32_t));
  std::memcpy(blob + t.rptr, s.rptr, (batch + 1) * sizeof(int32_t));
  if (info.num_wide > 0) std::memcpy(blob + t.wide, s.wide, info.num_wide * sizeof(int32_t));
}

bool split_pages(const int32_t* indptr, const int32_t* len, int batch, int workers, int min_splits,
                 const SplitOut& out, SplitInfo& info, int seg_cost) {
  info = SplitInfo{};
  auto pages_of = [len](int r) { return (static_cast<int64_t>(len[r]) + kPage - 1) / kPage; };
  int64_t total = 0;
  for (int r = 0; r < batch; ++r) {
    total += pages_of(r);
    info.total_tokens += len[r];
  }
  info.total_pages = total;
  const int64_t quota = total > 0 ? (total + workers - 1) / workers : 0;
  int64_t cap = quota;
  if (min_splits > 0 && total > 0) cap = std::max<int64_t>(1, std::min<int64_t>(quota, total / min_splits));

  // Worker page ranges. With seg_cost = 0, equal quotas. Otherwise every request a worker starts costs
  // seg_cost pages on top of its pages, and each worker fills up to a budget in request order; the
  // budget is the smallest for which `workers` workers cover every page (bisection). Walks the
  // requests from `x` (in request `r`, whose first page unit is `start_r`) and returns the end of
  // one worker's range.
  auto fill = [&](int64_t budget, int64_t x, int& r, int64_t& start_r) {
    int64_t cost = 0;
    while (x < total) {
      while (r < batch && start_r + pages_of(r) <= x) {
        start_r += pages_of(r);
        ++r;
      }
      const int64_t room = budget - cost - seg_cost;
      if (room <= 0) break;
      const int64_t take = std::min(room, start_r + pages_of(r) - x);
      cost += seg_cost + take;
      x += take;
      if (x < start_r + pages_of(r)) break;   // the budget ended inside this request
    }
    return x;
  };
  int64_t budget = quota;
  if (seg_cost > 0 && total > 0) {
    auto covers = [&](int64_t bgt) {
      int64_t x = 0, start_r = 0;
      int r = 0;
      for (int w = 0; w < workers && x < total; ++w) x = fill(bgt, x, r, start_r);
      return x >= total;
    };
    int64_t lo = quota, hi = quota + static_cast<int64_t>(seg_cost) * (batch + 1) + 1;
    while (!covers(hi)) hi *= 2;
    while (lo < hi) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (covers(mid)) hi = mid; else lo = mid + 1;
    }
    budget = lo;
    // ranges may exceed the equal quota now: cut them only for a requested minimum of splits
    cap = min_splits > 0 ? std::max<int64_t>(1, std::min<int64_t>(budget, total / min_splits)) : total;
  }

  info.max_pages = 0;
  info.min_pages = total > 0 ? INT32_MAX : 0;
  int64_t n = 0, start_r = 0;   // segments so far; first page unit of request r
  int r = 0;
  int64_t fx = 0, fstart_r = 0;
  int fr = 0;
  for (int w = 0; w < workers; ++w) {
    if (out.wptr) out.wptr[w] = static_cast<int32_t>(n);
    int64_t a, b;
    if (seg_cost > 0) {
      a = fx;
      b = fill(budget, fx, fr, fstart_r);
      fx = b;
    } else {
      a = std::min(total, w * quota);
      b = std::min(total, (w + 1) * quota);
    }
    info.max_pages = std::max<int32_t>(info.max_pages, static_cast<int32_t>(b - a));
    if (total > 0) info.min_pages = std::min<int32_t>(info.min_pages, static_cast<int32_t>(b - a));
    int64_t x = a;
    while (x < b) {
      while (r < batch && start_r + pages_of(r) <= x) {
        start_r += pages_of(r);
        ++r;
      }
      const int64_t y = std::min(b, start_r + pages_of(r));
      for (int64_t c = x; c < y; c += cap) {
        const int64_t e = std::min(y, c + cap);
        if (out.segs) {
          if (n >= out.max_segs) return false;
          Segment g{};
          g.req = r;
          g.page_begin = static_cast<int32_t>(indptr[r] + (c - start_r));
          g.num_pages = static_cast<int32_t>(e - c);
          g.num_tokens = static_cast<int32_t>(std::min<int64_t>(len[r], (e - start_r) * kPage) - (c - start_r) * kPage);
          g.partial = 0;
          out.segs[n] = g;
        }
        ++n;
      }
      x = y;
    }
  }
  if (out.wptr) out.wptr[workers] = static_cast<int32_t>(n);
  info.num_segments = n;
  if (!out.segs) return true;
  // per-request segment ranges; a request with one segment writes its output directly
  int64_t k = 0;
  for (int q = 0; q < batch; ++q) {
    if (out.rptr) out.rptr[q] = static_cast<int32_t>(k);
    const int64_t k0 = k;
    while (k < n && out.segs[k].req == q) ++k;
    const int64_t m = k - k0;
    if (m == 0) ++info.empty_reqs;
    if (m >= 2) ++info.split_reqs;
    info.max_req_segs = std::max<int32_t>(info.max_req_segs, static_cast<int32_t>(m));
    if (m > kCombineWideSegs) {
      if (out.wide) out.wide[info.num_wide] = q;
      ++info.num_wide;
    }
    for (int64_t i = k0; i < k; ++i) out.segs[i].partial = m == 1 ? -1 : info.partials++;
  }
  if (out.rptr) out.rptr[batch] = static_cast<int32_t>(k);
  return true;
}

}  // namespace qkvp
