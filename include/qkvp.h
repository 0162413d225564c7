/*
 * qkvp.h - C ABI of libqkvp: paged MLA decode attention that reads a quantized latent KV cache
 * (FP8 E4M3 or NVFP4) directly, for NVIDIA GB300 (sm_103a).
 *
 * The problem, as the source pages state it:
 *  - Each token stores one 576-wide latent: kv_lora_rank 512 ("nope") + qk_rope_head_dim 64. All
 *    query heads share it. Attention uses K = the whole latent and V = its first 512 dims ("The
 *    Smoking Gun: Tracing the FP8-to-BF16 KV Cache Cast", section "The Investigation Leading to This
 *    Message": pool shape [495552, 1, 576]).
 *  - The pool is paged and addressed through a CSR page table (qo_indptr, kv_indptr, kv_indices,
 *    kv_len_arr), with num_heads, kv_lora_rank, qk_rope_head_dim, page_size, sm_scale and the KV
 *    dtype given to a host-side plan() before a device-side run() ("The Smoking Gun", section
 *    "What Message 1408 Actually Reveals").
 *  - The KV cache is FP8 E4M3 (float8_e4m3fn; "The FP8 KV Cache Wall", section "Context and
 *    Motivation") or NVFP4: E2M1 values, one E4M3 scale per 16 values, one FP32 global scale per
 *    tensor ("SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "NVFP4 format").
 *  - Decode reads the quantized pages directly and dequantizes inside the kernel; nothing casts the
 *    pool to BF16 first (same page, section "SGLang implementation", item 3).
 *
 * Memory layout (all device buffers are caller-owned; the library allocates no device memory. Its
 * only global state: per device, four pinned host staging buffers and events for the work table
 * upload of mla_decode_plan, and the fixed device scratch array of mla_decode_noalloc with its
 * static host table):
 *  - slot s = page * page_size + offset; page_size must be 64.
 *  - FP8 pool  : kv_data uint8 [num_pages][64][576], one E4M3 byte per latent element. The decode
 *                entry points read kv_data (any pool type) with 32-byte loads: it must be 32-byte aligned.
 *  - NVFP4 pool: kv_data uint8 [num_pages][64][288] packed E2M1 pairs (element 2k in the low nibble
 *                of byte k, 2k+1 in the high nibble) and kv_scale uint8 [num_pages][64][36] E4M3
 *                block scales (block j covers elements 16j..16j+15). 324 bytes per token = 9/16 of
 *                FP8. An element decodes to global_scale * scale(block) * e2m1(code).
 *  - FP8 pool with per-token scales (QKVP_KV_FP8_PER_TOKEN): kv_data uint8 [num_pages][37120]:
 *                page p holds the 64 token rows of 576 E4M3 codes (bytes 0..36863), then the 64
 *                FP32 token scales (bytes 36864..37119, little-endian). 580 bytes per token. An
 *                element decodes to scale(token) * e4m3(code). The layout is the pages' indexer key
 *                cache (FP8 elements + 4 scale bytes per token in a paged [npages, page_bytes] uint8
 *                buffer, 64 tokens per page: "The Precision Frontier: Implementing bf16 Index Keys",
 *                section "The Message: Planning the bf16-K Implementation") carrying the latent.
 *  - BF16 pool : kv_data uint16 [num_pages][64][576] (the cast-then-attend baseline only).
 *  - q         : bf16 [batch][num_heads][576], row-major, contiguous.
 *  - out       : bf16 [batch][num_heads][512], 16-byte aligned (the attend kernels store 16-byte
 *                vectors); lse: float [batch][num_heads] (natural log), or NULL.
 *
 * Errors: every call returns an int status (qkvp_status). Arguments are checked before anything is
 * launched; a failed check launches nothing. QKVP_E_CUDA reports a CUDA error from a launch or copy
 * issued by the call. Faults that occur asynchronously inside a kernel surface at the caller's next
 * synchronisation. Indices read from device memory (slot ids, page ids) are bounds-checked in the
 * kernels: out-of-range entries are skipped (append) or read as masked tokens (decode); they never
 * cause an out-of-bounds access.
 *
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are asynchronous
 * with respect to the host unless stated. The library is re-entrant across distinct streams and
 * workspaces.
 */
#ifndef QKVP_H_
#define QKVP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* qkvp_stream_t; /* identical to cudaStream_t */

typedef enum {
  QKVP_OK = 0,
  QKVP_E_INVALID = -1,     /* bad argument: null pointer, negative size, inconsistent page table */
  QKVP_E_UNSUPPORTED = -2, /* valid but not supported: page size, head count, dtype combination */
  QKVP_E_WORKSPACE = -3,   /* workspace missing or smaller than plan->workspace_bytes */
  QKVP_E_CUDA = -4         /* a CUDA runtime call or launch failed */
} qkvp_status;

typedef enum {
  QKVP_KV_FP8_E4M3 = 1,
  QKVP_KV_NVFP4 = 2,
  QKVP_KV_BF16 = 3,
  QKVP_KV_FP8_PER_TOKEN = 4
} qkvp_kv_dtype;
typedef enum { QKVP_SRC_FP8_E4M3 = 1, QKVP_SRC_BF16 = 2 } qkvp_src_dtype;

/* Decode kernel families. AUTO lets the planner choose. */
typedef enum {
  QKVP_ALGO_AUTO = 0,
  QKVP_ALGO_MMA_SYNC = 1,  /* warp-level mma.sync split-KV kernel, any supported head count */
  QKVP_ALGO_TCGEN05 = 2,   /* tcgen05/TMEM CTA-pair split-KV kernel: always 128 head rows (fewer heads
                              ride as zero rows), so its cost does not shrink with the heads; AUTO picks
                              it above 64 heads (from 64 for BF16 pools) */
  QKVP_ALGO_MMA_FP8 = 3,   /* the mma.sync kernel with Q.K^T on the FP8 tensor-core path, for FP8 and
                              per-token-scaled FP8 pools (others: QKVP_E_UNSUPPORTED): K is the page's
                              E4M3 bytes as stored, Q is split per head row into two E4M3 terms,
                              q ~ (hi + lo / 16) / sc with sc = 2^floor(log2(448 / max|q|)),
                              hi = E4M3(q sc), lo = E4M3(16 (q sc - hi)), and the two products are
                              summed in FP32; P.V stays FP16. The pages' decode dequantizes "to FP8 or
                              BF16" ("SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "SGLang
                              implementation", item 3); a single E4M3 term for Q (or for P) misses
                              the output tolerance on the outlier-channel workloads, two terms for Q
                              meet it. 16 or 32 heads per CTA. On GB300 it takes 1.5-1.8x the
                              time of QKVP_ALGO_MMA_SYNC (two MMAs per 32 dims, and the legacy FP8
                              MMA path gains no rate over FP16), so AUTO never picks it. */
  QKVP_ALGO_TCGEN05_TOKENS = 4 /* tcgen05/TMEM kernel with the page's tokens as the rows of both
                              products (M = 64 tokens for Q.K^T, M = 128 output dims for P.V) and the
                              heads as the columns (N = 16, 32 or 64; 48 heads ride in 64): 16 to 64
                              heads, FP8, NVFP4 and per-token-scaled FP8 pools (others:
                              QKVP_E_UNSUPPORTED); one CTA per SM. Same arithmetic and tolerance as
                              the other families. AUTO picks it for quantized pools at 32 to 64 heads,
                              where it measured fastest on GB300 (FP8 44 x 32K at 32 / 64 heads:
                              287 / 405 us against 311 / 495 us for the other families; NVFP4 1M:
                              236 / 333 against 347 / 361 us). At 16 heads the mma.sync kernel is
                              faster. */
} qkvp_algo;

#define QKVP_LATENT_DIM 576
#define QKVP_V_DIM 512
#define QKVP_PAGE_SIZE 64

/* Host-side plan produced by mla_decode_plan and consumed by mla_decode_run. Plain data: it may be
 * copied, and one plan serves any number of runs (e.g. one per layer) with the same page table,
 * lengths, head count and KV dtype, as long as the workspace it was uploaded to is left intact. */
typedef struct {
  int32_t batch, num_heads, page_size, kv_dtype;
  int32_t algo;              /* the kernel family the plan was made for */
  int32_t num_workers;       /* independent split-KV workers (one CTA pair or CTA group each) */
  int32_t ctas_per_worker;   /* CTAs that cooperate on one worker's token ranges */
  int32_t num_segments;      /* (request, page range) pieces; each writes one partial or output */
  int32_t num_split_requests;/* requests whose pages span more than one segment (need a combine) */
  int32_t num_empty_requests;/* requests with no tokens (output 0, lse -inf) */
  int32_t max_worker_pages;  /* most pages given to one worker (load balance) */
  int32_t min_worker_pages;  /* fewest pages given to one worker */
  int32_t num_partials;      /* FP32 split partials held in the workspace */
  int32_t max_request_segments; /* most segments one request is cut into */
  int32_t num_wide_requests; /* requests cut into more than 8 segments: the combine gives each of
                                them several CTAs per head instead of one thread per 8 output dims */
  int64_t total_pages;       /* sum over requests of ceil(len / 64) */
  int64_t total_tokens;      /* sum of lengths */
  uint64_t workspace_bytes;  /* device workspace the run needs (table + split partials) */
  uint64_t table_bytes;      /* bytes of the work table at the start of the workspace */
  uint64_t partial_o_offset; /* byte offset of the FP32 partial outputs in the workspace */
  uint64_t partial_lse_offset;
  uint64_t status_offset;    /* int32 device status word in the workspace: 0 after planning; a
                                decode kernel that gave up waiting on its own pipeline (a bug, never
                                expected) sets bits in it, and its outputs are then undefined */
  uint64_t magic;            /* set by a successful plan; checked by run */
} qkvp_plan;

/*
 * kv_append_quant - quantize-on-append: write n_tokens new latent rows into the paged pool.
 *
 * Source: "SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "SGLang implementation", items 1-2
 * (quantize KV from FP8 into NVFP4 and write it to the persistent cache); section "NVFP4 format"
 * (two-level scaling). For an FP8 pool: E4M3 storage of the latent ("The FP8 KV Cache Wall").
 *
 *  src          device, [n_tokens][576]: E4M3 bytes (src_dtype QKVP_SRC_FP8_E4M3) or BF16
 *               (QKVP_SRC_BF16).
 *  slot_mapping device int64 [n_tokens]: destination slot page * page_size + offset; a negative slot
 *               skips the token; a slot >= num_pages * page_size is skipped too.
 *  kv_data      device pool (layout above) for kv_dtype QKVP_KV_FP8_E4M3, QKVP_KV_NVFP4 or
 *               QKVP_KV_FP8_PER_TOKEN.
 *  kv_scale     device NVFP4 block-scale pool; must be NULL for the FP8 pools.
 *  global_scale NVFP4 decode multiplier g (> 0, finite): an element decodes to g * s * e. Must be
 *               1.0 for the FP8 pools.
 *
 * FP8 pool: FP8 sources are copied; BF16 sources round to nearest even, saturating at +-448; NaN
 * gives 0x7F. NVFP4 pool, per block of 16 consecutive elements x (FP32 arithmetic, one rounding per
 * operation): amax = max|x| (NaN if any x is NaN); s8 = E4M3(amax / (6 g)) rounded to nearest even
 * and saturated; sd = value(s8) * g; codes = 0 where sd == 0, else E2M1(x / sd) rounded to nearest
 * even and saturated at +-6 (NaN gives 0). FP8 pool with per-token scales, per token x (FP32
 * arithmetic, one rounding per operation): amax = max|x|; scale = amax / 448, or the NaN 0x7FC00000
 * if any x is NaN; codes = E4M3(x / scale) rounded to nearest even and saturated (NaN gives 0x7F),
 * or E4M3(x) (a signed zero) when scale == 0. The stored bytes are bit-identical to the CPU oracle.
 * If two tokens of one call name the same slot, which of them is stored is unspecified.
 */
int kv_append_quant(const void* src, int32_t src_dtype, int64_t n_tokens,
                    const int64_t* slot_mapping, void* kv_data, uint8_t* kv_scale,
                    int32_t kv_dtype, float global_scale, int32_t page_size, int64_t num_pages,
                    qkvp_stream_t stream);

/*
 * mla_decode_plan - split the batch's pages into balanced work for the decode kernel.
 *
 * Source: the plan/run split and CSR page table of the pages' plan() call ("The Smoking Gun",
 * section "What Message 1408 Actually Reveals"). The split-KV decomposition itself is not on the
 * pages; its partial results are merged by log-sum-exp in mla_decode_run.
 *
 *  kv_indptr_host host int32 [batch + 1], in pages: request r owns kv_indices[kv_indptr[r] ..
 *                 kv_indptr[r+1]). Must start at 0 and be non-decreasing.
 *  kv_len_host    host int32 [batch], tokens per request; ceil(len / 64) must not exceed the
 *                 request's page count. len 0 is allowed (output 0, lse -inf).
 *  num_heads      query heads: a multiple of 16 in [16, 128].
 *  page_size      must be 64.
 *  num_sms        streaming multiprocessors to plan for; <= 0 queries the current device (a CUDA
 *                 runtime call, also in query mode).
 *  min_splits     lower bound on the number of segments (e.g. 148 to spread one long request over
 *                 every SM); 0 for none.
 *  algo           a qkvp_algo; QKVP_ALGO_AUTO picks the fastest supported family.
 *  workspace      device buffer that receives the work table; NULL makes this a pure host query
 *                 that only fills *plan (including plan->workspace_bytes) and touches no device.
 *  stream         stream of the table upload: an asynchronous copy from one of four library-owned
 *                 pinned buffers (per device, reused once its previous copy has completed), so the
 *                 call does not wait for earlier work on the stream and the host arrays may be
 *                 reused as soon as it returns. If pinned memory is refused it copies from
 *                 pageable memory instead (staged by the runtime before the call returns).
 *
 * Returns QKVP_E_WORKSPACE (with plan->workspace_bytes filled) when workspace is non-NULL but
 * smaller than needed, and QKVP_E_UNSUPPORTED when workspace is non-NULL and `stream` is being
 * captured into a CUDA graph: the upload reads host memory that belongs to this call only, so a
 * replayed graph would read it after it is gone. Plan outside capture; mla_decode_run,
 * mla_decode_attend and mla_decode_combine only launch kernels and may be captured.
 */
int mla_decode_plan(const int32_t* kv_indptr_host, const int32_t* kv_len_host, int32_t batch,
                    int32_t num_heads, int32_t page_size, int32_t kv_dtype, int32_t num_sms,
                    int32_t min_splits, int32_t algo, void* workspace, uint64_t workspace_bytes,
                    qkvp_stream_t stream, qkvp_plan* plan);

/*
 * mla_decode_run - paged MLA decode attention over the quantized pool, for one layer.
 *
 * Computes, per request r and head h over its tokens t < len_r (in natural-log terms),
 *   z_t = sm_scale * g * sum_{d<576} q[r,h,d] * k_t[d]
 *   out[r,h,v] = g * sum_t softmax(z)_t * k_t[v] (v < 512),   lse[r,h] = log sum_t exp(z_t)
 * where k_t is the dequantized latent without the global scale g (g = 1 for FP8 and BF16 pools;
 * "SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "SGLang implementation", item 3: the global
 * scale enters through the matrix-multiply scaling, not per element). The kernels dequantize in
 * registers and run Q.K^T and P.V on the tensor cores with FP16 operands and FP32 accumulation:
 * every dequantized K/V value is exact in FP16, Q is converted from BF16 exactly (a row holding a
 * value of 2^15 or more is first scaled by a power of two, folded into the logit scale), and the
 * probabilities P keep 11 mantissa bits. The softmax runs online in FP32; each segment writes one
 * partial, and partials are merged by log-sum-exp.
 *
 *  plan       from mla_decode_plan with the same kv_dtype, uploaded into this workspace.
 *  q          device bf16 [batch][num_heads][576].
 *  kv_data    device pool for plan->kv_dtype; kv_scale the NVFP4 scale pool (NULL otherwise).
 *  num_pages  pages in the pool; page ids outside [0, num_pages) read as masked tokens.
 *  kv_indices device int32 page ids addressed by the plan's kv_indptr.
 *  sm_scale   logit scale (finite); global_scale: NVFP4 g (> 0, finite), must be 1.0 otherwise.
 *  out, lse   outputs (lse may be NULL).
 *  workspace  the buffer given to mla_decode_plan, at least plan->workspace_bytes.
 */
int mla_decode_run(const qkvp_plan* plan, const void* q, const void* kv_data,
                   const uint8_t* kv_scale, int64_t num_pages, const int32_t* kv_indices,
                   float sm_scale, float global_scale, void* out, float* lse, void* workspace,
                   uint64_t workspace_bytes, qkvp_stream_t stream);

/*
 * mla_decode_attend / mla_decode_combine - the two halves of mla_decode_run, for callers that
 * schedule or time them separately. attend runs the split-KV decode kernel: requests covered by a
 * single segment get their final out/lse, the others leave FP32 partials (normalised output and
 * base-2 log-sum-exp) in the workspace. combine merges those partials by log-sum-exp into out/lse
 * and writes zeros / -inf for empty requests. combine must follow attend on the same stream with
 * the same plan, workspace, global_scale, out and lse. Arguments as for mla_decode_run.
 */
int mla_decode_attend(const qkvp_plan* plan, const void* q, const void* kv_data,
                      const uint8_t* kv_scale, int64_t num_pages, const int32_t* kv_indices,
                      float sm_scale, float global_scale, void* out, float* lse, void* workspace,
                      uint64_t workspace_bytes, qkvp_stream_t stream);
int mla_decode_combine(const qkvp_plan* plan, float global_scale, void* out, float* lse,
                       void* workspace, uint64_t workspace_bytes, qkvp_stream_t stream);

/*
 * mla_decode_noalloc - mla_decode_plan (algo QKVP_ALGO_MMA_SYNC) followed by mla_decode_run, for callers
 * that cannot allocate device memory: a serving loop that has already given every free byte of the
 * GPU to a pre-sized KV pool, or a latency-critical decode step that must not risk the device-wide
 * synchronisation an allocation can bring. The source pages have no counterpart for this call.
 *
 * The work table and the split partials live in one fixed device array of
 * QKVP_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the library holds until
 * the process exits. The call allocates nothing (no cudaMalloc or cudaFree, no allocating library
 * routine, no host heap). Problems that do not fit return QKVP_E_WORKSPACE before any device work:
 * more than QKVP_NOALLOC_MAX_BATCH requests, more than QKVP_NOALLOC_MAX_SEGMENTS segments, or a
 * table plus partials above the array size (at 128 heads, about 250 split partials).
 *
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current, and later calls on that device reuse it: a cudaDeviceReset between calls
 * would leave that address stale, so do not reset a device between calls. Every call shares the
 * one array and leaves its partials there; calls whose GPU work overlaps (different streams or host
 * threads) race on it, so the caller must serialise them. Nothing in the array needs to start at
 * zero: each call uploads its own table and writes every partial before reading it.
 * The table is copied from static, pageable host memory, so the call returns only after the work
 * already queued on `stream` has drained. It returns QKVP_E_UNSUPPORTED while `stream` is being
 * captured into a CUDA graph (a replay would read a host table that later calls overwrite).
 * It runs the mma.sync kernel family with the same split as mla_decode_plan for that family and
 * the same SM count, so its output equals that of plan + run bit for bit.
 * Arguments as for mla_decode_plan and mla_decode_run (page size 64).
 */
#define QKVP_NOALLOC_SCRATCH_BYTES (64ull << 20)
#define QKVP_NOALLOC_MAX_BATCH 8192
#define QKVP_NOALLOC_MAX_SEGMENTS 16384
int mla_decode_noalloc(const int32_t* kv_indptr_host, const int32_t* kv_len_host, int32_t batch,
                       int32_t num_heads, int32_t kv_dtype, int32_t num_sms, int32_t min_splits,
                       const void* q, const void* kv_data, const uint8_t* kv_scale,
                       int64_t num_pages, const int32_t* kv_indices, float sm_scale,
                       float global_scale, void* out, float* lse, qkvp_stream_t stream);

/*
 * kv_pool_cast_bf16 - the cast-then-attend baseline's pool-wide cast: every E4M3 byte of an FP8
 * pool to its BF16 value (exact; NaN bytes 0x7F/0xFF become 0x7FC0). Source: "The Smoking Gun",
 * section "The Investigation Leading to This Message" (k_buffer = pool.to(q.dtype) over the whole
 * [495552, 1, 576] pool, every layer). Used only to measure that baseline.
 *  in  device uint8 [n_elems]; out device uint16 [n_elems]; both 16-byte aligned.
 */
int kv_pool_cast_bf16(const uint8_t* in, int64_t n_elems, void* out, qkvp_stream_t stream);

/*
 * kv_gather_fp8 - the extend path's gather: each request's cached tokens into one contiguous FP8
 * E4M3 workspace, the buffer a chunked-prefill step attends over and that every layer reuses.
 * Source: "SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "SGLang implementation", item 2 (the
 * cached prefix is gathered and dequantized into an FP8 workspace shared across layers, then joined
 * with the current chunk's KV for FP8 attention).
 *   Workspace row tok_indptr[r] + t (t < tok_indptr[r+1] - tok_indptr[r]) is token t of request r,
 *   read from page kv_indices[kv_indptr[r] + t / 64], offset t % 64.
 *   FP8 pool: the bytes are copied. NVFP4 pool: element i becomes E4M3_RNE_satfinite(v) with
 *   v = fp32(scale(block) * e2m1(code)) * global_scale (the first product is exact; the second is one
 *   FP32 rounding): the workspace holds the E4M3 domain the cache was quantized from. The page does
 *   not say how the workspace is scaled; this is the plain reading.
 *  kv_data, kv_scale  device pool as for mla_decode_run (kv_scale NULL for FP8); 16-byte aligned.
 *  kv_dtype           QKVP_KV_FP8_E4M3 or QKVP_KV_NVFP4; global_scale 1 for FP8, finite > 0 for NVFP4.
 *  kv_indptr          device int32 [batch + 1] (pages); kv_indices device int32 [nnz] page ids.
 *  tok_indptr         device int64 [batch + 1], non-decreasing, tok_indptr[0] = 0,
 *                     tok_indptr[batch] = total_tokens (the caller's contract; rows are matched to
 *                     requests by binary search over it).
 *  out                device uint8 [total_tokens][576], 16-byte aligned; every row is written.
 * Every table entry is bounds-checked on the device: a row whose entry lies outside the request's
 * pages, the table (nnz) or the pool (num_pages) is written as zeros. Errors: QKVP_E_INVALID for
 * bad arguments, QKVP_E_UNSUPPORTED for page_size != 64, a BF16 pool or a per-token-scaled pool
 * (whose scale has no place in a plain E4M3 workspace).
 */
int kv_gather_fp8(const void* kv_data, const uint8_t* kv_scale, int32_t kv_dtype, float global_scale,
                  int32_t page_size, int64_t num_pages, const int32_t* kv_indptr, const int32_t* kv_indices,
                  int64_t nnz, const int64_t* tok_indptr, int32_t batch, int64_t total_tokens, uint8_t* out,
                  qkvp_stream_t stream);

/*
 * kv_gather_pages_bf16 - the gather-then-cast baseline: only the pages a batch reads, cast to BF16
 * into a compact pool that a BF16 decode then reads with page ids 0..n_pages-1. Source: "The FP8 KV
 * Cache Wall", sections "The Message" and "Aftermath" (Option B: cast only the active tokens, not
 * the whole pool; measured there at +29%). Used only to measure that baseline.
 *  kv_data   device FP8 pool [num_pages][64][576], 16-byte aligned.
 *  page_ids  device int32 [n_pages]; out device BF16 [n_pages][64][576], 16-byte aligned.
 * Page i of out is pool page page_ids[i] cast exactly (NaN bytes become 0x7FC0); an id outside the
 * pool gives a zero page. Errors: QKVP_E_INVALID for bad arguments, QKVP_E_UNSUPPORTED for
 * page_size != 64.
 */
int kv_gather_pages_bf16(const uint8_t* kv_data, int32_t page_size, int64_t num_pages, const int32_t* page_ids,
                         int64_t n_pages, void* out, qkvp_stream_t stream);

/*
 * qkvp_encode_f32 - the device rounding routines of kv_append_quant applied to raw FP32 values:
 * fmt 1 -> E4M3 (nearest even, saturating at +-448, NaN -> 0x7F); fmt 2 -> E2M1 (nearest even,
 * saturating at +-6, NaN -> 0x0). One code byte per input. Exposed so the rounding can be checked
 * exhaustively against the CPU oracle.
 */
int qkvp_encode_f32(const float* x, int64_t n, int32_t fmt, uint8_t* codes, qkvp_stream_t stream);

/* Static description of a status code; never NULL. */
const char* qkvp_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int qkvp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QKVP_H_ */
