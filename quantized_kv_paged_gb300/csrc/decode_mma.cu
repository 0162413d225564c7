// Split-KV paged MLA decode with warp-level mma.sync (FP16 operands, FP32 accumulate).
//
// The attention computed is the one of the pages' plan()/run() call ("The Smoking Gun", section
// "What Message 1408 Actually Reveals"): per request and head, softmax(sm_scale * q . k) v over the
// request's tokens, K = the whole 576-wide latent and V = its first 512 dims. Pages are read in
// their stored format and dequantized in registers ("SGLang x Qwen x NVIDIA ... NVFP4 KV Cache",
// section "SGLang implementation", item 3); the global NVFP4 scale is folded into the logit scale
// and the output scale.
//
// Operand precision. The pages compute in BF16. Here both products take FP16 operands: every
// dequantized K/V value is exact in FP16, and the softmax probabilities P keep 11 mantissa bits
// instead of 8, which is what holds the output within 2e-2 of the FP64 result when a few tokens
// carry large value channels (|O| ~ 100). Q arrives in BF16 and is converted to FP16 once per CTA
// after multiplying by a power of two 2^-s chosen from the largest |q| of the CTA's heads (so no
// value overflows FP16); 2^s is folded into the logit scale, which keeps the product exact.
//
// Decomposition. A worker owns a list of segments (request, page range). Each worker runs
// H / HC CTAs, one per group of HC query heads (HC = 16..64). Within a CTA, warps come in pairs
// that own the same 16 heads: warp (g, 0) holds output dims 0..255 and computes the logits over
// latent dims 0..287, warp (g, 1) holds output dims 256..511 and computes the logits over dims
// 288..575; the two partial logit tiles are summed through shared memory in a fixed order, so both
// warps see bit-identical logits, maxima and probabilities. Per page:
//   cp.async raw page -> smem  |  dequantize -> FP16 tile [64 tokens][576]  |  S = Q K^T (mma.sync)
//   |  exchange + online softmax (FP32, base 2)  |  O += P V (mma.sync, P from registers).
// The next page's raw bytes are fetched while the current page is multiplied.
#include <cuda.h>          // CUtensorMap and the tensor-map encoder's types (fetched from the driver at run time)
#include <cfloat>
#include <cstdint>
#include <cstring>

#include "qkvp_device.cuh"
#include "qkvp_internal.h"
#include "tc_ptx.cuh"

namespace qkvp {
namespace {

constexpr int kRow = kLatent + 8;          // padded smem row of the 16-bit tiles (1168 bytes)
constexpr int kRowBytes = kRow * 2;
constexpr int kSigByte = kLatent * 2;      // a per-token-scaled page keeps the token's scale here

// FP8 pools take the raw-operand path: no dequantized tile. A page's stored bytes are brought into
// shared memory by four tensor-map loads (TMA), one per 144-dim column box, each box laid out as 64
// rows of 144 bytes: byte (token t, dim d) sits at (d / 144) * 9216 + 144 t + d % 144. A 144-byte
// pitch is nine 16-byte bank groups (an odd number), so eight rows fall in eight distinct groups
// whenever their token indices differ mod 8. K fragments come from a plain ldmatrix of the bytes (4
// consecutive dims per lane: two E4M3 pairs, converted exactly to the two F16x2 registers of an
// m16n8k16 B fragment under a fixed permutation of the contraction dims, which Q's shared-memory copy
// follows), V fragments from the transposing byte ldmatrix (4 consecutive rows per lane: the P.V B
// fragment under a token permutation that the Q.K^T output columns follow, so P passes from the
// logit registers into the A fragments unchanged). Within each 16-token tile, row r of those loads is
// token rho(r) = r ^ 2 for r >= 8 (r below 8): with it, the 8 tokens of every ldmatrix phase are
// distinct mod 8.
// FP8 pools take it at every head count; NVFP4 pools only at 16 heads per CTA: with more head groups
// each group would unpack and scale the same codes again (the FP8 conversion is one instruction per
// pair, the NVFP4 one several), and one shared dequantized tile is cheaper.
template <int KV, int HC>
constexpr bool raw_operands() { return KV == KV_FP8 || KV == KV_FP8PT || (KV == KV_NVFP4 && HC == 16); }
constexpr int kBoxDims = 144;                        // dims per TMA box
constexpr int kBoxBytes = kPage * kBoxDims;          // 9,216
constexpr int kRawRows = 4 * kBoxBytes;              // 36,864; a per-token-scaled page's scales follow
constexpr int kNvScaleOff = 2 * kBoxBytes;          // NVFP4: 288 packed bytes per row in two boxes, then
                                                     // the page's block scales [64][36]
__host__ __device__ constexpr int rho(int r) { return r ^ ((r >> 2) & 2); }
// byte offset of the 16-dim chunk c (0..35) of token row t
__host__ __device__ constexpr int raw_chunk_off(int t, int c) { return (c / 9) * kBoxBytes + t * kBoxDims + (c % 9) * 16; }

template <int KV>
constexpr int raw_bytes() {
  return KV == KV_FP8 ? kRawRows
       : KV == KV_NVFP4 ? kNvScaleOff + kPage * kScales : KV == KV_FP8PT ? kRawRows + 4 * kPage : 0;
}
template <int KV, int HC>
constexpr int tile_bytes() { return raw_operands<KV, HC>() ? 0 : kPage * kRowBytes; }

constexpr int kNT = 256;                   // threads per CTA: every warp dequantizes

// MMA warp pairs of a CTA with HC heads (see the token groups in the kernel).
template <int HC>
constexpr int pairs() { return (HC / 16) * ((HC / 16) >= 3 ? 1 : 4 / (HC / 16)); }

// Token groups per CTA (16 heads: 4 of 16 tokens; 32: 2 of 32; 48 and 64: 1 of 64) and pages per
// iteration: on the raw-operand path with 16 heads each warp takes its 16 tokens of two pages at once
// (twice the independent MMA chains per warp, half the per-page barriers and exchanges).
template <int HC>
constexpr int token_groups() { return (HC / 16) >= 3 ? 1 : 4 / (HC / 16); }
template <int KV, int HC>
constexpr int pages_per_iter() { return raw_operands<KV, HC>() && token_groups<HC>() == 4 ? 2 : 1; }
// Logit exchange buffer of one warp: its partial logits (2 n8 tiles x 4 x 32 floats per 16-token
// tile); two sets (alternate iterations) on the raw-operand path, whose warps run without a CTA-wide
// barrier per page.
template <int KV, int HC>
constexpr int xfloats() {
  // the tile path keeps 1024 floats per warp: its merge slots at segment end reuse this space
  return raw_operands<KV, HC>() ? 256 * (kPage / token_groups<HC>() / 16) * pages_per_iter<KV, HC>() : 1024;
}
template <int KV, int HC>
constexpr int xbuf_bytes() { return pairs<HC>() * 2 * xfloats<KV, HC>() * 4 * (raw_operands<KV, HC>() ? 2 : 1); }

// Raw page buffers: as many as fit up to four (pages fetched that far ahead), at least one.
template <int KV, int HC>
constexpr int raw_bufs_fit(int nb) {
  return HC * kRowBytes + tile_bytes<KV, HC>() + nb * raw_bytes<KV>() + xbuf_bytes<KV, HC>() + 64 <= 232448 - 1024;
}
template <int KV, int HC>
constexpr int raw_bufs() {
  return KV == KV_BF16 ? 0 : raw_bufs_fit<KV, HC>(4) ? 4 : raw_bufs_fit<KV, HC>(3) ? 3 : raw_bufs_fit<KV, HC>(2) ? 2 : 1;
}

template <int KV, int HC>
constexpr int smem_bytes() {
  return HC * kRowBytes + tile_bytes<KV, HC>() + raw_bufs<KV, HC>() * raw_bytes<KV>() + xbuf_bytes<KV, HC>() + 64;
}

// Raw bytes of one page (FP8, per-token-scaled FP8: the page; NVFP4: data then block scales) into a
// raw buffer with bulk
// asynchronous copies, counted on `bar` (one expect-tx arrival by the issuing thread). A page id
// outside the pool copies nothing; the arrival alone completes the phase and the page reads as empty.
template <int KV>
__device__ __forceinline__ void fetch_page(const DecodeArgs& a, int64_t page, uint32_t s_raw, uint32_t bar) {
  if (page < 0 || page >= a.num_pages) {
    tc::mbar_arrive(bar);
    return;
  }
  if (KV == KV_FP8 || KV == KV_FP8PT) {
    tc::mbar_arrive_expect_tx(bar, raw_bytes<KV>());
    tc::bulk_load(s_raw, a.kv + page * raw_bytes<KV>(), raw_bytes<KV>(), bar);
  } else {
    tc::mbar_arrive_expect_tx(bar, kPage * (kPacked + kScales));
    tc::bulk_load(s_raw, a.kv + page * (kPage * kPacked), kPage * kPacked, bar);
    tc::bulk_load(s_raw + kPage * kPacked, a.kv_scale + page * (kPage * kScales), kPage * kScales, bar);
  }
}

// Raw-operand path: the page's 64 rows as four 144-dim boxes (and a per-token-scaled page's 64 scales)
// into a raw buffer, counted on `bar` by one expect-tx arrival of the issuing thread. Rows past the
// page's tokens come along and are zeroed after the wait. A page id outside the pool copies nothing;
// the arrival alone completes the phase.
template <int KV>
__device__ __forceinline__ void fetch_raw_page(const DecodeArgs& a, const CUtensorMap* map, int64_t page,
                                               uint32_t s_raw, uint32_t bar) {
  if (page < 0 || page >= a.num_pages) {
    tc::mbar_arrive(bar);
    return;
  }
  tc::mbar_arrive_expect_tx(bar, raw_bytes<KV>());
  constexpr int kBoxes = KV == KV_NVFP4 ? 2 : 4;
#pragma unroll
  for (int b = 0; b < kBoxes; ++b) tc::tma_load_3d(s_raw + b * kBoxBytes, map, b * kBoxDims, 0, static_cast<int>(page), bar);
  if (KV == KV_FP8PT) tc::bulk_load(s_raw + kRawRows, a.kv + page * kPtPageBytes + kPtScaleOff, 4 * kPage, bar);
  if (KV == KV_NVFP4) tc::bulk_load(s_raw + kNvScaleOff, a.kv_scale + page * (kPage * kScales), kPage * kScales, bar);
}

// Fetch the raw bytes of one page (or, for BF16, the page itself) with cp.async.
template <int KV, int NT>
__device__ __forceinline__ void issue_page(const DecodeArgs& a, int64_t page, int valid,
                                           uint32_t s_raw, uint32_t s_kv, int tid) {
  if (page < 0 || page >= a.num_pages) return;
  if (KV == KV_FP8) {
    const uint8_t* g = a.kv + page * (kPage * kLatent);
    for (int c = tid; c < valid * (kLatent / 16); c += NT) dev::cp_async16(s_raw + c * 16, g + c * 16);
  } else if (KV == KV_NVFP4) {
    const uint8_t* g = a.kv + page * (kPage * kPacked);
    for (int c = tid; c < valid * (kPacked / 16); c += NT) dev::cp_async16(s_raw + c * 16, g + c * 16);
    const uint8_t* gs = a.kv_scale + page * (kPage * kScales);
    for (int c = tid; c < kPage * kScales / 16; c += NT)
      dev::cp_async16(s_raw + kPage * kPacked + c * 16, gs + c * 16);
  } else {
    const uint8_t* g = a.kv + page * (kPage * kLatent * 2);
    for (int c = tid; c < valid * (kLatent * 2 / 16); c += NT) {
      const int row = c / (kLatent * 2 / 16), ch = c % (kLatent * 2 / 16);
      dev::cp_async16(s_kv + row * kRowBytes + ch * 16, g + c * 16);
    }
  }
  dev::cp_async_commit();
}

// Raw page bytes in smem -> FP16 tile rows [0, valid); rows >= valid (or a bad page) -> zeros.
template <int KV, int NT>
__device__ __forceinline__ void dequant_page(const uint8_t* s_raw, uint8_t* s_kv, int valid, int tid) {
  if (KV == KV_FP8) {
    for (int c = tid; c < valid * (kLatent / 16); c += NT) {
      const int row = c / (kLatent / 16), ch = c % (kLatent / 16);
      const uint4 v = *reinterpret_cast<const uint4*>(s_raw + c * 16);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        o[2 * k] = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xFFFFu));
        o[2 * k + 1] = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16));
      }
      uint4* dst = reinterpret_cast<uint4*>(s_kv + row * kRowBytes + ch * 32);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  } else if (KV == KV_FP8PT) {
    // the codes exactly (as FP8), the token scale into the row's padding: it multiplies the token's
    // logit and its probability in FP32, so no operand carries an extra rounding
    for (int c = tid; c < valid * (kLatent / 16); c += NT) {
      const int row = c / (kLatent / 16), ch = c % (kLatent / 16);
      const uint4 v = *reinterpret_cast<const uint4*>(s_raw + c * 16);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        o[2 * k] = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xFFFFu));
        o[2 * k + 1] = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16));
      }
      uint4* dst = reinterpret_cast<uint4*>(s_kv + row * kRowBytes + ch * 32);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
    const float* s_sc = reinterpret_cast<const float*>(s_raw + kPtScaleOff);
    for (int row = tid; row < kPage; row += NT)
      *reinterpret_cast<float*>(s_kv + row * kRowBytes + kSigByte) = row < valid ? s_sc[row] : 0.0f;
  } else if (KV == KV_NVFP4) {
    // one 4-byte word (8 codes, inside one 16-element block) per thread and one 16-byte store: the
    // lanes of a warp write consecutive 16-byte chunks, so the stores are free of bank conflicts
    // (64-byte chunks per thread, stored in order, hit 4-way conflicts that bound this path)
    const uint8_t* s_sc = s_raw + kPage * kPacked;
    constexpr int kWords = kPacked / 4;               // 72 words per row
    for (int c = tid; c < valid * kWords; c += NT) {
      const int row = c / kWords, w = c % kWords;
      const uint32_t v = *reinterpret_cast<const uint32_t*>(s_raw + row * kPacked + 4 * w);
      const uint32_t sb = s_sc[row * kScales + (w >> 1)];
      const uint32_t hs = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(sb | (sb << 8)));
      uint32_t c4[4];
      dev::e2m1x8_to_f16x2x4(v, c4);
      *reinterpret_cast<uint4*>(s_kv + row * kRowBytes + w * 16) =
          make_uint4(dev::hmul2_f16(c4[0], hs), dev::hmul2_f16(c4[1], hs), dev::hmul2_f16(c4[2], hs),
                     dev::hmul2_f16(c4[3], hs));
    }
  } else {
    // BF16 pool: the rows were copied in as BF16; convert them to FP16 in place
    for (int c = tid; c < valid * (kLatent * 2 / 16); c += NT) {
      const int row = c / (kLatent * 2 / 16), ch = c % (kLatent * 2 / 16);
      uint4* p = reinterpret_cast<uint4*>(s_kv + row * kRowBytes + ch * 16);
      const uint4 v = *p;
      *p = make_uint4(dev::bf16x2_to_f16x2(v.x), dev::bf16x2_to_f16x2(v.y), dev::bf16x2_to_f16x2(v.z),
                      dev::bf16x2_to_f16x2(v.w));
    }
  }
  // zero the rows past the valid tokens (their bytes are never read into the result)
  for (int c = tid; c < (kPage - valid) * (kLatent * 2 / 16); c += NT) {
    const int row = valid + c / (kLatent * 2 / 16), ch = c % (kLatent * 2 / 16);
    *reinterpret_cast<uint4*>(s_kv + row * kRowBytes + ch * 16) = make_uint4(0, 0, 0, 0);
  }
}

// ---- FP8 Q.K^T (QKVP_ALGO_MMA_FP8): Q as two E4M3 terms, K straight from the FP8 page ----
// D += A B, m16n8k32, E4M3 inputs, FP32 accumulators. A (16 x 32, row): a0 / a1 rows g and g + 8 of
// k 4t .. 4t + 3, a2 / a3 the same rows at k 16 + 4t ..; B (32 x 8, col): b0 k 4t .. 4t + 3, b1 k 16 +
// 4t .. of column g (g = lane / 4, t = lane % 4); D as for m16n8k16.
__device__ __forceinline__ void mma_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The power of two sc = 2^floor(log2(448 / max|q|)) of a head row from its largest |q| (BF16 magnitude
// bits): the row times sc has its largest magnitude in (224, 448]. All-zero and non-finite rows use 1.
__device__ __forceinline__ float f8_row_scale(uint32_t mbits) {
  if (mbits == 0u || mbits >= 0x7F80u) return 1.0f;
  const float x = __fdiv_rn(448.0f, __uint_as_float(mbits << 16));   // exact IEEE quotient
  const int e = static_cast<int>((__float_as_uint(x) >> 23) & 0xFFu);  // floor(log2(x)) + 127 (x normal)
  return __uint_as_float(static_cast<uint32_t>(min(max(e, 1), 254)) << 23);
}

// Two FP32 values scaled into E4M3 range -> (hi pair, lo pair): hi = E4M3(x), lo = E4M3(16 (x - hi)),
// both rounded to nearest even (the difference and the factor 16 are exact in FP32). Low byte = x0.
__device__ __forceinline__ void f8_two_term(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = dev::f32x2_to_e4m3x2(x0, x1);
  const uint32_t d = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(hi));
  const float d0 = __half2float(__ushort_as_half(static_cast<unsigned short>(d & 0xFFFFu)));
  const float d1 = __half2float(__ushort_as_half(static_cast<unsigned short>(d >> 16)));
  lo = dev::f32x2_to_e4m3x2((x0 - d0) * 16.0f, (x1 - d1) * 16.0f);
}

template <int KV, int HC, bool F8>
__global__ void __launch_bounds__(kNT, 1) decode_mma_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kv_map) {
  static_assert(!F8 || ((KV == KV_FP8 || KV == KV_FP8PT) && HC <= 32), "FP8 Q.K^T: FP8 pools, 16 or 32 heads per CTA");
  constexpr int NG = HC / 16;       // 16-head groups in this CTA
  // With few heads the page's 64 tokens are split among warp pairs too, so that all 8 warps do
  // math: TG token groups of TPG tokens, each pair with its own softmax state, merged at the end
  // of a segment. 16 heads: 4 x 16 tokens; 32: 2 x 32; 48 and 64: 1 x 64.
  constexpr int TG = token_groups<HC>();
  constexpr int NPAIR = NG * TG;
  constexpr int TPG = kPage / TG;
  constexpr int NP = TPG / 16;      // 16-token tiles per token group
  constexpr int NT = kNT;
  constexpr int NB = raw_bufs<KV, HC>();
  constexpr int NBx = NB > 0 ? NB : 1;
  constexpr bool RAW = raw_operands<KV, HC>();
  constexpr int PPI = pages_per_iter<KV, HC>();   // pages per iteration
  constexpr int NPI = NP * PPI;                   // 16-token tiles per warp per iteration
  constexpr int XF = xfloats<KV, HC>();
  static_assert(2 * NPI * 4 * 32 <= XF, "exchange buffer");
  static_assert(PPI == 1 || NB >= 2 * PPI, "two pages in flight ahead of the pair in use");
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* s_q = smem;
  uint8_t* s_kv = s_q + HC * kRowBytes;      // the dequantized page tile (not on the raw-operand path)
  uint8_t* s_raw = s_kv + tile_bytes<KV, HC>();
  float* s_x = reinterpret_cast<float*>(s_raw + NB * raw_bytes<KV>());
  uint32_t* s_qmax = reinterpret_cast<uint32_t*>(s_x + NPAIR * 2 * XF * (RAW ? 2 : 1));
  // NB FULL barriers, then (raw-operand path) NB EMPTY barriers: 8-byte aligned
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_qmax + 2);
  const uint32_t a_q = dev::smem_u32(s_q), a_kv = dev::smem_u32(s_kv), a_raw = dev::smem_u32(s_raw);
  const uint32_t a_bar = dev::smem_u32(s_bar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pi = warp >> 1, half = warp & 1;
  const int grp = pi % NG, tg = pi / NG;  // head group and token group of this warp's pair
  const int t0 = tg * TPG;                // first token of the page this pair attends
  const int g8 = lane >> 2, t4 = lane & 3;
  const int worker = blockIdx.x / a.ctas_per_worker;
  const int h0 = (blockIdx.x % a.ctas_per_worker) * HC;
  const int seg_b = a.worker_ptr[worker], seg_e = a.worker_ptr[worker + 1];
  const bool mma_warp = warp < 2 * NPAIR;
  if (KV != KV_BF16 && tid == 0) {
    for (int b = 0; b < NB; ++b) tc::mbar_init(a_bar + 8 * b, 1);
    if (RAW)
      for (int b = 0; b < NB; ++b) tc::mbar_init(a_bar + 8 * (NB + b), NT / 32);   // one arrival per warp
    tc::fence_mbar_init();
  }
  int fills[NBx];                   // completed phases of each raw buffer's barrier
#pragma unroll
  for (int b = 0; b < NBx; ++b) fills[b] = 0;

  // ldmatrix lane addresses (bytes, relative to the tile bases)
  const uint32_t q_lane = ((grp * 16 + (lane & 15)) * kRow + (lane >> 4) * 8) * 2;
  // FP8 Q planes: row r keeps its hi bytes at [0, 576) and its lo bytes at [576, 1152) of the row
  const uint32_t q8_lane = (grp * 16 + (lane & 15)) * kRowBytes + (lane >> 4) * 16;
  float qf8[2] = {0.0f, 0.0f};      // FP8 Q.K^T: logit factor (sm_scale g log2 e / sc) of rows g8, g8 + 8
  const uint32_t k_lane = (((lane & 7) + ((lane >> 4) << 3)) * kRow + ((lane >> 3) & 1) * 8) * 2;
  const uint32_t v_lane = (((lane & 7) + ((lane >> 3) & 1) * 8) * kRow + half * 256 + (lane >> 4) * 8) * 2;
  float* const x_mine0 = s_x + (pi * 2 + half) * XF;
  float* const x_peer0 = s_x + (pi * 2 + (half ^ 1)) * XF;

  int cur_req = -1;
  float q_scale_log2 = a.scale_log2;
  for (int si = seg_b; si < seg_e; ++si) {
    const Segment seg = a.segs[si];
    __syncthreads();  // the previous segment is done with s_q / s_kv / s_raw
    if (seg.req != cur_req) {
      const uint8_t* gq = reinterpret_cast<const uint8_t*>(a.q) + (static_cast<int64_t>(seg.req) * a.heads + h0) * kLatent * 2;
      // (the FP8 Q.K^T stages the BF16 rows densely in the first raw buffer, free until this
      // segment's pages are fetched, and converts them into the Q area)
      for (int c = tid; c < HC * (kLatent * 2 / 16); c += NT) {
        const int row = c / (kLatent * 2 / 16), ch = c % (kLatent * 2 / 16);
        const uint32_t dst = F8 ? a_raw + row * (kLatent * 2) + ch * 16 : a_q + row * kRowBytes + ch * 16;
        dev::cp_async16(dst, gq + static_cast<int64_t>(row) * kLatent * 2 + ch * 16);
      }
      dev::cp_async_commit();
      if (tid == 0) *s_qmax = 0u;
      if (F8)
        for (int r = tid; r < HC; r += NT) reinterpret_cast<uint32_t*>(s_x)[r] = 0u;
      dev::cp_async_wait_all();
      __syncthreads();
      // largest |q| of this CTA's heads, as BF16 magnitude bits (integer order = magnitude order)
      uint32_t mx = 0;
      for (int c = F8 ? NT * HC * kLatent : tid; c < HC * (kLatent * 2 / 16); c += NT) {
        const int row = c / (kLatent * 2 / 16), ch = c % (kLatent * 2 / 16);
        const uint4 v = *reinterpret_cast<const uint4*>(s_q + row * kRowBytes + ch * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
      }
      mx = __reduce_max_sync(0xffffffffu, mx);
      if (lane == 0) atomicMax(s_qmax, mx);
      __syncthreads();
      // q * 2^-s puts the largest |q| in [2^14, 2^15); inf / NaN / all-zero tiles keep s = 0
      const uint32_t qm = *s_qmax;
      int sh = 0;
      if (qm != 0u && qm < 0x7F80u) sh = max(-100, min(113, static_cast<int>(qm >> 7) - 127 - 14));
      const float down = __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
      q_scale_log2 = a.scale_log2 * __uint_as_float(static_cast<uint32_t>(127 + sh) << 23);
      if constexpr (F8) {
        // Q as two E4M3 terms per head row (sc = f8_row_scale of the row's largest |q|):
        // hi = E4M3(q sc), lo = E4M3(16 (q sc - hi)), q ~ (hi + lo / 16) / sc, from the BF16 rows
        // staged in the first raw buffer into the Q area (hi at bytes [0, 576) of a row, lo at
        // [576, 1152)).
        static_assert(!F8 || HC * kLatent * 2 <= raw_bytes<KV>(), "Q staging fits one raw buffer");
        const uint8_t* qst = s_raw;
        uint32_t* rmax = reinterpret_cast<uint32_t*>(s_x);
        for (int c = tid; c < HC * (kLatent * 2 / 16); c += NT) {
          const int row = c / (kLatent * 2 / 16);
          const uint4 v = reinterpret_cast<const uint4*>(qst)[c];
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          uint32_t m = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) m = max(m, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
          atomicMax(rmax + row, m);
        }
        __syncthreads();
        for (int c = tid; c < HC * (kLatent / 16); c += NT) {
          const int row = c / (kLatent / 16), ch = c % (kLatent / 16);
          const float sc = f8_row_scale(rmax[row]);
          const uint4 v0 = reinterpret_cast<const uint4*>(qst)[2 * c];
          const uint4 v1 = reinterpret_cast<const uint4*>(qst)[2 * c + 1];
          const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          uint32_t hv[4], lv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {       // dims 4k .. 4k + 3 of the chunk
            uint32_t h01, l01, h23, l23;
            f8_two_term(__uint_as_float(w[2 * k] << 16) * sc, __uint_as_float(w[2 * k] & 0xFFFF0000u) * sc, h01, l01);
            f8_two_term(__uint_as_float(w[2 * k + 1] << 16) * sc, __uint_as_float(w[2 * k + 1] & 0xFFFF0000u) * sc, h23, l23);
            hv[k] = (h01 & 0xFFFFu) | (h23 << 16);
            lv[k] = (l01 & 0xFFFFu) | (l23 << 16);
          }
          *reinterpret_cast<uint4*>(s_q + row * kRowBytes + ch * 16) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          *reinterpret_cast<uint4*>(s_q + row * kRowBytes + kLatent + ch * 16) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint32_t m = rmax[grp * 16 + g8 + 8 * r];
          qf8[r] = m >= 0x7F80u ? __uint_as_float(0x7FC00000u) : __fdiv_rn(a.scale_log2, f8_row_scale(m));
        }
      } else if constexpr (RAW && KV == KV_NVFP4) {
        // NVFP4 raw-operand path: within every 32 dims (16 dim pairs), pair position i holds pair
        // 4(i % 4) + i / 4, the order a lane's K fragment bytes come in (a 4 x 4 transpose)
        for (int c = tid; c < HC * (kLatent / 32); c += NT) {
          const int row = c / (kLatent / 32), ch = c % (kLatent / 32);
          uint4* p = reinterpret_cast<uint4*>(s_q + row * kRowBytes + ch * 64);
          uint32_t w[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 v = p[u];
            w[4 * u] = v.x; w[4 * u + 1] = v.y; w[4 * u + 2] = v.z; w[4 * u + 3] = v.w;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            p[u] = make_uint4(dev::bf16x2_to_f16x2(w[u], down), dev::bf16x2_to_f16x2(w[4 + u], down),
                              dev::bf16x2_to_f16x2(w[8 + u], down), dev::bf16x2_to_f16x2(w[12 + u], down));
        }
      } else if constexpr (RAW) {
        // raw-operand path: within every 16 dims, position 2a + e holds dim 4a + e and position
        // 8 + 2a + e holds dim 4a + 2 + e (a < 4, e < 2), the order a lane's K fragment bytes come in
        for (int c = tid; c < HC * (kLatent / 16); c += NT) {
          const int row = c / (kLatent / 16), ch = c % (kLatent / 16);
          uint4* p = reinterpret_cast<uint4*>(s_q + row * kRowBytes + ch * 32);
          const uint4 v0 = p[0], v1 = p[1];
          p[0] = make_uint4(dev::bf16x2_to_f16x2(v0.x, down), dev::bf16x2_to_f16x2(v0.z, down),
                            dev::bf16x2_to_f16x2(v1.x, down), dev::bf16x2_to_f16x2(v1.z, down));
          p[1] = make_uint4(dev::bf16x2_to_f16x2(v0.y, down), dev::bf16x2_to_f16x2(v0.w, down),
                            dev::bf16x2_to_f16x2(v1.y, down), dev::bf16x2_to_f16x2(v1.w, down));
        }
      } else {
        for (int c = tid; c < HC * (kLatent * 2 / 16); c += NT) {
          const int row = c / (kLatent * 2 / 16), ch = c % (kLatent * 2 / 16);
          uint4* p = reinterpret_cast<uint4*>(s_q + row * kRowBytes + ch * 16);
          const uint4 v = *p;
          *p = make_uint4(dev::bf16x2_to_f16x2(v.x, down), dev::bf16x2_to_f16x2(v.y, down),
                          dev::bf16x2_to_f16x2(v.z, down), dev::bf16x2_to_f16x2(v.w, down));
        }
      }
      cur_req = seg.req;
      // every warp reads Q (ldmatrix) only after every thread's conversion (and, for the FP8 Q.K^T,
      // its read of the row maxima in the exchange buffer) is done
      __syncthreads();
    }
    float o[32][4];
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.0f, 0.0f};

    // raw pages of this segment stream in NB ahead of the page being used
    if constexpr (RAW) {
      if (tid == 0) {
        for (int k = 0; k < NB && k < seg.num_pages; ++k)
          fetch_raw_page<KV>(a, &kv_map, a.kv_indices[seg.page_begin + k], a_raw + k * raw_bytes<KV>(), a_bar + 8 * k);
      }
    } else if (KV != KV_BF16 && tid == 0) {
      for (int k = 0; k < NB && k < seg.num_pages; ++k)
        fetch_page<KV>(a, a.kv_indices[seg.page_begin + k], a_raw + k * raw_bytes<KV>(), a_bar + 8 * k);
    }
    int64_t page = a.kv_indices[seg.page_begin];
    for (int j = 0; j < seg.num_pages; j += PPI) {
      if (RAW && tid == 0 && j >= PPI) {
        // the buffers of the previous iteration's pages take the pages NB further on once every warp
        // is done with them (each buffer's fills[]-th use: EMPTY completes once per use)
#pragma unroll
        for (int u = 0; u < PPI; ++u) {
          const int pp = j - PPI + u;
          if (pp + NB < seg.num_pages) {
            const int pb = pp % NBx;
            if (!tc::mbar_wait(a_bar + 8 * (NB + pb), (fills[pb] - 1) & 1)) atomicOr(a.status, 16);
            tc::fence_proxy_async_smem();
            fetch_raw_page<KV>(a, &kv_map, a.kv_indices[seg.page_begin + pp + NB], a_raw + pb * raw_bytes<KV>(),
                               a_bar + 8 * pb);
          }
        }
      }
      // this iteration's pages: buffer, valid tokens (0 past the segment: such a tile reads page j's
      // buffer and is masked whole)
      int live_u[PPI], buf_u[PPI];
      uint32_t rb_u[PPI];
      uint8_t* rbuf_u[PPI];
      bool any_partial = false;
#pragma unroll
      for (int u = 0; u < PPI; ++u) {
        const int jp = j + u;
        const bool has = jp < seg.num_pages;
        const int64_t pg_u = u == 0 ? page : (has ? static_cast<int64_t>(a.kv_indices[seg.page_begin + jp]) : -1);
        const int valid_u = has ? min(kPage, seg.num_tokens - jp * kPage) : 0;
        buf_u[u] = NB > 0 ? (has ? jp : j) % NB : 0;
        if (has) {
          if (KV == KV_BF16) {
            issue_page<KV, NT>(a, pg_u, valid_u, a_raw, a_kv, tid);
            dev::cp_async_wait_all();
          } else {
            // bounded wait: a timeout sets a status bit, and the page then reads as whatever is there
            if (!tc::mbar_wait(a_bar + 8 * buf_u[u], fills[buf_u[u]] & 1)) {
              if (lane == 0) atomicOr(a.status, 16);
            }
            ++fills[buf_u[u]];
          }
        }
        live_u[u] = (pg_u >= 0 && pg_u < a.num_pages) ? valid_u : 0;
        rb_u[u] = a_raw + buf_u[u] * raw_bytes<KV>();
        rbuf_u[u] = s_raw + buf_u[u] * raw_bytes<KV>();
        any_partial |= has && live_u[u] < kPage;
      }
      const int live = live_u[0];
      const int buf = buf_u[0];
      uint8_t* rbuf = rbuf_u[0];
      const uint32_t a_rb = rb_u[0];
      // tile p of this iteration: page j + p / NP, tokens t0 + 16 (p % NP) of it
      auto tt0 = [&](int p) { return t0 + 16 * (p % NP); };
      auto trb = [&](int p) { return rb_u[p / NP]; };
      auto trbuf = [&](int p) { return rbuf_u[p / NP]; };
      auto tlive = [&](int p) { return live_u[p / NP]; };
      // logit exchange buffers of this iteration (two sets on the raw-operand path: a warp may write
      // iteration i + 1's while its peer still reads iteration i's; i + 2 waits for the pair barrier of
      // i + 1)
      float* x_mine = x_mine0 + (RAW && ((j / PPI) & 1) ? NPAIR * 2 * XF : 0);
      float* x_peer = x_peer0 + (RAW && ((j / PPI) & 1) ? NPAIR * 2 * XF : 0);
      if constexpr (RAW) {
        // rows past a page's tokens (and their scales) read as zeros: P is 0 there, and V must not
        // bring NaN codes into P.V
        if (any_partial) {
#pragma unroll
          for (int u = 0; u < PPI; ++u) {
            if (j + u >= seg.num_pages || live_u[u] >= kPage) continue;
            uint8_t* rb = rbuf_u[u];
            const int lv = live_u[u];
            constexpr int kChunks = KV == KV_NVFP4 ? kPacked / 16 : kLatent / 16;
            for (int c = tid; c < (kPage - lv) * kChunks; c += NT) {
              const int t = lv + c / kChunks, ch = c % kChunks;
              *reinterpret_cast<uint4*>(rb + raw_chunk_off(t, ch)) = make_uint4(0, 0, 0, 0);
            }
            if (KV == KV_FP8PT)
              for (int t = lv + tid; t < kPage; t += NT) reinterpret_cast<float*>(rb + kRawRows)[t] = 0.0f;
            if (KV == KV_NVFP4)      // block scales too: an unused slot's scale may be the NaN code
              for (int c = tid; c < (kPage - lv) * (kScales / 4); c += NT)
                reinterpret_cast<uint32_t*>(rb + kNvScaleOff + lv * kScales)[c] = 0u;
          }
          __syncthreads();
        }
        if (j + PPI < seg.num_pages) page = a.kv_indices[seg.page_begin + j + PPI];
      } else {
        __syncthreads();
        dequant_page<KV, NT>(rbuf, s_kv, live, tid);
        __syncthreads();
        if (j + 1 < seg.num_pages) page = a.kv_indices[seg.page_begin + j + 1];
        if (KV != KV_BF16 && tid == 0 && j + NB < seg.num_pages) {
          tc::fence_proxy_async_smem();   // this buffer's reads are done before the copy refills it
          fetch_page<KV>(a, a.kv_indices[seg.page_begin + j + NB], a_rb, a_bar + 8 * buf);
        }
      }
      if (mma_warp) {

      // ---- S partial = Q[:, my dims] K[my tokens, my dims]^T  (16 heads x TPG tokens) ----
      float s[2 * NPI][4];
#pragma unroll
      for (int n = 0; n < 2 * NPI; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.0f;
      if constexpr (F8) {
        // FP8 Q.K^T: per 32-dim k-step an m16n8k32 E4M3 MMA with the hi plane of Q into s and one with
        // the lo plane into s2, both with the page's own bytes as B. The byte ldmatrix of the raw
        // path gives lane l, per 16-dim chunk, dims 4t4 .. 4t4 + 3 of the row of logit column g8:
        // chunks 2u and 2u + 1 of a block of four are the b0 / b1 of k-step u. Q needs no permutation.
        const int kr = lane & 7;
        float s2[2 * NPI][4];
#pragma unroll
        for (int n = 0; n < 2 * NPI; ++n) s2[n][0] = s2[n][1] = s2[n][2] = s2[n][3] = 0.0f;
#pragma unroll
        for (int kb = 0; kb < 5; ++kb) {       // 16-dim chunks 4kb .. 4kb + 3 of the half (two in the last)
          uint32_t ah[2][4], al[2][4];
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (2 * kb + u < 9) {
              const uint32_t qa = a_q + q8_lane + half * 288 + 32 * (2 * kb + u);
              dev::ldsm_x4(qa, ah[u][0], ah[u][1], ah[u][2], ah[u][3]);
              dev::ldsm_x4(qa + kLatent, al[u][0], al[u][1], al[u][2], al[u][3]);
            }
#pragma unroll
          for (int p = 0; p < NPI; ++p)
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const uint32_t addr = trb(p) + raw_chunk_off(tt0(p) + rho(4 * (kr >> 1) + (kr & 1) + 2 * jj),
                                                           half * 18 + 4 * kb + (lane >> 3));
              uint32_t r[4];
              if (kb < 4) dev::ldsm_x4(addr, r[0], r[1], r[2], r[3]);
              else dev::ldsm_x2(addr, r[0], r[1]);
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                if (2 * kb + u >= 9) continue;
                mma_e4m3(s[2 * p + jj], ah[u], r[2 * u], r[2 * u + 1]);
                mma_e4m3(s2[2 * p + jj], al[u], r[2 * u], r[2 * u + 1]);
              }
            }
        }
#pragma unroll
        for (int n = 0; n < 2 * NPI; ++n)
#pragma unroll
          for (int i = 0; i < 4; ++i) s[n][i] = fmaf(s2[n][i], 0.0625f, s[n][i]);
      } else if constexpr (RAW && KV == KV_NVFP4) {
        // NVFP4: a 16-byte chunk c of a row is 32 dims, two 16-element blocks. As for FP8, lane l
        // addresses row rho(4((l & 7) >> 1) + (l & 1) + 2jj) of tile p, chunk (l >> 3) of a pair; it
        // receives bytes 4t4 .. 4t4+3 of the row of logit column g8: dims 32c + 8t4 .. +7, all in
        // block 2c + (t4 >> 1). Bytes 4t4, 4t4+1 form the B fragment of k-step 2c, bytes 4t4+2,
        // 4t4+3 that of k-step 2c + 1 (Q is stored to match); each code pair times the block scale
        // in F16 is exact.
        const int kr = lane & 7;
        constexpr bool kSplit = NPI <= 2;
        float s2[kSplit ? 2 * NPI : 1][4];
#pragma unroll
        for (int n = 0; n < (kSplit ? 2 * NPI : 1); ++n) s2[n][0] = s2[n][1] = s2[n][2] = s2[n][3] = 0.0f;
#pragma unroll
        for (int cb = 0; cb < 5; ++cb) {       // chunks 2cb, 2cb + 1 of the half's nine (one in the last)
          constexpr int kChunks = 9;
          uint32_t aq[4][4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (2 * cb + i / 2 < kChunks)
              dev::ldsm_x4(a_q + q_lane + (half * 288 + 16 * (4 * cb + i)) * 2, aq[i][0], aq[i][1], aq[i][2], aq[i][3]);
#pragma unroll
          for (int p = 0; p < NPI; ++p)
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const uint32_t addr = trb(p) + raw_chunk_off(tt0(p) + rho(4 * (kr >> 1) + (kr & 1) + 2 * jj),
                                                           half * 9 + 2 * cb + (lane >> 3));
              const int mytok = tt0(p) + rho(4 * (g8 >> 1) + (g8 & 1) + 2 * jj);
              const uint8_t* sc = trbuf(p) + kNvScaleOff;
              uint32_t r[2];
              if (cb < 4) dev::ldsm_x2(addr, r[0], r[1]);
              else dev::ldsm_x1(addr, r[0]);
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                if (2 * cb + u >= kChunks) continue;
                const uint32_t sb = sc[mytok * kScales + 2 * (half * 9 + 2 * cb + u) + (t4 >> 1)];
                const uint32_t sh2 = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(sb | (sb << 8)));
                uint32_t c4[4];
                dev::e2m1x8_to_f16x2x4(r[u], c4);
                dev::mma_f16(s[2 * p + jj], aq[2 * u][0], aq[2 * u][1], aq[2 * u][2], aq[2 * u][3],
                             dev::hmul2_f16(c4[0], sh2), dev::hmul2_f16(c4[1], sh2));
                dev::mma_f16(kSplit ? s2[kSplit ? 2 * p + jj : 0] : s[2 * p + jj],
                             aq[2 * u + 1][0], aq[2 * u + 1][1], aq[2 * u + 1][2], aq[2 * u + 1][3],
                             dev::hmul2_f16(c4[2], sh2), dev::hmul2_f16(c4[3], sh2));
              }
            }
        }
        if constexpr (kSplit) {
#pragma unroll
          for (int n = 0; n < 2 * NPI; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) s[n][i] += s2[n][i];
        }
      } else if constexpr (RAW) {
        // K fragments straight from the page bytes: per 16-token tile p and n8 tile jj, lane l
        // addresses tile row rho(4((l & 7) >> 1) + (l & 1) + 2jj), k-step (l >> 3) of a block of
        // four; it receives dims 4t4 .. 4t4+3 of the row of logit column g8, i.e. B[2t4, 2t4+1] and
        // B[8 + 2t4, 9 + 2t4] in Q's permuted dim order
        const int kr = lane & 7;
        // with one or two 16-token tiles, odd k-steps accumulate apart: twice the independent
        // chains of dependent MMAs (four tiles have enough already)
        constexpr bool kSplit = NPI <= 2;
        float s2[kSplit ? 2 * NPI : 1][4];
#pragma unroll
        for (int n = 0; n < (kSplit ? 2 * NPI : 1); ++n) s2[n][0] = s2[n][1] = s2[n][2] = s2[n][3] = 0.0f;
#pragma unroll
        for (int kb = 0; kb < 5; ++kb) {       // k-steps 4kb .. 4kb + 3 (two in the last block)
          constexpr int kSteps = 18;
          uint32_t aq[4][4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (4 * kb + i < kSteps)
              dev::ldsm_x4(a_q + q_lane + (half * 288 + 16 * (4 * kb + i)) * 2, aq[i][0], aq[i][1], aq[i][2], aq[i][3]);
#pragma unroll
          for (int p = 0; p < NPI; ++p)
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const uint32_t addr = trb(p) + raw_chunk_off(tt0(p) + rho(4 * (kr >> 1) + (kr & 1) + 2 * jj),
                                                           half * 18 + 4 * kb + (lane >> 3));
              uint32_t r[4];
              if (kb < 4) dev::ldsm_x4(addr, r[0], r[1], r[2], r[3]);
              else dev::ldsm_x2(addr, r[0], r[1]);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (4 * kb + i < kSteps)
                  dev::mma_f16((kSplit && (i & 1)) ? s2[kSplit ? 2 * p + jj : 0] : s[2 * p + jj], aq[i][0], aq[i][1], aq[i][2], aq[i][3],
                               dev::e4m3x2_to_f16x2(static_cast<uint16_t>(r[i] & 0xFFFFu)),
                               dev::e4m3x2_to_f16x2(static_cast<uint16_t>(r[i] >> 16)));
            }
        }
        if constexpr (kSplit) {
#pragma unroll
          for (int n = 0; n < 2 * NPI; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) s[n][i] += s2[n][i];
        }
      } else {
#pragma unroll 2
      for (int ks = 0; ks < 18; ++ks) {
        const int kk = half * 288 + ks * 16;
        uint32_t a0, a1, a2, a3;
        dev::ldsm_x4(a_q + q_lane + kk * 2, a0, a1, a2, a3);
#pragma unroll
        for (int p = 0; p < NPI; ++p) {
          uint32_t b0, b1, b2, b3;
          dev::ldsm_x4(a_kv + k_lane + ((t0 + p * 16) * kRow + kk) * 2, b0, b1, b2, b3);
          dev::mma_f16(s[2 * p], a0, a1, a2, a3, b0, b1);
          dev::mma_f16(s[2 * p + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      }
      // ---- exchange the partial logits with the peer warp; sum in a fixed order ----
#pragma unroll
      for (int n = 0; n < 2 * NPI; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) x_mine[(n * 4 + i) * 32 + lane] = s[n][i];
      dev::named_bar_sync(1 + pi, 64);
#pragma unroll
      for (int n = 0; n < 2 * NPI; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float peer = x_peer[(n * 4 + i) * 32 + lane];
          s[n][i] = half == 0 ? (s[n][i] + peer) : (peer + s[n][i]);
        }
      // ---- online softmax in base 2 (rows g8 and g8 + 8 of the 16 heads) ----
      // per-token-scaled pages: the token scale multiplies the logit and the probability (not l)
      // page token of logit column 2t4 + e of n8 tile n: on the raw-operand path tile 2p + jj holds
      // tile rows {0,1,4,5,8,9,12,13} + 2jj (the order the P.V B fragments take them in), through rho
      auto tok_of = [&](int n, int e) {
        return RAW ? tt0(n >> 1) + rho(4 * t4 + e + 2 * (n & 1)) : t0 + n * 8 + 2 * t4 + e;
      };
      float sig[2 * NPI][2];
#pragma unroll
      for (int n = 0; n < 2 * NPI; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          sig[n][e] = KV != KV_FP8PT ? 1.0f
              : RAW ? reinterpret_cast<const float*>(trbuf(n >> 1) + kRawRows)[tok_of(n, e)]
                    : *reinterpret_cast<const float*>(s_kv + tok_of(n, e) * kRowBytes + kSigByte);
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < 2 * NPI; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tok = tok_of(n, i & 1);
          const float x = KV == KV_FP8PT ? s[n][i] * sig[n][i & 1] : s[n][i];
          const float v = tok < (RAW ? tlive(n >> 1) : live) ? x * (F8 ? qf8[i >> 1] : q_scale_log2) : -INFINITY;
          s[n][i] = v;
          mx[i >> 1] = fmaxf(mx[i >> 1], v);
        }
      float alpha[2], mref[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float m_new = fmaxf(m_r[r], mx[r]);
        mref[r] = m_new == -INFINITY ? 0.0f : m_new;
        alpha[r] = dev::fast_exp2(m_r[r] - mref[r]);
        m_r[r] = m_new;
        l_r[r] *= alpha[r];
      }
#pragma unroll
      for (int n = 0; n < 2 * NPI; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float p = dev::fast_exp2(s[n][i] - mref[i >> 1]);
          s[n][i] = p;
          l_r[i >> 1] += p;
        }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        o[i][0] *= alpha[0]; o[i][1] *= alpha[0];
        o[i][2] *= alpha[1]; o[i][3] *= alpha[1];
      }
      // ---- O[:, my 256 dims] += P V ----
#pragma unroll
      for (int kt = 0; kt < NPI; ++kt) {
        const float* sa = sig[2 * kt];
        const float* sb = sig[2 * kt + 1];
        const uint32_t pa0 = dev::pack_f16x2(s[2 * kt][0] * sa[0], s[2 * kt][1] * sa[1]);
        const uint32_t pa1 = dev::pack_f16x2(s[2 * kt][2] * sa[0], s[2 * kt][3] * sa[1]);
        const uint32_t pa2 = dev::pack_f16x2(s[2 * kt + 1][0] * sb[0], s[2 * kt + 1][1] * sb[1]);
        const uint32_t pa3 = dev::pack_f16x2(s[2 * kt + 1][2] * sb[0], s[2 * kt + 1][3] * sb[1]);
        if constexpr (RAW && KV == KV_NVFP4) {
          // NVFP4 V fragments: the transposing byte ldmatrix gives lane l, per 16-byte chunk (32
          // dims), tile rows 4t4 .. 4t4+3 of byte column g8 (dims 2g8, 2g8 + 1: low and high
          // nibbles) and of byte column 8 + g8 (dims 16 + 2g8, 17 + 2g8). Nibble shuffles pair
          // the four tokens' codes per dim; each code pair times its two tokens' block scales in
          // F16 is exact. Output tiles come per dim parity: o[4c] holds dims 32c + 2n, o[4c + 1]
          // dims 32c + 2n + 1, o[4c + 2] and o[4c + 3] the same 16 dims higher (c = chunk of the
          // warp's 256 dims); the epilogue writes them back in order.
          const int vt = tt0(kt) + rho(lane & 15);
          const uint8_t* sc = trbuf(kt) + kNvScaleOff;
          int stok[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) stok[u] = tt0(kt) + rho(4 * t4 + u);
#pragma unroll
          for (int vq = 0; vq < 4; ++vq) {        // chunks 2vq, 2vq + 1 of the warp's eight
            uint32_t r[4];
            dev::ldsm_t8_x2(trb(kt) + raw_chunk_off(vt, half * 8 + 2 * vq + (lane >> 4)), r[0], r[1], r[2], r[3]);
            // the four tokens' scales of blocks 2c .. 2c + 3 (c = the pair's first chunk in the row)
            const int blk0 = 2 * (half * 8 + 2 * vq);
            uint32_t sw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) sw[u] = *reinterpret_cast<const uint32_t*>(sc + stok[u] * kScales + blk0);
#pragma unroll
            for (int m = 0; m < 4; ++m) {          // r[m]: chunk 2vq + m / 2, dims +16 * (m & 1)
              const int b = m;                       // block 2c + m within the four loaded
              const uint32_t s01 = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(__byte_perm(sw[0], sw[1], b | ((4 + b) << 4))));
              const uint32_t s23 = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(__byte_perm(sw[2], sw[3], b | ((4 + b) << 4))));
              // each token's byte converts to {even dim, odd dim}; byte permutes regroup the halves
              // into token pairs per dim
              uint32_t cc[4];
              dev::e2m1x8_to_f16x2x4(r[m], cc);
              const uint32_t c0 = cc[0], c1 = cc[1], c2 = cc[2], c3 = cc[3];
              const int nt = 4 * (2 * vq + (m >> 1)) + 2 * (m & 1);
              dev::mma_f16(o[nt], pa0, pa1, pa2, pa3, dev::hmul2_f16(__byte_perm(c0, c1, 0x5410), s01),
                           dev::hmul2_f16(__byte_perm(c2, c3, 0x5410), s23));
              dev::mma_f16(o[nt + 1], pa0, pa1, pa2, pa3, dev::hmul2_f16(__byte_perm(c0, c1, 0x7632), s01),
                           dev::hmul2_f16(__byte_perm(c2, c3, 0x7632), s23));
            }
          }
        } else if constexpr (RAW) {
          // V fragments straight from the page bytes: lanes 0..15 address the tile's 16 rows (token
          // rho(r) for row r) at a 16-dim block, lanes 16..31 at the next block; each lane receives
          // rows 4t4 .. 4t4+3 (P's k order above) of dims g8 and 8 + g8 of each block
          const int vt = tt0(kt) + rho(lane & 15);
#pragma unroll
          for (int vq = 0; vq < 8; ++vq) {
            uint32_t r[4];
            dev::ldsm_t8_x2(trb(kt) + raw_chunk_off(vt, half * 16 + 2 * vq + (lane >> 4)), r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dev::mma_f16(o[4 * vq + u], pa0, pa1, pa2, pa3, dev::e4m3x2_to_f16x2(static_cast<uint16_t>(r[u] & 0xFFFFu)),
                           dev::e4m3x2_to_f16x2(static_cast<uint16_t>(r[u] >> 16)));
          }
        } else {
#pragma unroll
        for (int vp = 0; vp < 16; ++vp) {
          uint32_t b0, b1, b2, b3;
          dev::ldsm_x4_t(a_kv + v_lane + ((t0 + kt * 16) * kRow + vp * 16) * 2, b0, b1, b2, b3);
          dev::mma_f16(o[2 * vp], pa0, pa1, pa2, pa3, b0, b1);
          dev::mma_f16(o[2 * vp + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
        }
      }
      }
      if constexpr (RAW) {
        // this warp is done with the iteration's buffers
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int u = 0; u < PPI; ++u)
            if (j + u < seg.num_pages) tc::mbar_arrive(a_bar + 8 * (NB + buf_u[u]));
        }
      } else {
        __syncthreads();  // s_kv and the exchange buffers are reused by the next page
      }
    }
    // raw-operand path: every warp is done with the segment's pages (the merge below reuses the raw
    // buffers) and no copy is in flight (the last pages were consumed)
    if constexpr (RAW) __syncthreads();
    if (!mma_warp) continue;

    // ---- epilogue: normalise; write the output directly or a split partial ----
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
      l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
    }
    if (TG > 1) {
      // merge the token groups of each head group by their maxima, in group order, through the
      // page tile and raw buffers (no page of this segment is read any more): pairs tg > 0 store
      // (O, m, l) in their fragment order, the tg = 0 pair of the same heads reads them back
      float* mrg = reinterpret_cast<float*>(s_kv);
      constexpr int kSlot = 32 * 128 + 32 * 4;            // one warp's O fragments, then m and l
      static_assert(NG * (TG - 1) * 2 * kSlot * 4 <= tile_bytes<KV, HC>() + NB * raw_bytes<KV>() + xbuf_bytes<KV, HC>(),
                    "merge slots fit in the page tile, raw buffers and exchange buffers");
      auto slot = [&](int g, int t, int hf) { return mrg + ((g * (TG - 1) + (t - 1)) * 2 + hf) * kSlot; };
      if (tg > 0) {
        float* d = slot(grp, tg, half);
#pragma unroll
        for (int u = 0; u < 128; ++u) d[u * 32 + lane] = o[u >> 2][u & 3];
        d[4096 + lane] = m_r[0]; d[4096 + 32 + lane] = m_r[1];
        d[4096 + 64 + lane] = l_r[0]; d[4096 + 96 + lane] = l_r[1];
      }
      dev::named_bar_sync(15, 64 * NPAIR);
      if (tg > 0) continue;
      float mt[TG][2], f[TG][2];
#pragma unroll
      for (int t = 0; t < TG; ++t)
#pragma unroll
        for (int r = 0; r < 2; ++r) mt[t][r] = t == 0 ? m_r[r] : slot(grp, t, half)[4096 + 32 * r + lane];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float mstar = mt[0][r];
#pragma unroll
        for (int t = 1; t < TG; ++t) mstar = fmaxf(mstar, mt[t][r]);
        float lsum = 0.0f;
#pragma unroll
        for (int t = 0; t < TG; ++t) {
          f[t][r] = mt[t][r] == -INFINITY ? 0.0f : dev::fast_exp2(mt[t][r] - mstar);
          lsum += (t == 0 ? l_r[r] : slot(grp, t, half)[4096 + 64 + 32 * r + lane]) * f[t][r];
        }
        m_r[r] = mstar;
        l_r[r] = lsum;
      }
#pragma unroll
      for (int u = 0; u < 128; ++u) {
        float v = o[u >> 2][u & 3] * f[0][(u & 3) >> 1];
#pragma unroll
        for (int t = 1; t < TG; ++t) v += slot(grp, t, half)[u * 32 + lane] * f[t][(u & 3) >> 1];
        o[u >> 2][u & 3] = v;
      }
    }
    const float inv[2] = {l_r[0] > 0.0f ? 1.0f / l_r[0] : 0.0f, l_r[1] > 0.0f ? 1.0f / l_r[1] : 0.0f};
    const float lse2[2] = {l_r[0] > 0.0f ? m_r[0] + __log2f(l_r[0]) : -INFINITY,
                           l_r[1] > 0.0f ? m_r[1] + __log2f(l_r[1]) : -INFINITY};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int head = h0 + grp * 16 + g8 + 8 * r;
      // output dim of element e (0..3) of a lane's four consecutive dims 4t4 + e: NVFP4 tiles hold
      // even / odd dims apart (o[4c + 2h + (e & 1)][2r + (e >> 1)] for dims 32c + 16h + 4t4 + e),
      // the other pools consecutive pairs (o[q][2r + (e & 1)] for dims 8q + 2t4 + e)
      if (seg.partial < 0) {
        uint16_t* dst = a.out + (static_cast<int64_t>(seg.req) * a.heads + head) * kDv + half * 256;
        const float sc = inv[r] * a.out_scale;
        if constexpr (RAW && KV == KV_NVFP4) {
#pragma unroll
          for (int q = 0; q < 16; ++q) {         // 16-dim groups: chunk q / 2, half q & 1
            const int nt = 4 * (q >> 1) + 2 * (q & 1);
            *reinterpret_cast<uint2*>(dst + 16 * q + 4 * t4) =
                make_uint2(dev::pack_bf16x2(o[nt][2 * r] * sc, o[nt + 1][2 * r] * sc),
                           dev::pack_bf16x2(o[nt][2 * r + 1] * sc, o[nt + 1][2 * r + 1] * sc));
          }
        } else {
#pragma unroll
          for (int nt = 0; nt < 32; ++nt)
            reinterpret_cast<uint32_t*>(dst)[(nt * 8 + 2 * t4) / 2] = dev::pack_bf16x2(o[nt][2 * r] * sc, o[nt][2 * r + 1] * sc);
        }
        if (half == 0 && t4 == 0 && a.lse) a.lse[static_cast<int64_t>(seg.req) * a.heads + head] = lse2[r] * 0.69314718055994531f;
      } else {
        float* dst = a.part_o + (static_cast<int64_t>(seg.partial) * a.heads + head) * kDv + half * 256;
        if constexpr (RAW && KV == KV_NVFP4) {
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int nt = 4 * (q >> 1) + 2 * (q & 1);
            *reinterpret_cast<float4*>(dst + 16 * q + 4 * t4) =
                make_float4(o[nt][2 * r] * inv[r], o[nt + 1][2 * r] * inv[r], o[nt][2 * r + 1] * inv[r], o[nt + 1][2 * r + 1] * inv[r]);
          }
        } else {
#pragma unroll
          for (int nt = 0; nt < 32; ++nt)
            reinterpret_cast<float2*>(dst)[(nt * 8 + 2 * t4) / 2] = make_float2(o[nt][2 * r] * inv[r], o[nt][2 * r + 1] * inv[r]);
        }
        if (half == 0 && t4 == 0) a.part_lse[static_cast<int64_t>(seg.partial) * a.heads + head] = lse2[r];
      }
    }
  }
}

// The pool as a 3-D tensor of bytes {row bytes, 64 tokens, pages} (576 per row and a page stride of
// 36,864 or 37,120 for the FP8 pools, 288 and 18,432 for NVFP4 codes) for the raw-operand path's TMA
// loads: box {144, 64, 1}, no swizzle, no interleave.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t encode_kv_map(const DecodeArgs& a, int64_t row_bytes, int64_t page_bytes, CUtensorMap* map) {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
      return cudaErrorNotSupported;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(kPage),
                              static_cast<cuuint64_t>(a.num_pages)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(page_bytes)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBoxDims), static_cast<cuuint32_t>(kPage), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(a.kv), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int KV, int HC, bool F8 = false>
cudaError_t launch_kv_hc(const DecodeArgs& a, cudaStream_t s) {
  constexpr int smem = smem_bytes<KV, HC>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<KV, HC, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  CUtensorMap map;
  std::memset(&map, 0, sizeof(map));
  if (raw_operands<KV, HC>() && a.num_pages > 0) {
    const cudaError_t e = KV == KV_NVFP4 ? encode_kv_map(a, kPacked, kPage * kPacked, &map)
                        : encode_kv_map(a, kLatent, KV == KV_FP8PT ? kPtPageBytes : kPage * kLatent, &map);
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = static_cast<unsigned>(a.num_workers * a.ctas_per_worker);
  decode_mma_kernel<KV, HC, F8><<<grid, kNT, smem, s>>>(a, map);
  return cudaGetLastError();
}

template <int KV>
cudaError_t launch_kv(const DecodeArgs& a, cudaStream_t s) {
  if constexpr (KV == KV_FP8 || KV == KV_FP8PT) {
    if (a.fp8_qk) {
      switch (mma_fp8_heads_per_cta(a.heads)) {
        case 16: return launch_kv_hc<KV, 16, true>(a, s);
        case 32: return launch_kv_hc<KV, 32, true>(a, s);
        default: return cudaErrorInvalidValue;
      }
    }
  }
  if (a.fp8_qk) return cudaErrorInvalidValue;
  switch (mma_heads_per_cta(a.heads)) {
    case 16: return launch_kv_hc<KV, 16>(a, s);
    case 32: return launch_kv_hc<KV, 32>(a, s);
    case 48: return launch_kv_hc<KV, 48>(a, s);
    case 64: return launch_kv_hc<KV, 64>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int mma_fp8_heads_per_cta(int heads) {
  if (heads < 16 || heads > 128 || heads % 16) return 0;
  return heads % 32 == 0 ? 32 : 16;
}

int mma_heads_per_cta(int heads) {
  if (heads < 16 || heads > 128 || heads % 16) return 0;
  for (int hc : {64, 48, 32, 16})
    if (heads % hc == 0) return hc;
  return 0;
}

cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t s) {
  if (a.num_segments == 0) return cudaSuccess;
  switch (a.kv_dtype) {
    case KV_FP8: return launch_kv<KV_FP8>(a, s);
    case KV_NVFP4: return launch_kv<KV_NVFP4>(a, s);
    case KV_BF16: return launch_kv<KV_BF16>(a, s);
    case KV_FP8PT: return launch_kv<KV_FP8PT>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qkvp
