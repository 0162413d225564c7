// Split-KV paged MLA decode on the 5th-generation tensor cores for 16 to 64 query heads, with the
// page's tokens as the rows of every product (token-major).
//
// The attention is the one of the pages' plan()/run() call ("The Smoking Gun", section "What
// Message 1408 Actually Reveals"): per request and head, softmax(sm_scale * q . k) v over the
// request's tokens, K = the 576-wide latent, V = its first 512 dims, read from quantized pages and
// dequantized on chip ("SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "SGLang implementation",
// item 3). Products take FP16 operands with FP32 accumulation, the same arithmetic as the other two
// kernel families (exact K/V, Q converted exactly or rescaled by a power of two, 11-bit P).
//
// Orientation. A heads-major product (M = heads) pads 16-64 heads to 128 rows, and its N = 32 or 64
// token columns leave the tensor cores waiting on operand traffic. Here the 64 tokens of a page are
// the M dimension and the HN heads (16, 32 or 64; 48 heads ride in 64) the N dimension:
//   S^T [64 tokens x HN]   = K_page [64 x 576] . Q^T          M = 64,  K = 576: 36 MMAs
//   O^T [512 dims x HN]   += V_page^T [512 x 64] . P [64 x HN]  4 M-tiles of 128 dims, K = 64: 16 MMAs
// The page's dequantized FP16 tile (token rows of 64-dim atoms, 128-byte swizzle) is the K-major A
// operand of the first product and, unchanged, the MN-major A operand of the second; Q (rows =
// heads) and P (rows = tokens) are the B operands. The accumulator of an M = 64 product sits in TMEM
// lanes 32 (r / 16) + r % 16 (measured), so softmax warp w finds tokens 16w .. 16w + 15 in lanes 0 .. 15
// of its quarter; the 16x256b load shape spreads them over all 32 threads (two tokens and a quarter of
// the heads each). O^T puts one output dim per TMEM lane.
//
// Per CTA (512 threads, one CTA per SM, persistent over its worker's segments):
//   warps 0-3 (softmax): at a new request convert its Q rows to FP16 (rows holding |q| >= 2^15 are
//     scaled by a power of two folded into the head's logit scale); per page read the thread's logits,
//     update the per-head running maxima lazily (only when a logit passes the maximum by more than 2^8,
//     base 2; the decision is taken jointly by the four warps), rescale O^T and the row sums then,
//     write the thread's words of P (up to 32 heads computed against the current maxima before the
//     joint decision and kept unless it renews them; from 48 heads after it); at a segment's end sum
//     the row sums over the 64 tokens and write O / l (or the normalised partial and its
//     log2-sum-exp) from TMEM, one output dim per lane.
//   warps 4-11 (dequant): raw page bytes from global memory (32-byte loads, the next page's in flight
//     while the current one is written) into one of two FP16 tile slots; rows past the page's valid
//     tokens are written as zeros.
//   two Q.K^T warps: one thread each issues half of every page's 36 MMAs (latent dims 0-287 /
//     288-575) into its own accumulator; the softmax adds the two in a fixed order. A thread waits
//     ~50-70 cycles after each tcgen05.mma it issues, so two halves in flight halve the page's latency.
//   two P.V warps: one thread each issues the MMAs of two of the four M-tiles of every page into O^T.
// TMEM: logit buffers [page parity][K half] at [0, 4 HN), O^T [4 HN, 8 HN).
// Every wait is bounded; a timeout sets bits in the status word and the CTA drains and exits.
#include <cstdint>

#include "qkvp_device.cuh"
#include "qkvp_internal.h"
#include "decode_common.cuh"
#include "tc_ptx.cuh"

namespace qkvp {
namespace {

using kern::Cursor;
using kern::Sync;
using kern::ldg_nc32;
using kern::page_ok;
using kern::sts128;

constexpr int kCols = kLatent / 64;             // 64-dim atom columns of a tile
constexpr uint32_t kColBytes = kPage * 128;     // 64 token rows x 64 FP16 dims
constexpr uint32_t kTileBytes = kCols * kColBytes;
constexpr int kStatusBase = 16;                 // status bits of this kernel's timeouts: 16 << role

enum : uint32_t {
  B_T_FULL = 0, B_T_EMPTY = 2, B_S_FULL = 4, B_S_FREE = 6, B_P_FULL = 8, B_P_FREE = 10, B_O_FREE = 12,
  B_SYNC = 13, B_FINAL = 14, NUM_BARS = 15
};

template <int HN>
struct Cfg {
  static constexpr uint32_t kQCol = HN * 128;           // Q atom column: HN rows x 64 dims
  static constexpr uint32_t kQBytes = kCols * kQCol;
  static constexpr uint32_t kPRow = HN * 2;             // P row of one token: HN FP16
  static constexpr uint32_t kPBytes = kPage * kPRow;
  static constexpr int kPBufs = HN == 64 ? 1 : 2;       // 64 heads: shared memory holds one P buffer
  static constexpr bool kSpecP = HN <= 32;              // P before the maxima agreement (see role_softmax)
  static constexpr uint32_t kPSwizzle = HN == 16 ? tc::kSwizzle32 : HN == 32 ? tc::kSwizzle64 : tc::kSwizzle128;
  static constexpr uint32_t OFF_T = 0;
  static constexpr uint32_t OFF_Q = OFF_T + 2 * kTileBytes;
  static constexpr uint32_t OFF_P = OFF_Q + kQBytes;
  static constexpr uint32_t OFF_MRUN = OFF_P + kPBufs * kPBytes;   // HN floats: running maxima (scaled, base 2)
  static constexpr uint32_t OFF_QSC = OFF_MRUN + 4 * HN;           // HN floats: logit scale of each head
  static constexpr uint32_t OFF_ALPHA = OFF_QSC + 4 * HN;          // HN floats: rescale factors, row sums
  static constexpr uint32_t OFF_RED = OFF_ALPHA + 4 * HN;          // [4 warps][HN] floats
  static constexpr uint32_t OFF_FLAG = OFF_RED + 16 * HN;          // [2][4] ints
  static constexpr uint32_t OFF_BAR = OFF_FLAG + 32;
  static constexpr uint32_t OFF_TSLOT = OFF_BAR + 8 * NUM_BARS;
  static constexpr uint32_t OFF_ABORT = OFF_TSLOT + 4;
  static constexpr uint32_t OFF_QVER = OFF_ABORT + 4;
  static constexpr uint32_t kSmemUsed = OFF_QVER + 8;
  static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;      // slack to align the base to 1024 bytes
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0, "swizzle atoms");
  // logit buffers [page parity][K half], then O^T
  static constexpr uint32_t TM_S = 0, TM_O = 4 * HN;
  static_assert(8 * HN <= 512, "TMEM columns");
  // Warps: 0-3 softmax, 4-11 dequant, then one P.V, two Q.K^T and a second P.V issuing warp; 16 warps
  // leave 128 registers a thread.
  static constexpr int kPvThreads = 2;
  static constexpr int kDqWarps = 8;
  static constexpr int kDQ = 32 * kDqWarps;
  static constexpr int kPvWarp0 = 4 + kDqWarps, kQkWarp0 = kPvWarp0 + 1, kPvWarp1 = kPvWarp0 + 3;
  static constexpr int kThreads = 32 * (4 + kDqWarps + 2 + kPvThreads);
  static constexpr int kChunk = HN < 32 ? HN : 32;      // logit columns per TMEM load
};

__host__ __device__ constexpr uint32_t p_offset(int hn, uint32_t row, uint32_t chunk) {
  return hn == 16 ? tc::sw32_offset(row, chunk) : hn == 32 ? tc::sw64_offset(row, chunk) : tc::sw128_offset(row, chunk);
}

// ---- dequantization of a page into an FP16 tile slot -------------------------------------------------
// Tile: 9 atom columns (latent dims 64c .. 64c + 63), each 64 token rows of 128 bytes, 128-byte swizzle.
template <int KV, int NT> struct Dequant;

template <int NT> struct Dequant<KV_FP8, NT> {
  // 32 dims (one 32-byte load) per item; item q: atom column q / 128, token (q % 128) / 2, half q % 2.
  // A warp's 32 items are 16 tokens x both halves of one column: every 8 lanes of each 16-byte row
  // store land in 8 distinct bank groups.
  static constexpr int kItems = kPage * kLatent / 32;
  static constexpr int kIters = (kItems + NT - 1) / NT;
  struct Raw { uint32_t v[kIters][8]; };
  __device__ static const uint8_t* page_ptr(const DecodeArgs& a, int64_t page) { return a.kv + page * (kPage * kLatent); }
  __device__ static void load(Raw& r, const uint8_t* base, int valid, int t) {
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + NT * i;
      const int tok = (q & 127) >> 1;
      if (q < kItems && tok < valid) ldg_nc32(base + tok * kLatent + (q >> 7) * 64 + (q & 1) * 32, r.v[i]);
    }
  }
  __device__ static void store(const Raw& r, int valid, int t, uint32_t tile) {
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + NT * i;
      if (q >= kItems) continue;
      const int tok = (q & 127) >> 1, half = q & 1;
      uint32_t o[16];
#pragma unroll
      for (int b = 0; b < 16; ++b)
        o[b] = tok < valid ? dev::e4m3x2_to_f16x2(static_cast<uint16_t>(r.v[i][b >> 1] >> (16 * (b & 1)))) : 0u;
      const uint32_t at = tile + (q >> 7) * kColBytes;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        sts128(at + tc::sw128_offset(tok, 4 * half + u), make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]));
    }
  }
};

template <int NT> struct Dequant<KV_FP8PT, NT> : Dequant<KV_FP8, NT> {
  // the codes of a per-token-scaled page (its token scales follow the 64 rows and are applied by
  // the softmax threads, one per token, in FP32)
  __device__ static const uint8_t* page_ptr(const DecodeArgs& a, int64_t page) { return a.kv + page * kPtPageBytes; }
};

template <int NT> struct Dequant<KV_NVFP4, NT> {
  // 64 dims per item: 32 packed bytes (one 32-byte load) and the four E4M3 block scales (one 4-byte
  // load); item q: atom column q / 64, token q % 64, so a warp's 32 items are 32 rows of one column.
  static constexpr int kItems = kPage * kCols;
  static constexpr int kIters = (kItems + NT - 1) / NT;
  struct Raw { uint32_t v[kIters][8]; uint32_t s[kIters]; };
  struct Ptr { const uint8_t* data; const uint8_t* scales; };
  __device__ static Ptr page_ptr(const DecodeArgs& a, int64_t page) {
    return Ptr{a.kv + page * (kPage * kPacked), a.kv_scale + page * (kPage * kScales)};
  }
  __device__ static void load(Raw& r, const Ptr& p, int valid, int t) {
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + NT * i;
      const int tok = q & 63, col = q >> 6;
      if (q < kItems && tok < valid) {
        ldg_nc32(p.data + tok * kPacked + col * 32, r.v[i]);
        r.s[i] = __ldg(reinterpret_cast<const uint32_t*>(p.scales + tok * kScales + col * 4));
      }
    }
  }
  __device__ static void store(const Raw& r, int valid, int t, uint32_t tile) {
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + NT * i;
      if (q >= kItems) continue;
      const int tok = q & 63, col = q >> 6;
      uint32_t o[32];
      if (tok < valid) {
        uint32_t h[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t sk = (r.s[i] >> (8 * k)) & 0xFFu;
          h[k] = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(sk | (sk << 8)));
        }
#pragma unroll
        for (int wv = 0; wv < 8; ++wv) {
          uint32_t c4[4];
          dev::e2m1x8_to_f16x2x4(r.v[i][wv], c4);
#pragma unroll
          for (int k = 0; k < 4; ++k) o[4 * wv + k] = dev::hmul2_f16(c4[k], h[wv >> 1]);
        }
      } else {
#pragma unroll
        for (int b = 0; b < 32; ++b) o[b] = 0u;
      }
      const uint32_t at = tile + col * kColBytes;
#pragma unroll
      for (int u = 0; u < 8; ++u) sts128(at + tc::sw128_offset(tok, u), make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]));
    }
  }
};

// L2 prefetch of a whole FP8 page (the raw loads of a page run two pages behind the prefetch).
template <int KV>
__device__ __forceinline__ void prefetch_page(const DecodeArgs& a, int64_t page) {
  if constexpr (KV == KV_FP8) tc::bulk_prefetch_l2(a.kv + page * (kPage * kLatent), kPage * kLatent);
}

template <int KV, int NT>
__device__ void role_dequant(const DecodeArgs& a, const Sync& sy, int seg_b, int seg_e, int t, uint32_t tiles) {
  using D = Dequant<KV, NT>;
  Cursor cur;
  cur.begin(a, seg_b, seg_e);
  if (cur.done()) return;
  // One register set: a page's raw loads are issued right after the previous page is written, so they
  // land while the thread waits for the next tile slot (copying a second set would stall on them).
  typename D::Raw rw;
  Cursor nx = cur;
  nx.next(a);
  int64_t npg = nx.done() ? 0 : nx.page(a);
  const int64_t pg0 = cur.page(a);
  int valid = page_ok(a, pg0) ? cur.valid() : 0;
  if (valid > 0) D::load(rw, D::page_ptr(a, pg0), valid, t);
  // one thread keeps the pages four ahead flowing into L2
  constexpr int kAhead = KV == KV_FP8 ? 4 : 0;
  Cursor pf = cur;
  int64_t pf_pg = -1;                 // read an iteration before its prefetch is issued
  if (kAhead > 0 && t == 0) {
    for (int i = 0; i < kAhead && !pf.done(); ++i) {
      if (i >= 2 && page_ok(a, pf.page(a))) prefetch_page<KV>(a, pf.page(a));
      pf.next(a);
    }
    if (!pf.done()) pf_pg = pf.page(a);
  }
  for (int g = 0; !cur.done(); ++g) {
    if (kAhead > 0 && t == 0 && !pf.done()) {
      if (page_ok(a, pf_pg)) prefetch_page<KV>(a, pf_pg);
      pf.next(a);
      pf_pg = pf.done() ? -1 : pf.page(a);
    }
    Cursor nn = nx;
    if (!nn.done()) nn.next(a);
    const int64_t nnpg = nn.done() ? 0 : nn.page(a);
    const int nvalid = nx.done() ? 0 : (page_ok(a, npg) ? nx.valid() : 0);
    const int slot = g & 1;
    // slot last held page g - 2: its P.V completion frees it
    if (g >= 2 && !sy.wait(B_T_EMPTY + slot, ((g >> 1) - 1) & 1, false, kStatusBase << 0)) return;
    D::store(rw, valid, t, tiles + slot * kTileBytes);
    tc::fence_proxy_async_smem();
    tc::mbar_arrive(sy.bar(B_T_FULL + slot));
    if (nvalid > 0) D::load(rw, D::page_ptr(a, npg), nvalid, t);
    cur = nx;
    nx = nn;
    npg = nnpg;
    valid = nvalid;
  }
}

// One thread issues half of S^T = K_page . Q^T (18 MMAs, M 64 x N HN x K 16, latent dims 288 half ..
// 288 half + 287) for every page, into its own accumulator of the page parity's logit buffer.
template <int HN>
__device__ void role_qk(const DecodeArgs& a, const Sync& sy, int seg_b, int seg_e, int half, uint32_t tbase,
                        uint32_t tiles, uint32_t qs, uint32_t qver) {
  using C = Cfg<HN>;
  Cursor cq;
  cq.begin(a, seg_b, seg_e);
  constexpr uint32_t kIdesc = tc::idesc_f16(64, HN, 0, 0);
  const tc::Desc2 td = tc::split_desc(tc::smem_desc(tiles, 16, 1024, tc::kSwizzle128));
  const tc::Desc2 qd = tc::split_desc(tc::smem_desc(qs, 16, 1024, tc::kSwizzle128));
  // requests are counted in page order, as the softmax loads their Q
  int qcount = 0, q_req = -1, q_waited = -1;
  for (int g = 0; !cq.done(); ++g, cq.next(a)) {
    if (cq.j == 0 && cq.seg.req != q_req) { q_req = cq.seg.req; ++qcount; }
    const int slot = g & 1;
    if (!sy.wait(B_T_FULL + slot, (g >> 1) & 1, false, kStatusBase << 1)) break;
    // logit buffer `slot` was last read out for page g - 2
    if (g >= 2 && !sy.wait(B_S_FREE + slot, ((g >> 1) - 1) & 1, false, kStatusBase << 1)) break;
    if (q_waited != qcount) {
      if (!kern::wait_counter(sy, qver, static_cast<uint32_t>(qcount), kStatusBase << 5)) break;
      q_waited = qcount;
    }
    tc::tc_fence_after();
    const uint32_t ts = tbase + C::TM_S + (2 * slot + half) * HN;
    const uint32_t tile = slot * kTileBytes;
#pragma unroll
    for (int k = 0; k < 18; ++k) {
      const int ks = 18 * half + k;
      const uint64_t ad = td.at(tile + (ks >> 2) * kColBytes + 32 * (ks & 3));
      const uint64_t bd = qd.at((ks >> 2) * C::kQCol + 32 * (ks & 3));
      if (k == 0) tc::mma_ss_k<false>(ts, ad, bd, kIdesc);
      else tc::mma_ss_k<true>(ts, ad, bd, kIdesc);
    }
    tc::mma_commit(sy.bar(B_S_FULL + slot));
  }
  tc::mma_commit(sy.bar(B_FINAL));
}

// One thread issues O^T += V_page^T . P for its M-tiles of 128 dims (4 / kPvThreads of them, 4 K-steps of
// 16 tokens each) for every page.
template <int HN>
__device__ void role_pv(const DecodeArgs& a, const Sync& sy, int seg_b, int seg_e, int part, uint32_t tbase,
                        uint32_t tiles, uint32_t pbuf) {
  using C = Cfg<HN>;
  Cursor cp;
  cp.begin(a, seg_b, seg_e);
  constexpr uint32_t kIdesc = tc::idesc_f16(128, HN, 1, 1);
  // MN-major V^T: 64 dims per 128-byte row, the next 64 dims one atom column further, 8-token groups 1 KB apart
  const uint64_t v0 = tc::smem_desc(tiles, kColBytes, 1024, tc::kSwizzle128);
  // MN-major P: HN heads per row, 8-token groups 8 rows apart
  const uint64_t p0 = tc::smem_desc(pbuf, kColBytes, 8 * C::kPRow, C::kPSwizzle);
  int si = 0;                                   // segments started
  for (int g = 0; !cp.done(); ++g) {
    const int pb = g % C::kPBufs;
    if (!sy.wait(B_P_FULL + pb, (g / C::kPBufs) & 1, false, kStatusBase << 2)) break;
    // already complete (Q.K^T of this page waited for it); the tile cannot be refilled before this P.V
    if (!sy.wait(B_T_FULL + (g & 1), (g >> 1) & 1, false, kStatusBase << 2)) break;
    const bool first = cp.j == 0;
    if (first) {
      // O^T of the previous segment has been read out
      if (si > 0 && !sy.wait(B_O_FREE, (si - 1) & 1, false, kStatusBase << 2)) break;
      ++si;
    }
    tc::tc_fence_after();
    const uint64_t vd = tc::desc_add(v0, (g & 1) * kTileBytes);
    const uint64_t pd = tc::desc_add(p0, pb * C::kPBytes);
    constexpr int kTiles = 4 / C::kPvThreads;
#pragma unroll
    for (int m = 0; m < kTiles; ++m) {
      const int mt = kTiles * part + m;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t av = tc::desc_add(vd, mt * 2 * kColBytes + kk * 2048);
        const uint64_t bp = tc::desc_add(pd, kk * 16 * C::kPRow);
        const uint32_t d = tbase + C::TM_O + mt * HN;
        if (first && kk == 0) tc::mma_ss_k<false>(d, av, bp, kIdesc);
        else tc::mma_ss_k<true>(d, av, bp, kIdesc);
      }
    }
    tc::mma_commit(sy.bar(B_T_EMPTY + (g & 1)));
    tc::mma_commit(sy.bar(B_P_FREE + pb));
    cp.next(a);
  }
  tc::mma_commit(sy.bar(B_FINAL));
}

// 16 or 32 columns of the warp's 32 TMEM lanes into / from registers (the arrays stay in registers:
// nothing takes their address).
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 16) tc::tmem_ld16(taddr, r);
  else tc::tmem_ld32(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 16) tc::tmem_st16(taddr, r);
  else tc::tmem_st32(taddr, r);
}

// 16 TMEM lanes x 8N columns, 16x256b shape: thread t of the warp gets lanes t / 4 and t / 4 + 8 of its
// quarter and, of every 8-column group g, columns 8g + 2 (t % 4) and + 1: r[4g], r[4g + 1] from the
// first lane, r[4g + 2], r[4g + 3] from the second (measured on the GPU).
template <int N>
__device__ __forceinline__ void tmem_ld_16x256(uint32_t taddr, uint32_t (&r)[4 * N]) {
  static_assert(N == 2 || N == 4 || N == 8, "2, 4 or 8 column groups");
  if constexpr (N == 2) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
  } else if constexpr (N == 4) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x4.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
  } else {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x8.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
                   "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
  }
}

// Barrier of the four softmax warps: lane 0 of each warp arrives, every thread waits (bounded). All
// 128 threads pass the same sequence of these, so each phase is waited for in turn.
struct SoftmaxSync {
  uint32_t bar;
  int phase;
  __device__ bool operator()(const Sync& sy) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) tc::mbar_arrive(bar);
    const bool ok = sy.wait(B_SYNC, phase & 1, false, kStatusBase << 3);
    ++phase;
    return __all_sync(0xffffffffu, ok);
  }
};

// Q rows of request `req` in FP16 (K-major atom columns, rows = heads; rows >= heads zero) and the
// logit scale of each head. BF16 -> FP16 is exact for magnitudes in [2^-14, 2^15); a row holding
// 2^15 or more is scaled by 2^-sh (its largest |q| then lies in [2^14, 2^15)) and 2^sh joins the
// head's logit scale. 128 / HN consecutive threads share a row.
template <int HN>
__device__ void load_q(const DecodeArgs& a, int req, int tid, uint32_t qs, float* qsc) {
  constexpr int kTpr = 128 / HN, kChunks = kLatent / 8, kCpt = kChunks / kTpr;
  constexpr int kBatch = 9;                          // 16-byte loads in flight per thread
  static_assert(kCpt % kBatch == 0, "batches of chunks");
  const int h = tid / kTpr, part = tid % kTpr;
  const bool live = h < a.heads;
  const uint4* qrow = reinterpret_cast<const uint4*>(a.q) + (static_cast<int64_t>(req) * a.heads + (live ? h : 0)) * (kLatent / 8);
  auto big = [](uint32_t w) { return (w & 0x7FFFu) >= 0x4700u || ((w >> 16) & 0x7FFFu) >= 0x4700u; };
  // the row unscaled, in batches of loads in flight; a value of 2^15 or more (or inf / NaN) makes the
  // row convert again below with a power-of-two scale
  bool hot = false;
#pragma unroll 1
  for (int i0 = 0; i0 < kCpt; i0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) v[i] = live ? __ldg(qrow + part + kTpr * (i0 + i)) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int chunk = part + kTpr * (i0 + i);         // 8 dims
      hot |= big(v[i].x) || big(v[i].y) || big(v[i].z) || big(v[i].w);
      sts128(qs + (chunk >> 3) * Cfg<HN>::kQCol + tc::sw128_offset(h, chunk & 7),
             make_uint4(dev::bf16x2_to_f16x2(v[i].x), dev::bf16x2_to_f16x2(v[i].y), dev::bf16x2_to_f16x2(v[i].z),
                        dev::bf16x2_to_f16x2(v[i].w)));
    }
  }
  // the kTpr threads of a row agree (aligned groups of consecutive lanes)
#pragma unroll
  for (int off = 1; off < kTpr; off <<= 1) hot |= __shfl_xor_sync(0xffffffffu, hot ? 1 : 0, off) != 0;
  float sc = a.scale_log2;
  if (__any_sync(0xffffffffu, hot) && hot) {
    uint32_t mx = 0;
#pragma unroll 1
    for (int i = 0; i < kCpt; ++i) {
      const uint4 v = __ldg(qrow + part + kTpr * i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
    }
#pragma unroll
    for (int off = 1; off < kTpr; off <<= 1) mx = max(mx, __shfl_xor_sync(__activemask(), mx, off));
    if (mx < 0x7F80u) {                               // inf / NaN rows stay unscaled
      const int sh = max(-100, min(113, static_cast<int>(mx >> 7) - 127 - 14));
      const float down = __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
      sc = a.scale_log2 * __uint_as_float(static_cast<uint32_t>(127 + sh) << 23);
#pragma unroll 1
      for (int i = 0; i < kCpt; ++i) {
        const int chunk = part + kTpr * i;
        const uint4 v = __ldg(qrow + chunk);
        sts128(qs + (chunk >> 3) * Cfg<HN>::kQCol + tc::sw128_offset(h, chunk & 7),
               make_uint4(dev::bf16x2_to_f16x2(v.x, down), dev::bf16x2_to_f16x2(v.y, down),
                          dev::bf16x2_to_f16x2(v.z, down), dev::bf16x2_to_f16x2(v.w, down)));
      }
    }
  }
  if (part == 0) qsc[h] = sc;
}

// Scaled logits y = (S_lo + S_hi) * token scale * head scale of this thread's two tokens and HN / 4
// heads (16x256b layout: y[4g + k] token 0, y[4g + 2 + k] token 1, head 8g + hq + k), read from TMEM
// (-inf for rows that are not valid tokens). The softmax reads a buffer again rather than holding it
// in registers: it cannot be refilled before the page's P.V has freed the tile anyway.
template <int HN>
__device__ __forceinline__ void logits(uint32_t tl, int s, int hq, bool live0, bool live1, float sig0, float sig1,
                                       const float* qsc, float (&y)[HN / 2]) {
  uint32_t ra[HN / 2], rb[HN / 2];
  tmem_ld_16x256<HN / 8>(tl + Cfg<HN>::TM_S + (2 * s) * HN, ra);
  tmem_ld_16x256<HN / 8>(tl + Cfg<HN>::TM_S + (2 * s + 1) * HN, rb);
  tc::tmem_wait_ld();
#pragma unroll
  for (int g = 0; g < HN / 8; ++g) {
    const float2 q2 = *reinterpret_cast<const float2*>(qsc + 8 * g + hq);
    y[4 * g] = live0 ? (__uint_as_float(ra[4 * g]) + __uint_as_float(rb[4 * g])) * sig0 * q2.x : -INFINITY;
    y[4 * g + 1] = live0 ? (__uint_as_float(ra[4 * g + 1]) + __uint_as_float(rb[4 * g + 1])) * sig0 * q2.y : -INFINITY;
    y[4 * g + 2] = live1 ? (__uint_as_float(ra[4 * g + 2]) + __uint_as_float(rb[4 * g + 2])) * sig1 * q2.x : -INFINITY;
    y[4 * g + 3] = live1 ? (__uint_as_float(ra[4 * g + 3]) + __uint_as_float(rb[4 * g + 3])) * sig1 * q2.y : -INFINITY;
  }
}

// Per head of this thread, the reduction (max or sum) of v over the warp's 16 tokens: the 8 lane groups
// with the same lane % 4 hold the same heads; lanes 0-3 then write the warp's values to red.
template <int HN, bool kMax>
__device__ __forceinline__ void warp_reduce_heads(float (&v)[HN / 4], float* red_w, int lane) {
#pragma unroll
  for (int off = 4; off <= 16; off <<= 1)
#pragma unroll
    for (int i = 0; i < HN / 4; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], off);
      v[i] = kMax ? fmaxf(v[i], o) : v[i] + o;
    }
  if (lane < 4) {
#pragma unroll
    for (int g = 0; g < HN / 8; ++g)
      *reinterpret_cast<float2*>(red_w + 8 * g + 2 * lane) = make_float2(v[2 * g], v[2 * g + 1]);
  }
}

template <int KV, int HN>
__device__ void role_softmax(const DecodeArgs& a, const Sync& sy, int seg_b, int seg_e, int tid, uint32_t tbase,
                             uint32_t base, uint8_t* sbase) {
  using C = Cfg<HN>;
  const int w = tid >> 5, lane = tid & 31;
  // this thread's tokens (rows of the warp's 16) and heads (2 of every 8-column group)
  const int tok0 = 16 * w + (lane >> 2), tok1 = tok0 + 8, hq = 2 * (lane & 3);
  const uint32_t tl = tbase + (static_cast<uint32_t>(32 * w) << 16);
  float* m_run = reinterpret_cast<float*>(sbase + C::OFF_MRUN);
  float* qsc = reinterpret_cast<float*>(sbase + C::OFF_QSC);
  float* alpha = reinterpret_cast<float*>(sbase + C::OFF_ALPHA);
  float* red = reinterpret_cast<float*>(sbase + C::OFF_RED);
  volatile int* flags = reinterpret_cast<volatile int*>(sbase + C::OFF_FLAG);
  const uint32_t qs = base + C::OFF_Q, pbuf = base + C::OFF_P, qver = base + C::OFF_QVER;
  SoftmaxSync ssync{sy.bar(B_SYNC), 0};
  auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
    const bool ok = sy.wait(bar, parity, false, kStatusBase << 4);
    return __all_sync(0xffffffffu, ok);
  };
  float lp[HN / 4];                                // this thread's two tokens' share of its heads' row sums
  Cursor cur;
  cur.begin(a, seg_b, seg_e);
  int cur_req = -1, nq = 0;
  // the page index (and a per-token-scaled page's token scales) is read one page ahead
  auto page_info = [&](const Cursor& c, int& valid, float& s0, float& s1) {
    const int64_t pg = c.page(a);
    valid = page_ok(a, pg) ? c.valid() : 0;
    s0 = s1 = 1.0f;
    if (KV == KV_FP8PT) {
      const float* sp = reinterpret_cast<const float*>(a.kv + pg * kPtPageBytes + kPtScaleOff);
      if (tok0 < valid) s0 = __ldg(sp + tok0);
      if (tok1 < valid) s1 = __ldg(sp + tok1);
    }
  };
  int valid_n = 0;
  float sig0_n = 1.0f, sig1_n = 1.0f;
  if (!cur.done()) page_info(cur, valid_n, sig0_n, sig1_n);
  for (int g = 0; !cur.done(); ++g) {
    const Segment seg = cur.seg;
    if (cur.j == 0) {
      // segment start; at a new request also its Q (Q.K^T of every earlier page has completed: their
      // logits were read, so Q may be replaced)
      const bool new_q = seg.req != cur_req;
      if (new_q) {
        load_q<HN>(a, seg.req, tid, qs, qsc);
        tc::fence_proxy_async_smem();
        cur_req = seg.req;
      }
      if (tid < HN) m_run[tid] = -INFINITY;
#pragma unroll
      for (int i = 0; i < HN / 4; ++i) lp[i] = 0.0f;
      if (!ssync(sy)) return;
      if (new_q) {
        ++nq;   // the Q.K^T threads count requests the same way
        if (tid == 0) tc::st_release_u32(qver, static_cast<uint32_t>(nq));
      }
    }
    const int valid = valid_n;
    const float sig0 = sig0_n, sig1 = sig1_n;
    const bool live0 = tok0 < valid, live1 = tok1 < valid;
    {
      Cursor nx = cur;
      nx.next(a);
      if (!nx.done()) page_info(nx, valid_n, sig0_n, sig1_n);
    }
    const int s = g & 1;
    if (!wait(B_S_FULL + s, (g >> 1) & 1)) return;
    tc::tc_fence_after();
    const int pb = g % C::kPBufs;
    const uint32_t prow = pbuf + pb * C::kPBytes;
    // the four warps agree whether any logit passes its head's running maximum by more than 2^8
    auto agree = [&](bool flag) -> int {
      const bool wflag = __any_sync(0xffffffffu, flag);
      if (lane == 0) flags[(ssync.phase & 1) * 4 + w] = wflag ? 1 : 0;
      if (!ssync(sy)) return -1;
      const int fp = ((ssync.phase - 1) & 1) * 4;
      return (flags[fp] | flags[fp + 1] | flags[fp + 2] | flags[fp + 3]) ? 1 : 0;
    };
    // the page's maximum of each head over its 64 tokens, the renewed maxima (and, in red, the ones
    // they replace), and O^T's head columns rescaled
    auto renew_maxima = [&]() -> bool {
      {
        float y[HN / 2], mx[HN / 4];
        logits<HN>(tl, s, hq, live0, live1, sig0, sig1, qsc, y);
#pragma unroll
        for (int gg = 0; gg < HN / 8; ++gg) {
          mx[2 * gg] = fmaxf(y[4 * gg], y[4 * gg + 2]);
          mx[2 * gg + 1] = fmaxf(y[4 * gg + 1], y[4 * gg + 3]);
        }
        warp_reduce_heads<HN, true>(mx, red + w * HN, lane);
      }
      if (!ssync(sy)) return false;
      if (tid < HN) {
        const float pm = fmaxf(fmaxf(red[tid], red[HN + tid]), fmaxf(red[2 * HN + tid], red[3 * HN + tid]));
        const float mo = m_run[tid];
        const bool renew = pm > mo + 8.0f;
        const float mn = renew ? pm : mo;
        alpha[tid] = renew ? dev::fast_exp2(mo - mn) : 1.0f;   // 0 when mo is -inf
        m_run[tid] = mn;
        if (C::kSpecP) red[tid] = mo;
      }
      if (!ssync(sy)) return false;
      if (cur.j > 0) {
        // O^T holds this segment's earlier pages: rescale its head columns once PV(g - 1) has completed
        const int pq = (g - 1) % C::kPBufs;
        if (!wait(B_P_FREE + pq, ((g - 1) / C::kPBufs) & 1)) return false;
        tc::tc_fence_after();
        constexpr int CH = C::kChunk;
#pragma unroll 1
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll 1
          for (int c0 = 0; c0 < HN; c0 += CH) {
            uint32_t o[CH];
            tmem_ld_cols<CH>(tl + C::TM_O + mt * HN + c0, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < CH; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[c0 + h]);
            tmem_st_cols<CH>(tl + C::TM_O + mt * HN + c0, o);
          }
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
      }
      return true;
    };
    // P buffer pb was last read by PV(g - kPBufs)
    const bool pfree_wait = g >= C::kPBufs;
    const uint32_t pfree_par = ((g / C::kPBufs) - 1) & 1;
    if constexpr (C::kSpecP) {
      // ---- up to 32 heads, P = 2^(y - m) at once against the current maxima, FP16 (per-token-scaled
      // pages: times the token's scale), one 4-byte word (two heads) per token and 8-head chunk,
      // stored once the buffer is free. A logit that passes its maximum by more than 2^8 keeps its p
      // out of the row sum and has the maxima renewed and P taken again. ----
      bool flag = false;
      uint32_t pw[HN / 4];
      {
        float y[HN / 2];
        logits<HN>(tl, s, hq, live0, live1, sig0, sig1, qsc, y);
#pragma unroll
        for (int gg = 0; gg < HN / 8; ++gg) {
          const float2 m2 = *reinterpret_cast<const float2*>(m_run + 8 * gg + hq);
          const float mx = m2.x == -INFINITY ? 0.0f : m2.x, my = m2.y == -INFINITY ? 0.0f : m2.y;
          const float p00 = dev::fast_exp2(y[4 * gg] - mx), p01 = dev::fast_exp2(y[4 * gg + 1] - my);
          const float p10 = dev::fast_exp2(y[4 * gg + 2] - mx), p11 = dev::fast_exp2(y[4 * gg + 3] - my);
          const bool k00 = !(y[4 * gg] > m2.x + 8.0f), k01 = !(y[4 * gg + 1] > m2.y + 8.0f);
          const bool k10 = !(y[4 * gg + 2] > m2.x + 8.0f), k11 = !(y[4 * gg + 3] > m2.y + 8.0f);
          flag |= !(k00 && k01 && k10 && k11);
          lp[2 * gg] += (k00 ? p00 : 0.0f) + (k10 ? p10 : 0.0f);
          lp[2 * gg + 1] += (k01 ? p01 : 0.0f) + (k11 ? p11 : 0.0f);
          pw[2 * gg] = KV == KV_FP8PT ? dev::pack_f16x2(p00 * sig0, p01 * sig0) : dev::pack_f16x2(p00, p01);
          pw[2 * gg + 1] = KV == KV_FP8PT ? dev::pack_f16x2(p10 * sig1, p11 * sig1) : dev::pack_f16x2(p10, p11);
        }
      }
      const int any = agree(flag);
      if (any < 0) return;
      if (!any) {
        if (pfree_wait && !wait(B_P_FREE + pb, pfree_par)) return;
#pragma unroll
        for (int gg = 0; gg < HN / 8; ++gg) {
          tc::sts_u32(prow + p_offset(HN, tok0, gg) + 2 * hq, pw[2 * gg]);
          tc::sts_u32(prow + p_offset(HN, tok1, gg) + 2 * hq, pw[2 * gg + 1]);
        }
      } else {
        if (!renew_maxima()) return;
        if (pfree_wait && !wait(B_P_FREE + pb, pfree_par)) return;
        // P against the renewed maxima; a renewed head's row sums drop the terms the first P gave
        // them, are rescaled, and take the new ones
        float y[HN / 2];
        logits<HN>(tl, s, hq, live0, live1, sig0, sig1, qsc, y);
#pragma unroll
        for (int gg = 0; gg < HN / 8; ++gg) {
          float pn[4];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int h = 8 * gg + hq + k;
            const float mo = red[h], mn = m_run[h], al = alpha[h];
            const float mref = mn == -INFINITY ? 0.0f : mn;
            pn[k] = dev::fast_exp2(y[4 * gg + k] - mref);
            pn[2 + k] = dev::fast_exp2(y[4 * gg + 2 + k] - mref);
            if (!(mn == mo)) {
              const float moref = mo == -INFINITY ? 0.0f : mo;
              const float po0 = !(y[4 * gg + k] > mo + 8.0f) ? dev::fast_exp2(y[4 * gg + k] - moref) : 0.0f;
              const float po1 = !(y[4 * gg + 2 + k] > mo + 8.0f) ? dev::fast_exp2(y[4 * gg + 2 + k] - moref) : 0.0f;
              lp[2 * gg + k] = al * (lp[2 * gg + k] - po0 - po1) + pn[k] + pn[2 + k];
            }
          }
          const uint32_t w0 = KV == KV_FP8PT ? dev::pack_f16x2(pn[0] * sig0, pn[1] * sig0) : dev::pack_f16x2(pn[0], pn[1]);
          const uint32_t w1 = KV == KV_FP8PT ? dev::pack_f16x2(pn[2] * sig1, pn[3] * sig1) : dev::pack_f16x2(pn[2], pn[3]);
          tc::sts_u32(prow + p_offset(HN, tok0, gg) + 2 * hq, w0);
          tc::sts_u32(prow + p_offset(HN, tok1, gg) + 2 * hq, w1);
        }
      }
    } else {
      // ---- from 48 heads (one P buffer), the agreement first ----
      bool flag = false;
      {
        float y[HN / 2];
        logits<HN>(tl, s, hq, live0, live1, sig0, sig1, qsc, y);
#pragma unroll
        for (int gg = 0; gg < HN / 8; ++gg) {
          const float2 m2 = *reinterpret_cast<const float2*>(m_run + 8 * gg + hq);
          flag |= (y[4 * gg] > m2.x + 8.0f) | (y[4 * gg + 1] > m2.y + 8.0f) | (y[4 * gg + 2] > m2.x + 8.0f) |
                  (y[4 * gg + 3] > m2.y + 8.0f);
        }
      }
      const int any = agree(flag);
      if (any < 0) return;
      if (any) {
        if (!renew_maxima()) return;
#pragma unroll
        for (int gg = 0; gg < HN / 8; ++gg) {
          const float2 a2 = *reinterpret_cast<const float2*>(alpha + 8 * gg + hq);
          lp[2 * gg] *= a2.x;
          lp[2 * gg + 1] *= a2.y;
        }
      }
      // ---- P = 2^(y - m), FP16 (per-token-scaled pages: times the token's scale): each thread writes
      // one 4-byte word (2 heads) per 8-head chunk of both its token rows ----
      if (pfree_wait && !wait(B_P_FREE + pb, pfree_par)) return;
      float y[HN / 2];
      logits<HN>(tl, s, hq, live0, live1, sig0, sig1, qsc, y);
#pragma unroll
      for (int gg = 0; gg < HN / 8; ++gg) {
        const float2 m2 = *reinterpret_cast<const float2*>(m_run + 8 * gg + hq);
        const float mx = m2.x == -INFINITY ? 0.0f : m2.x, my = m2.y == -INFINITY ? 0.0f : m2.y;
        const float p00 = dev::fast_exp2(y[4 * gg] - mx), p01 = dev::fast_exp2(y[4 * gg + 1] - my);
        const float p10 = dev::fast_exp2(y[4 * gg + 2] - mx), p11 = dev::fast_exp2(y[4 * gg + 3] - my);
        lp[2 * gg] += p00 + p10;
        lp[2 * gg + 1] += p01 + p11;
        const uint32_t w0 = KV == KV_FP8PT ? dev::pack_f16x2(p00 * sig0, p01 * sig0) : dev::pack_f16x2(p00, p01);
        const uint32_t w1 = KV == KV_FP8PT ? dev::pack_f16x2(p10 * sig1, p11 * sig1) : dev::pack_f16x2(p10, p11);
        tc::sts_u32(prow + p_offset(HN, tok0, gg) + 2 * hq, w0);
        tc::sts_u32(prow + p_offset(HN, tok1, gg) + 2 * hq, w1);
      }
    }
    tc::tc_fence_before();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(sy.bar(B_S_FREE + s));
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(sy.bar(B_P_FULL + pb));
    const bool last = cur.j == seg.num_pages - 1;
    cur.next(a);
    if (!last) continue;

    // ---- segment end: row sums over the 64 tokens (fixed order), then O / l from TMEM ----
    warp_reduce_heads<HN, false>(lp, red + w * HN, lane);
    if (!ssync(sy)) return;
    if (tid < HN) alpha[tid] = (red[tid] + red[HN + tid]) + (red[2 * HN + tid] + red[3 * HN + tid]);
    if (!ssync(sy)) return;
    if (!wait(B_P_FREE + pb, (g / C::kPBufs) & 1)) return;     // PV(g) has completed
    tc::tc_fence_after();
    const int64_t row0 = static_cast<int64_t>(seg.req) * a.heads;
    constexpr int CH = C::kChunk;
#pragma unroll 1
    for (int mt = 0; mt < 4; ++mt) {
      const int dim = 128 * mt + 32 * w + lane;
#pragma unroll 1
      for (int c0 = 0; c0 < HN; c0 += CH) {
        uint32_t o[CH];
        tmem_ld_cols<CH>(tl + C::TM_O + mt * HN + c0, o);
        tc::tmem_wait_ld();
#pragma unroll 4
        for (int u = 0; u < CH; ++u) {
          const int h = c0 + u;
          if (h < a.heads) {                    // 48 heads ride in 64 columns
            const float lt = alpha[h];
            const float v = __uint_as_float(o[u]) * (lt > 0.0f ? 1.0f / lt : 0.0f);
            if (seg.partial < 0) {
              const uint32_t b = dev::pack_bf16x2(v * a.out_scale, 0.0f);
              a.out[(row0 + h) * kDv + dim] = static_cast<uint16_t>(b & 0xFFFFu);
            } else {
              a.part_o[(static_cast<int64_t>(seg.partial) * a.heads + h) * kDv + dim] = v;
            }
          }
        }
      }
    }
    tc::tc_fence_before();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(sy.bar(B_O_FREE));
    if (tid < HN && tid < a.heads) {
      const float lt = alpha[tid];
      const float lse2 = lt > 0.0f ? m_run[tid] + __log2f(lt) : -INFINITY;
      if (seg.partial < 0) { if (a.lse) a.lse[row0 + tid] = lse2 * 0.69314718055994531f; }
      else a.part_lse[static_cast<int64_t>(seg.partial) * a.heads + tid] = lse2;
    }
    // every thread is done with this segment's maxima and sums before the next segment resets them
    if (!ssync(sy)) return;
  }
}

template <int KV, int HN>
__global__ void __launch_bounds__(Cfg<HN>::kThreads, 1) decode_tm_kernel(const DecodeArgs a) {
  using C = Cfg<HN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int worker = blockIdx.x;
  const int seg_b = a.worker_ptr[worker], seg_e = a.worker_ptr[worker + 1];
  Sync sy;
  sy.bars = base + C::OFF_BAR;
  sy.abort = reinterpret_cast<volatile int*>(sbase + C::OFF_ABORT);
  sy.status = a.status;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(sy.bar(B_T_FULL + i), C::kDQ);
      tc::mbar_init(sy.bar(B_T_EMPTY + i), C::kPvThreads);   // the P.V commits of the page
      tc::mbar_init(sy.bar(B_S_FULL + i), 2);                // both K halves of the page's Q.K^T
      tc::mbar_init(sy.bar(B_S_FREE + i), 4);
    }
    for (int i = 0; i < C::kPBufs; ++i) {
      tc::mbar_init(sy.bar(B_P_FULL + i), 4);
      tc::mbar_init(sy.bar(B_P_FREE + i), C::kPvThreads);
    }
    tc::mbar_init(sy.bar(B_O_FREE), 4);
    tc::mbar_init(sy.bar(B_SYNC), 4);
    tc::mbar_init(sy.bar(B_FINAL), 2 + C::kPvThreads);   // one commit per MMA-issuing thread
    *sy.abort = 0;
    *reinterpret_cast<volatile uint32_t*>(sbase + C::OFF_QVER) = 0;
    tc::fence_mbar_init();
  }
  if (warp == C::kPvWarp0) {
    tc::tmem_alloc(base + C::OFF_TSLOT, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(sbase + C::OFF_TSLOT);

  if (warp < 4) {
    role_softmax<KV, HN>(a, sy, seg_b, seg_e, tid, tbase, base, sbase);
  } else if (warp < C::kPvWarp0) {
    role_dequant<KV, C::kDQ>(a, sy, seg_b, seg_e, tid - 128, base + C::OFF_T);
  } else if (warp == C::kPvWarp0 || warp == C::kPvWarp1) {
    if ((tid & 31) == 0)
      role_pv<HN>(a, sy, seg_b, seg_e, warp == C::kPvWarp0 ? 0 : 1, tbase, base + C::OFF_T, base + C::OFF_P);
  } else if ((tid & 31) == 0) {
    role_qk<HN>(a, sy, seg_b, seg_e, warp - C::kQkWarp0, tbase, base + C::OFF_T, base + C::OFF_Q, base + C::OFF_QVER);
  }
  // every MMA of the issuing threads has completed before TMEM is released
  if (warp >= C::kPvWarp0 && (tid & 31) == 0) sy.wait(B_FINAL, 0, false, kStatusBase << 6);
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == C::kPvWarp0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tbase, 512);
  }
}

template <int KV, int HN>
cudaError_t launch_kv_hn(const DecodeArgs& a, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_tm_kernel<KV, HN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<HN>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  decode_tm_kernel<KV, HN><<<static_cast<unsigned>(a.num_workers), Cfg<HN>::kThreads, Cfg<HN>::kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

template <int KV>
cudaError_t launch_kv(const DecodeArgs& a, cudaStream_t s) {
  switch (tm_heads_padded(a.heads)) {
    case 16: return launch_kv_hn<KV, 16>(a, s);
    case 32: return launch_kv_hn<KV, 32>(a, s);
    case 64: return launch_kv_hn<KV, 64>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int tm_heads_padded(int heads) {
  if (heads < 16 || heads > 64 || heads % 16) return 0;
  return heads <= 16 ? 16 : heads <= 32 ? 32 : 64;
}

cudaError_t launch_decode_tm(const DecodeArgs& a, cudaStream_t s) {
  if (a.num_segments == 0) return cudaSuccess;
  if (tm_heads_padded(a.heads) == 0 || a.ctas_per_worker != 1) return cudaErrorInvalidValue;
  switch (a.kv_dtype) {
    case KV_FP8: return launch_kv<KV_FP8>(a, s);
    case KV_NVFP4: return launch_kv<KV_NVFP4>(a, s);
    case KV_FP8PT: return launch_kv<KV_FP8PT>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qkvp
