// Split-KV paged MLA decode on the 5th-generation tensor cores (tcgen05, TMEM accumulators), 128 heads.
//
// The attention is the one of the pages' plan()/run() call ("The Smoking Gun", section "What
// Message 1408 Actually Reveals"): per request and head, softmax(sm_scale * q . k) v over the
// request's tokens, K = the 576-wide latent, V = its first 512 dims, read from quantized pages and
// dequantized on chip ("SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "SGLang
// implementation", item 3). Products take FP16 operands with FP32 accumulation (exact K/V, 11-bit
// probabilities), the same arithmetic as the mma.sync kernel.
//
// Work split. The FP32 output of 128 heads x 512 dims fills all 512 TMEM columns of an SM, so one
// work item runs on a pair of CTAs (a cluster of two), and the pair splits each 64-token page by
// tokens: CTA c computes the full 576-dim logits of tokens [32c, 32c + 32) for all 128 heads, the
// two CTAs trade their 128 row maxima (512 bytes) so that both scale by the same running maximum,
// and each sends its half of the probabilities P (128 x 32 FP16, 8 KB) to the other with one bulk
// asynchronous copy. CTA c then accumulates output dims [256c, 256c + 256) over all 64 tokens: the
// V rows of its own tokens are already in its operand tile, and it dequantizes the other 32 tokens'
// rows for its 256 dims itself (a second read of those bytes, served by L2). Trading logits
// instead (a split by dims) would move 32 KB per page over the SM-to-SM network, whose bandwidth
// (about 12 bytes per clock per SM) then bounds the whole kernel.
//
// Per CTA (384 threads, three warps per SM sub-partition):
//   warps 0-3 (softmax): thread h owns head h = TMEM lane h. Loads Q once per request (in this CTA's
//     contraction order: the first 384 dims into TMEM as the A operand of Q.K^T, the rest into
//     shared memory), then per page:
//     reads its 32 logits, trades the row maximum with the peer (asynchronous remote stores counted
//     on the peer's mbarrier, so no fence is needed), runs the FP32 online softmax (base
//     2, lazy rescale of O when the running maximum grows by more than 2^8), writes its row of P and
//     hands the half to the peer. At the end of a segment the two CTAs trade their row sums, and
//     each writes its 256 output dims.
//   warps 4-8 (dequant): per page, load the raw bytes of the own 32 tokens (all dims) and of the
//     other 32 tokens (own V dims), the next page's loads in flight while the current page is
//     converted, and write FP16 operand tiles (two rings, split by how long each part is read).
//   warps 11 and 9 (QK): one thread each issues S = Q.K^T (M 128 heads x N 32 tokens x K 576) into
//     TMEM for the even / odd pages (the two logit buffers).
//   warp 10 (PV): one thread issues O += P.V (M 128 x N 256 x K 64) into the TMEM accumulator; the
//     P.V commit that frees a P buffer goes to both CTAs. tcgen05.commit signals the other roles.
// TMEM: O [0, 256), Q dims 0..383 as FP16 pairs [256, 448), two logit buffers [448, 512).
// Barrier phases: every barrier is waited on by parity, which is only sound while the barrier is at
// most one phase away from the phase waited for; the comments at each wait say why that holds. A
// barrier whose waiter skips phases (a Q.K^T thread sees only every other page) would break that, so
// the Q.K^T threads wait only on their own K slot (one slot per parity, armed after both rings of the
// page are written), and the new-request Q is published as a counter instead of a barrier phase.
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
using kern::ldg_nc;
using kern::ldg_nc32;
using kern::page_ok;
using kern::sts128;
using kern::sts128_relaxed;

constexpr int kThreads = 384;
constexpr int kDQ = 160;                     // dequant threads (warps 4-8)
// MMA issue: one thread in each of warps 9 and 11 issues Q.K^T for odd / even pages, one in warp 10
// issues P.V. A thread waits a few tens of cycles after each tcgen05.mma it issues before the next one
// can go; several issuing threads overlap those waits and keep the tensor pipe fed.
constexpr int kQkWarpOdd = 9, kPvWarp = 10, kMmaWarp = 11;
constexpr int kHalf = 32;                    // tokens of a page per CTA
constexpr uint32_t kAtom = 4096;             // 32 token rows x 64 dims FP16, 128-byte swizzle
// Operand tiles of a page live in two rings by lifetime: the K-only ring holds the own tokens' dims
// that only Q.K^T reads (the other CTA's 256 nope dims and the 64 rope dims: 5 atoms), freed when
// Q.K^T completes; the V ring holds this CTA's 256 V dims of the own tokens (read by Q.K^T and P.V)
// and of the other 32 tokens (P.V only): 8 atoms, freed when P.V completes.
constexpr int kKSlots = 2, kVSlots = 3;
// Pages ahead that the dequant role prefetches into L2. Measured on one GB300: FP8 pools gain (44 x 32K:
// 515 -> 507 us); NVFP4 pools lose (10 x 160K: 724 -> 747 us), per-token-scaled FP8 pools too (44 x
// 32K: 584 -> 607 us four pages ahead, 617 us two ahead, the token rows alone or with their scales),
// and BF16 pools are unchanged. So FP8 only.
template <int KV>
constexpr int prefetch_ahead() { return KV == KV_FP8 ? 4 : 0; }
constexpr uint32_t kKSlot = 5 * kAtom;
constexpr uint32_t kVSlot = 8 * kAtom;
constexpr uint32_t kPHalf = 8192;            // 128 heads x 32 tokens FP16, 64-byte swizzle
constexpr uint32_t kPBytes = 2 * kPHalf;
constexpr uint32_t kQAtom = 16384;           // 128 heads x 64 dims FP16, 128-byte swizzle
constexpr int kQTmemDims = 384;              // Q dims held in TMEM; dims 384..575 in shared memory
constexpr int kQSmemAtoms = (kLatent - kQTmemDims) / 64;

constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_V = OFF_K + kKSlots * kKSlot;
constexpr uint32_t OFF_P = OFF_V + kVSlots * kVSlot;
constexpr uint32_t OFF_Q = OFF_P + 2 * kPBytes;
constexpr uint32_t OFF_RM = OFF_Q + kQSmemAtoms * kQAtom;   // 2 x 128 FP32: the peer's row maxima
constexpr uint32_t OFF_LX = OFF_RM + 2 * 512;               // 2 x 128 FP32: the peer's row sums
constexpr uint32_t OFF_SIG = OFF_LX + 2 * 512;             // per softmax warp, the page's own 32 token scales
constexpr uint32_t OFF_BAR = OFF_SIG + 4 * 128;
enum : uint32_t {
  B_K_FULL = 0, B_K_EMPTY = 2, B_V_FULL = 4, B_V_EMPTY = 7, B_S_FULL = 10, B_S_FREE = 12, B_P_LOCAL = 14,
  B_P_FULL = 16, B_P_FREE = 18, B_O_DONE = 20, B_Q_READY = 22, B_FINAL = 23, B_RM_FULL = 24, B_LX_FULL = 26,
  NUM_BARS = 28
};
constexpr uint32_t OFF_TSLOT = OFF_BAR + 8 * NUM_BARS;
constexpr uint32_t OFF_ABORT = OFF_TSLOT + 4;
constexpr uint32_t OFF_QVER = OFF_ABORT + 4;        // number of request Q rows published so far
constexpr uint32_t kSmemUsed = OFF_QVER + 8;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;   // slack to align the base to 1024 bytes
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(OFF_V % 1024 == 0 && OFF_P % 1024 == 0 && OFF_Q % 1024 == 0, "swizzle atoms");

// TMEM: O, Q dims 0..383 as FP16 pairs, two logit buffers of 32 columns
constexpr uint32_t TM_O = 0, TM_Q = 256, TM_S = 448;
static_assert(TM_Q + kQTmemDims / 2 == TM_S && TM_S + 2 * kHalf == 512, "TMEM columns");

constexpr uint32_t kIdescQK = tc::idesc_f16(128, kHalf, 0, 0);
constexpr uint32_t kIdescPV = tc::idesc_f16(128, 256, 0, 1);

// ---- dequantization of a page into the two operand rings -------------------------------------
// K slot: own tokens (rows 0..31 = tokens 32c..32c+31) x the 4 nope atoms of the other CTA's dims,
// then the rope atom. V slot: own tokens x this CTA's 4 nope atoms (dims 256c..256c+255), then the
// other 32 tokens (rows = tokens 32(1-c)..) x the same 4 atoms. Atoms are 64 dims x 32 rows, 4 KB,
// 128-byte swizzle. Work is cut into items of 16 raw bytes; consecutive items cover the 16-byte
// chunks of neighbouring rows of one atom so that every group of eight 16-byte shared stores lands
// in eight distinct bank groups. Rows of tokens past the page's valid count are written as zeros (the
// pool may hold anything there, NaN codes included).
struct Item {
  int tok;          // token within the page
  int row;          // row within the atom
  int dim;          // first latent dim of the item
  bool in_v;        // destination ring
  uint32_t off;     // byte offset of the item's atom within its slot
};

__device__ __forceinline__ Item item_at(int own_items, int q, int c, int per_atom, int j, int row) {
  Item it;
  const bool own = q < own_items;
  const int qq = own ? q : q - own_items;
  const int a = qq / per_atom;              // own: latent atom 0..8; other: V atom 0..3
  it.row = row;
  it.tok = own ? kHalf * c + row : kHalf * (1 - c) + row;
  it.dim = (own ? 0 : 256 * c) + 64 * a + j;
  if (!own) { it.in_v = true; it.off = (4 + a) * kAtom; }
  else if (a < 8 && (a >> 2) == c) { it.in_v = true; it.off = (a & 3) * kAtom; }
  else { it.in_v = false; it.off = (a < 8 ? (a & 3) : 4) * kAtom; }
  return it;
}

template <int KV> struct Dequant;

template <> struct Dequant<KV_FP8> {
  // 32 dims (32 raw bytes, one 32-byte load) per item, 2 items per atom row: own 32 rows x 18, other
  // 32 rows x 8. Wide loads halve the load instructions, which the per-SM queue of outstanding
  // global loads otherwise throttles.
  static constexpr int kOwn = 32 * 18, kItems = kOwn + 32 * 8;
  static constexpr int kIters = (kItems + kDQ - 1) / kDQ;
  struct Raw { uint32_t v[kIters][8]; };
  __device__ static Item at(int q, int c) {
    const int qq = q < kOwn ? q : q - kOwn;
    return item_at(kOwn, q, c, 64, 32 * (qq & 1), ((qq >> 3) & 7) * 4 + ((qq >> 1) & 3));
  }
  __device__ static void load(Raw& r, const DecodeArgs& a, int64_t page, int valid, int c, int t) {
    const uint8_t* base = a.kv + page * (kPage * kLatent);
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + kDQ * i;
      const Item it = at(q, c);
      if (q < kItems && it.tok < valid) ldg_nc32(base + it.tok * kLatent + it.dim, r.v[i]);
    }
  }
  __device__ static void store(const Raw& r, const DecodeArgs&, int64_t, int valid, int c, int t, uint32_t ks, uint32_t vs,
                               uint32_t) {
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + kDQ * i;
      if (q >= kItems) continue;
      const Item it = at(q, c);
      uint32_t o[16];
#pragma unroll
      for (int b = 0; b < 16; ++b)
        o[b] = it.tok < valid ? dev::e4m3x2_to_f16x2(static_cast<uint16_t>(r.v[i][b >> 1] >> (16 * (b & 1)))) : 0u;
      const uint32_t ch = ((it.dim & 63) >> 3), at = (it.in_v ? vs : ks) + it.off;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        sts128(at + tc::sw128_offset(it.row, ch + u), make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]));
    }
  }
};

template <> struct Dequant<KV_FP8PT> {
  // the FP8 items of a per-token-scaled page (codes converted exactly); the token scales are read by
  // the softmax warps, which apply them in FP32
  static constexpr int kIters = Dequant<KV_FP8>::kIters;
  using Raw = Dequant<KV_FP8>::Raw;
  __device__ static void load(Raw& r, const DecodeArgs& a, int64_t page, int valid, int c, int t) {
    const uint8_t* base = a.kv + page * kPtPageBytes;
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + kDQ * i;
      const Item it = Dequant<KV_FP8>::at(q, c);
      if (q < Dequant<KV_FP8>::kItems && it.tok < valid) ldg_nc32(base + it.tok * kLatent + it.dim, r.v[i]);
    }
  }
  __device__ static void store(const Raw& r, const DecodeArgs& a, int64_t page, int valid, int c, int t, uint32_t ks,
                               uint32_t vs, uint32_t sg) {
    Dequant<KV_FP8>::store(r, a, page, valid, c, t, ks, vs, sg);
  }
};

template <> struct Dequant<KV_NVFP4> {
  // 64 dims per item: 32 packed bytes in one 32-byte load and the four block scales in one 4-byte
  // load; one item fills one atom row (own 32 rows x 9 atoms, other 32 rows x 4). Items of 32 dims
  // took one 16-byte and one 2-byte load each, twice the load instructions for the same bytes.
  // A warp's 32 items are the 32 rows of one atom, so each of the 8 row stores hits eight distinct
  // bank groups per eight lanes.
  static constexpr int kOwn = 32 * 9, kItems = kOwn + 32 * 4;
  static constexpr int kIters = (kItems + kDQ - 1) / kDQ;
  struct Raw { uint32_t v[kIters][8]; uint32_t s[kIters]; };
  __device__ static Item at(int q, int c) {
    const int qq = q < kOwn ? q : q - kOwn;
    return item_at(kOwn, q, c, 32, 0, qq & 31);
  }
  __device__ static void load(Raw& r, const DecodeArgs& a, int64_t page, int valid, int c, int t) {
    const uint8_t* base = a.kv + page * (kPage * kPacked);
    const uint8_t* sbase = a.kv_scale + page * (kPage * kScales);
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + kDQ * i;
      const Item it = at(q, c);
      if (q < kItems && it.tok < valid) {
        ldg_nc32(base + it.tok * kPacked + it.dim / 2, r.v[i]);
        r.s[i] = *reinterpret_cast<const uint32_t*>(sbase + it.tok * kScales + it.dim / 16);
      }
    }
  }
  __device__ static void store(const Raw& r, const DecodeArgs&, int64_t, int valid, int c, int t, uint32_t ks, uint32_t vs,
                               uint32_t) {
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + kDQ * i;
      if (q >= kItems) continue;
      const Item it = at(q, c);
      uint32_t o[32];
      if (it.tok < valid) {
        uint32_t h[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t sk = (r.s[i] >> (8 * k)) & 0xFFu;
          h[k] = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(sk | (sk << 8)));
        }
#pragma unroll
        for (int wv = 0; wv < 8; ++wv) {
          // the word's four code pairs from byte registers: a shift and a mask per pair made this
          // loop the NVFP4 kernel's bound (10 x 160K: 725 us; a byte permute 665 us; this 604 us)
          uint32_t c4[4];
          dev::e2m1x8_to_f16x2x4(r.v[i][wv], c4);
#pragma unroll
          for (int k = 0; k < 4; ++k) o[4 * wv + k] = dev::hmul2_f16(c4[k], h[wv >> 1]);
        }
      } else {
#pragma unroll
        for (int b = 0; b < 32; ++b) o[b] = 0;
      }
      const uint32_t at = (it.in_v ? vs : ks) + it.off;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        sts128(at + tc::sw128_offset(it.row, u), make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]));
    }
  }
};

template <> struct Dequant<KV_BF16> {      // the cast-then-attend baseline: BF16 pages
  // 8 dims (16 bytes) per item, 8 items per atom row; converted in rounds of 12 items per thread
  static constexpr int kOwn = 32 * 72, kItems = kOwn + 32 * 32;
  static constexpr int kRound = 12;
  struct Raw {};
  __device__ static Item at(int q, int c) {
    const int qq = q < kOwn ? q : q - kOwn;
    return item_at(kOwn, q, c, 256, 8 * (qq & 7), (qq >> 3) & 31);
  }
  __device__ static void load(Raw&, const DecodeArgs&, int64_t, int, int, int) {}
  __device__ static void store(const Raw&, const DecodeArgs& a, int64_t page, int valid, int c, int t, uint32_t ks, uint32_t vs,
                               uint32_t) {
    const uint8_t* base = a.kv + page * (kPage * kLatent * 2);
#pragma unroll 1
    for (int r0 = 0; r0 < kItems; r0 += kDQ * kRound) {
      uint4 v[kRound];
#pragma unroll
      for (int i = 0; i < kRound; ++i) {
        const int q = r0 + t + kDQ * i;
        const Item it = at(q, c);
        if (q < kItems && it.tok < valid) v[i] = ldg_nc(base + (it.tok * kLatent + it.dim) * 2);
      }
#pragma unroll
      for (int i = 0; i < kRound; ++i) {
        const int q = r0 + t + kDQ * i;
        if (q >= kItems) continue;
        const Item it = at(q, c);
        uint4 o = make_uint4(0, 0, 0, 0);
        if (it.tok < valid) o = make_uint4(dev::bf16x2_to_f16x2(v[i].x), dev::bf16x2_to_f16x2(v[i].y),
                                           dev::bf16x2_to_f16x2(v[i].z), dev::bf16x2_to_f16x2(v[i].w));
        sts128((it.in_v ? vs : ks) + it.off + tc::sw128_offset(it.row, (it.dim & 63) >> 3), o);
      }
    }
  }
};

// ---- roles -------------------------------------------------------------------------------------------
// L2 prefetch of the bytes of a page that this CTA's raw loads start from: its own 32 token rows (and
// their scales). The peer prefetches the other 32 rows, whose 256 V dims this CTA also reads.
template <int KV>
__device__ __forceinline__ void prefetch_page(const DecodeArgs& a, int64_t page, int c) {
  if constexpr (KV == KV_FP8) {
    tc::bulk_prefetch_l2(a.kv + page * (kPage * kLatent) + 32 * c * kLatent, 32 * kLatent);
  } else if constexpr (KV == KV_FP8PT) {
    const uint8_t* base = a.kv + page * kPtPageBytes;
    tc::bulk_prefetch_l2(base + 32 * c * kLatent, 32 * kLatent);
    tc::bulk_prefetch_l2(base + kPtScaleOff + 128 * c, 128);
  } else if constexpr (KV == KV_NVFP4) {
    tc::bulk_prefetch_l2(a.kv + page * (kPage * kPacked) + 32 * c * kPacked, 32 * kPacked);
    tc::bulk_prefetch_l2(a.kv_scale + page * (kPage * kScales) + 32 * c * kScales, 32 * kScales);
  } else {
    tc::bulk_prefetch_l2(a.kv + page * (kPage * kLatent * 2) + 32 * c * kLatent * 2, 32 * kLatent * 2);
  }
}

template <int KV>
__device__ void role_dequant(const DecodeArgs& a, const Sync& sy, int seg_b, int seg_e, int c, int t, uint32_t kring,
                             uint32_t vring, uint32_t sigring) {
  using D = Dequant<KV>;
  // Page indices are read one page before they are needed (raw loads of page g + 1 are issued while
  // page g is converted, with the index of page g + 2 already in flight), so no iteration waits on a
  // dependent index load.
  Cursor cur;
  cur.begin(a, seg_b, seg_e);
  if (cur.done()) return;
  typename D::Raw raw_cur, raw_nxt;
  Cursor nx = cur;
  nx.next(a);
  int64_t pg = cur.page(a);
  int64_t npg = nx.done() ? 0 : nx.page(a);
  int valid = page_ok(a, pg) ? cur.valid() : 0;
  D::load(raw_cur, a, pg, valid, c, t);
  // One thread keeps pages kAhead ahead flowing into L2 (pages 2 .. kAhead - 1 at the start), so the
  // raw loads of the next page find them there instead of in HBM; the page index it needs is read
  // an iteration before its use.
  constexpr int kAhead = prefetch_ahead<KV>();
  Cursor pf = cur;
  int64_t pf_pg = -1;
  if (kAhead > 0 && t == 0) {
    for (int i = 0; i < kAhead && !pf.done(); ++i) {
      if (i >= 2) {
        const int64_t p2 = pf.page(a);
        if (page_ok(a, p2)) prefetch_page<KV>(a, p2, c);
      }
      pf.next(a);
    }
    if (!pf.done()) pf_pg = pf.page(a);
  }
  for (int g = 0; !cur.done(); ++g) {
    if (kAhead > 0 && t == 0 && !pf.done()) {
      if (page_ok(a, pf_pg)) prefetch_page<KV>(a, pf_pg, c);
      pf.next(a);
      pf_pg = pf.done() ? -1 : pf.page(a);
    }
    Cursor nn = nx;
    if (!nn.done()) nn.next(a);
    const int64_t nnpg = nn.done() ? 0 : nn.page(a);
    const int nvalid = nx.done() ? 0 : (page_ok(a, npg) ? nx.valid() : 0);
    if (!nx.done()) D::load(raw_nxt, a, npg, nvalid, c, t);
    const int kb = g % kKSlots, vb = g % kVSlots;
    // the K slot was last used by page g - 2 (its Q.K^T completion is that barrier's previous
    // phase), the V slot by page g - 3 (its P.V completion)
    if (g >= kKSlots && !sy.wait(B_K_EMPTY + kb, ((g / kKSlots) - 1) & 1, false, 2)) return;
    if (g >= kVSlots && !sy.wait(B_V_EMPTY + vb, ((g / kVSlots) - 1) & 1, false, 2)) return;
    D::store(raw_cur, a, pg, valid, c, t, kring + kb * kKSlot, vring + vb * kVSlot, sigring + vb * 128);
    tc::fence_proxy_async_smem();
    // the V slot first: the Q.K^T threads wait only on the K slot and take it as "page written"
    tc::mbar_arrive(sy.bar(B_V_FULL + vb));
    tc::mbar_arrive(sy.bar(B_K_FULL + kb));
    raw_cur = raw_nxt;
    cur = nx;
    nx = nn;
    pg = npg;
    npg = nnpg;
    valid = nvalid;
  }
}

// The 36 MMAs of one page's S = Q.K^T, issued back to back. The contraction runs over the latent
// dims in this CTA's order: its own 256 nope dims (V slot atoms 0..3), the other 256 nope dims (K slot
// atoms 0..3), then the rope dims (K slot atom 4); Q is stored in the same order (the first 384 of
// them in TMEM, the rest in shared memory). Every operand is then a compile-time offset from a
// per-page base, the same for both CTAs, so one unrolled body serves both.
__device__ __forceinline__ void issue_qk(uint32_t ts, uint32_t tq, const tc::Desc2& kd, const tc::Desc2& vd,
                                         const tc::Desc2& qd) {
#pragma unroll
  for (int ks = 0; ks < 36; ++ks) {             // permuted dims 16ks .. 16ks + 15
    constexpr int kTm = kQTmemDims / 16;
    const uint64_t b = ks < 16 ? vd.at((ks >> 2) * kAtom + 32 * (ks & 3))
                               : kd.at(((ks - 16) >> 2) * kAtom + 32 * (ks & 3));
    if (ks < kTm) {                             // A operand: Q from TMEM
      if (ks == 0) tc::mma_ts_k<false>(ts, tq, b, kIdescQK);
      else tc::mma_ts_k<true>(ts, tq + 8 * ks, b, kIdescQK);
    } else {                                    // A operand: Q from shared memory
      const int kq = ks - kTm;
      tc::mma_ss_k<true>(ts, qd.at((kq >> 2) * kQAtom + 32 * (kq & 3)), b, kIdescQK);
    }
  }
}

// MMA issue, split over two threads in different warps so that neither stream waits behind the
// other: one thread issues S = Q.K^T page after page (each needs its operand tile, the logit buffer
// read out for the previous page and, at a new request, the new Q), the other issues O += P.V as
// soon as both halves of P have arrived. A tcgen05.commit tracks only the MMAs of the thread that
// issues it, so each stream signals its own completions.
__device__ void role_qk(const DecodeArgs& a, const Sync& sy, int seg_b, int seg_e, int c, int parity, uint32_t tbase,
                        uint32_t kring, uint32_t vring, uint32_t qs, uint32_t qver) {
  Cursor cq;
  cq.begin(a, seg_b, seg_e);
  const uint64_t k_desc0 = tc::smem_desc(kring, 16, 1024, tc::kSwizzle128);       // K-major, rows = tokens
  const uint64_t v_desc0 = tc::smem_desc(vring, 16, 1024, tc::kSwizzle128);
  const tc::Desc2 qd = tc::split_desc(tc::smem_desc(qs, 16, 1024, tc::kSwizzle128));   // K-major, rows = heads
  // requests are counted over all pages (both parities), in the order the softmax loads their Q
  int qcount = 0, q_req = -1, q_waited = -1;
  for (int gq = 0; !cq.done(); ++gq, cq.next(a)) {
    if (cq.j == 0 && cq.seg.req != q_req) { q_req = cq.seg.req; ++qcount; }
    if ((gq & 1) != parity) continue;
    const int kb = gq % kKSlots, vb = gq % kVSlots, s = gq & 1;
    // K slot kb holds only pages of this parity, so this thread waits on each of its phases in turn;
    // the dequant arrives on it after writing both rings of the page (the V slot included)
    if (!sy.wait(B_K_FULL + kb, (gq / kKSlots) & 1, false, 4)) break;
    // logit buffer s was last read out for page gq - 2 (also this thread's)
    if (gq >= 2 && !sy.wait(B_S_FREE + s, ((gq >> 1) - 1) & 1, false, 4)) break;
    // the Q rows of this page's request: the qcount-th request Q published by the softmax threads
    if (q_waited != qcount) {
      if (!kern::wait_counter(sy, qver, static_cast<uint32_t>(qcount), 8)) break;
      q_waited = qcount;
    }
    tc::tc_fence_after();
    const tc::Desc2 kd = tc::split_desc(tc::desc_add(k_desc0, kb * kKSlot));
    const tc::Desc2 vd = tc::split_desc(tc::desc_add(v_desc0, vb * kVSlot));
    issue_qk(tbase + TM_S + kHalf * s, tbase + TM_Q, kd, vd, qd);
    tc::mma_commit(sy.bar(B_S_FULL + s));
    tc::mma_commit(sy.bar(B_K_EMPTY + kb));
  }
  // drain: every MMA issued by this thread has completed before TMEM is released
  tc::mma_commit(sy.bar(B_FINAL));
}

__device__ void role_pv(const DecodeArgs& a, const Sync& sy, int seg_b, int seg_e, int c, uint32_t tbase,
                        uint32_t vring, uint32_t pbuf) {
  Cursor cp;
  cp.begin(a, seg_b, seg_e);
  const uint64_t v_desc0 = tc::smem_desc(vring, kAtom, 1024, tc::kSwizzle128);    // MN-major (V), 4 dim atoms
  const uint64_t p_desc0 = tc::smem_desc(pbuf, 16, 512, tc::kSwizzle64);          // K-major, rows = heads
  for (int gp = 0; !cp.done(); ++gp) {
    const int s = gp & 1, vb = gp % kVSlots;
    if (!sy.wait(B_P_FULL + s, (gp >> 1) & 1, false, 4)) break;
    // already complete (Q.K^T of this page waited for it); cannot advance before this P.V frees it
    if (!sy.wait(B_V_FULL + vb, (gp / kVSlots) & 1, false, 4)) break;
    tc::tc_fence_after();
    const uint64_t pd = tc::desc_add(p_desc0, s * kPBytes);
    const uint64_t vown = tc::desc_add(v_desc0, vb * kVSlot);
    const uint64_t voth = tc::desc_add(v_desc0, vb * kVSlot + 4 * kAtom);
    // tokens 16kk .. 16kk + 15: P half kk / 2, V rows from the own K tile or the other-token V tile
    const uint64_t v0 = c == 0 ? vown : voth, v1 = c == 0 ? voth : vown;
    if (cp.j == 0) tc::mma_ss_k<false>(tbase + TM_O, pd, v0, kIdescPV);
    else tc::mma_ss_k<true>(tbase + TM_O, pd, v0, kIdescPV);
    tc::mma_ss_k<true>(tbase + TM_O, tc::desc_add(pd, 32), tc::desc_add(v0, 2048), kIdescPV);
    tc::mma_ss_k<true>(tbase + TM_O, tc::desc_add(pd, kPHalf), v1, kIdescPV);
    tc::mma_ss_k<true>(tbase + TM_O, tc::desc_add(pd, kPHalf + 32), tc::desc_add(v1, 2048), kIdescPV);
    tc::mma_commit(sy.bar(B_V_EMPTY + vb));
    tc::mma_commit_multicast(sy.bar(B_P_FREE + s), 0x3);
    tc::mma_commit(sy.bar(B_O_DONE + s));
    cp.next(a);
  }
  tc::mma_commit(sy.bar(B_FINAL));
}

// Softmax role. Per page: logits of the own 32 tokens from TMEM, row maximum traded with the peer,
// online softmax, own half of P written and copied to the peer. Every wait is followed by a warp
// vote, so the warps stay converged for the warp-collective tcgen05.ld / tcgen05.st and continue or
// give up as a whole.
// The exchange buffers need no "free" barriers: the peer writes the row-maximum slot of page g + 2
// (and the row-sum slot of a later segment end of the same parity) only after it has received this
// CTA's row maxima of page g + 1, which this CTA sends after it has read the slot of page g.
template <int KV>
__device__ void role_softmax(const DecodeArgs& a, const Sync& sy, int seg_b, int seg_e, int c, int h,
                             uint32_t tbase, uint32_t pbuf, uint32_t qs, uint32_t rm, uint32_t lx, uint32_t qver,
                             float* sig) {
  const uint32_t peer = c ^ 1u;
  const uint32_t tl = tbase + (static_cast<uint32_t>(h & ~31) << 16);   // this warp's TMEM lane quarter
  auto wait = [&](uint32_t bar, uint32_t parity, bool cluster, int code) -> bool {
    const bool ok = sy.wait(bar, parity, cluster, code);
    return __all_sync(0xffffffffu, ok);
  };
  float m_used = -INFINITY, l = 0.0f;          // running softmax state of the segment
  int lx_count[2] = {0, 0};                    // segment ends seen at even / odd pages
  Cursor cur;
  cur.begin(a, seg_b, seg_e);
  int cur_req = -1, nq = 0;
  float q_scale = a.scale_log2;
  int64_t pg = cur.done() ? 0 : cur.page(a);
  // per-token-scaled pages: lane i of every softmax warp reads the scale of own token i of the page
  // after the current one (zero past the valid tokens) and hands it to its warp through shared memory
  // when that page comes; each scale multiplies its token's logit and probability in FP32 (not the
  // row sum)
  float* sgp = sig + 32 * (h >> 5);
  auto token_scale = [&](const Cursor& cu, int64_t page) -> float {
    if (KV != KV_FP8PT || cu.done() || !page_ok(a, page)) return 0.0f;
    const int tok = kHalf * c + (h & 31);
    return tok < cu.valid() ? __ldg(reinterpret_cast<const float*>(a.kv + page * kPtPageBytes + kPtScaleOff) + tok) : 0.0f;
  };
  float sg_lane = token_scale(cur, pg);
  for (int g = 0; !cur.done(); ++g) {
    const Segment seg = cur.seg;
    if (cur.j == 0 && seg.req != cur_req) {
      // ---- Q row of head h (QK of the previous page has completed: its logits were read) ----
      // With fewer than 128 query heads the rows h >= heads hold zeros: their logits are 0, their
      // softmax runs on them harmlessly and nothing of theirs is written.
      // BF16 -> FP16 is exact for magnitudes in [2^-14, 2^15): the row is converted unscaled. A warp
      // holding a row with a value of 2^15 or more (or inf / NaN) converts again, with each such row
      // scaled by 2^-sh from its largest |q| (which then lies in [2^14, 2^15)); 2^sh joins the row's
      // logit scale. Both CTAs of the pair take the same decisions. Elements below 2^-14 become FP16
      // subnormals (flushed to zero below 2^-25); an unscaled row loses nothing else.
      const bool live = h < a.heads;
      const uint8_t* qrow = reinterpret_cast<const uint8_t*>(a.q) + (static_cast<int64_t>(seg.req) * a.heads + (live ? h : 0)) * (kLatent * 2);
      // latent dim of position d in this CTA's contraction order (own nope dims, other nope dims, rope)
      auto perm = [c](int d) { return d < 256 ? 256 * c + d : (d < 512 ? 256 * (1 - c) + d - 256 : d); };
      auto big = [](uint32_t w) { return (w & 0x7FFFu) >= 0x4700u || ((w >> 16) & 0x7FFFu) >= 0x4700u; };
      float down = 1.0f;
      q_scale = a.scale_log2;
#pragma unroll 1
      for (int attempt = 0; attempt < 2; ++attempt) {
        bool hot = false;
#pragma unroll 1
        for (int part = 0; part < kQTmemDims / 64; ++part) {   // 64 dims -> 32 TMEM columns
          uint32_t r[32];
          const uint8_t* src = qrow + perm(64 * part) * 2;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v = live ? *reinterpret_cast<const uint4*>(src + 16 * i) : make_uint4(0, 0, 0, 0);
            hot |= big(v.x) || big(v.y) || big(v.z) || big(v.w);
            r[4 * i] = dev::bf16x2_to_f16x2(v.x, down);
            r[4 * i + 1] = dev::bf16x2_to_f16x2(v.y, down);
            r[4 * i + 2] = dev::bf16x2_to_f16x2(v.z, down);
            r[4 * i + 3] = dev::bf16x2_to_f16x2(v.w, down);
          }
          __syncwarp();
          tc::tmem_st32<false>(tl + TM_Q + 32 * part, r);   // the next part's loads may go first
        }
#pragma unroll
        for (int i = 0; i < 8 * kQSmemAtoms; ++i) {     // positions 384..575 -> 64-dim atoms, row h
          const uint4 v = live ? *reinterpret_cast<const uint4*>(qrow + (perm(kQTmemDims + 64 * (i >> 3)) + 8 * (i & 7)) * 2)
                               : make_uint4(0, 0, 0, 0);
          hot |= big(v.x) || big(v.y) || big(v.z) || big(v.w);
          sts128_relaxed(qs + (i >> 3) * kQAtom + tc::sw128_offset(h, i & 7),
                         make_uint4(dev::bf16x2_to_f16x2(v.x, down), dev::bf16x2_to_f16x2(v.y, down),
                                    dev::bf16x2_to_f16x2(v.z, down), dev::bf16x2_to_f16x2(v.w, down)));
        }
        if (attempt == 1 || !__any_sync(0xffffffffu, hot)) break;
        if (hot) {                                      // this row: its largest |q|
          uint32_t mx = 0;
          for (int i = 0; i < kLatent * 2 / 16; ++i) {
            const uint4 v = *reinterpret_cast<const uint4*>(qrow + 16 * i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
          }
          int sh = 0;
          if (mx < 0x7F80u) sh = max(-100, min(113, static_cast<int>(mx >> 7) - 127 - 14));
          down = __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
          q_scale = a.scale_log2 * __uint_as_float(static_cast<uint32_t>(127 + sh) << 23);
        }
      }
      tc::tmem_wait_st();
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(sy.bar(B_Q_READY));
      // thread 0 sees every phase of Q_READY in turn (all 128 rows written) and publishes the count
      bool ok = true;
      if (h == 0) {
        ok = sy.wait(B_Q_READY, nq & 1, false, 16);
        if (ok) tc::st_release_u32(qver, static_cast<uint32_t>(nq + 1));
      }
      if (!__all_sync(0xffffffffu, ok)) return;
      ++nq;
      cur_req = seg.req;
    }
    if (cur.j == 0) { m_used = -INFINITY; l = 0.0f; }
    const int valid = page_ok(a, pg) ? cur.valid() : 0;
    Cursor nx = cur;                 // the next page's table entries load while this page runs
    nx.next(a);
    const int64_t npg = nx.done() ? 0 : nx.page(a);
    const int nv = min(max(valid - kHalf * c, 0), kHalf);
    const bool last = cur.j == seg.num_pages - 1;
    const int s = g & 1;

    // ---- logits of the own tokens (buffer s; refilled for page g + 2 only after S_FREE(s)) ----
    if (!wait(B_S_FULL + s, (g >> 1) & 1, false, 128)) return;
    if (KV == KV_FP8PT) {
      __syncwarp();
      sgp[h & 31] = sg_lane;
      __syncwarp();
      sg_lane = token_scale(nx, npg);
    }
    tc::tc_fence_after();
    uint32_t sr[32];
    tc::tmem_ld32(tl + TM_S + kHalf * s, sr);
    tc::tmem_wait_ld();
    tc::tc_fence_before();
    tc::mbar_arrive(sy.bar(B_S_FREE + s));
    float x[32], mx8[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
    if (KV == KV_FP8PT) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 sg4 = reinterpret_cast<const float4*>(sgp)[u];
        sr[4 * u] = __float_as_uint(__uint_as_float(sr[4 * u]) * sg4.x);
        sr[4 * u + 1] = __float_as_uint(__uint_as_float(sr[4 * u + 1]) * sg4.y);
        sr[4 * u + 2] = __float_as_uint(__uint_as_float(sr[4 * u + 2]) * sg4.z);
        sr[4 * u + 3] = __float_as_uint(__uint_as_float(sr[4 * u + 3]) * sg4.w);
      }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      x[i] = i < nv ? __uint_as_float(sr[i]) : -INFINITY;
      mx8[i & 7] = fmaxf(mx8[i & 7], x[i]);
    }
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
      for (int u = 0; u < w; ++u) mx8[u] = fmaxf(mx8[u], mx8[u + w]);
    const float r_own = mx8[0];

    // ---- trade row maxima: both CTAs take the same maximum and make the same rescale decision ----
    tc::st_async_f32(rm + s * 512 + 4 * h, r_own, sy.bar(B_RM_FULL + s), peer);
    if (h == 0) tc::mbar_arrive_expect_tx(sy.bar(B_RM_FULL + s), 512);
    // p = 2^(x * scale - m): one FMA and one exp2 per logit. While the peer's maximum is in flight,
    // compute P against the current running maximum; when the agreed maximum keeps it (no rescale,
    // almost every page after a segment's first), these are exactly the values computed after the wait.
    uint32_t pk[16];
    float lsum = 0.0f;
    auto exp_row = [&](float mref) {
      float l4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = dev::fast_exp2(fmaf(x[2 * i], q_scale, -mref));
        const float p1 = dev::fast_exp2(fmaf(x[2 * i + 1], q_scale, -mref));
        l4[i & 3] += p0 + p1;
        if (KV == KV_FP8PT) {
          const float2 sg2 = reinterpret_cast<const float2*>(sgp)[i];
          pk[i] = dev::pack_f16x2(p0 * sg2.x, p1 * sg2.y);
        } else {
          pk[i] = dev::pack_f16x2(p0, p1);
        }
      }
      lsum = (l4[0] + l4[1]) + (l4[2] + l4[3]);
    };
    const bool spec = m_used != -INFINITY && !(r_own * q_scale > m_used + 8.0f);
    if (spec) exp_row(m_used);
    // own half of P goes to the local buffer s, then one bulk copy into the peer's buffer. P_FREE(s)
    // counts the P.V of page g - 2 in both CTAs (both read this buffer pair). The speculative row is
    // stored while the peer's maximum is still in flight and rewritten below if it does not hold.
    if (g >= 2 && !wait(B_P_FREE + s, ((g >> 1) - 1) & 1, false, 1024)) return;
    const uint32_t prow = pbuf + s * kPBytes + c * kPHalf;
    auto store_row = [&]() {
#pragma unroll
      for (int u = 0; u < 4; ++u) sts128(prow + tc::sw64_offset(h, u), make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]));
    };
    if (spec) store_row();
    if (!wait(B_RM_FULL + s, (g >> 1) & 1, true, 256)) return;
    const float r_peer = tc::lds_f32(rm + s * 512 + 4 * h);
    const float rmax = fmaxf(r_own, r_peer) * q_scale;
    const bool renew = rmax > -INFINITY && (m_used == -INFINITY || rmax > m_used + 8.0f);
    const float alpha = renew ? dev::fast_exp2(m_used - rmax) : 1.0f;   // 0 when m_used is -inf
    // O holds earlier pages of this segment scaled to the old maximum: rescale the rows that renew
    // (the whole warp takes part in the TMEM traffic) once PV(g - 1) has completed
    const bool rescale_row = renew && cur.j > 0 && m_used != -INFINITY;
    if (__any_sync(0xffffffffu, rescale_row)) {
      if (!wait(B_O_DONE + ((g - 1) & 1), ((g - 1) >> 1) & 1, false, 512)) return;
      tc::tc_fence_after();
      const float f = rescale_row ? alpha : 1.0f;
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        uint32_t orow[32];
        tc::tmem_ld32(tl + TM_O + 32 * cc, orow);
        tc::tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 32; ++u) orow[u] = __float_as_uint(__uint_as_float(orow[u]) * f);
        tc::tmem_st32(tl + TM_O + 32 * cc, orow);
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
    }
    if (renew) {
      l *= alpha;
      m_used = rmax;
    }
    if (!spec || renew) {
      exp_row(m_used == -INFINITY ? 0.0f : m_used);
      store_row();
    }
    l += lsum;
    // each warp hands its own 32 rows (2 KB, contiguous in the 64-byte swizzle) to the peer as soon as
    // they are written: no CTA-wide wait before the copies. P_FULL(s) completes with the four local
    // warps' arrivals and the peer's four 2 KB copies.
    tc::fence_proxy_async_smem();
    __syncwarp();
    if ((h & 31) == 0) {
      const uint32_t wrows = pbuf + s * kPBytes + c * kPHalf + (h >> 5) * (kPHalf / 4);
      tc::bulk_copy_to_peer(wrows, wrows, kPHalf / 4, sy.bar(B_P_FULL + s), peer);
      tc::mbar_arrive_expect_tx(sy.bar(B_P_FULL + s), kPHalf / 4);
    }
    cur = nx;
    pg = npg;
    if (!last) continue;

    // ---- segment end: trade row sums (fixed order of the two terms), then O / l for this CTA's
    // 256 output dims once PV(g) has completed ----
    tc::st_async_f32(lx + s * 512 + 4 * h, l, sy.bar(B_LX_FULL + s), peer);
    if (h == 0) tc::mbar_arrive_expect_tx(sy.bar(B_LX_FULL + s), 512);
    if (!wait(B_LX_FULL + s, lx_count[s] & 1, true, 4096)) return;
    ++lx_count[s];
    const float l_peer = tc::lds_f32(lx + s * 512 + 4 * h);
    const float lt = c == 0 ? l + l_peer : l_peer + l;
    if (!wait(B_O_DONE + s, (g >> 1) & 1, false, 2048)) return;
    tc::tc_fence_after();
    const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
    const float lse2 = lt > 0.0f ? m_used + __log2f(lt) : -INFINITY;
    const int64_t row = static_cast<int64_t>(seg.req) * a.heads + h;
#pragma unroll 1
    for (int cc = 0; cc < 8; ++cc) {
      uint32_t orow[32];
      tc::tmem_ld32(tl + TM_O + 32 * cc, orow);
      tc::tmem_wait_ld();
      if (h >= a.heads) continue;            // a padding row (the TMEM load above is warp-wide)
      if (seg.partial < 0) {
        const float sc = inv * a.out_scale;
        uint4* dst = reinterpret_cast<uint4*>(a.out + row * kDv + 256 * c + 32 * cc);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          dst[u] = make_uint4(dev::pack_bf16x2(__uint_as_float(orow[8 * u]) * sc, __uint_as_float(orow[8 * u + 1]) * sc),
                              dev::pack_bf16x2(__uint_as_float(orow[8 * u + 2]) * sc, __uint_as_float(orow[8 * u + 3]) * sc),
                              dev::pack_bf16x2(__uint_as_float(orow[8 * u + 4]) * sc, __uint_as_float(orow[8 * u + 5]) * sc),
                              dev::pack_bf16x2(__uint_as_float(orow[8 * u + 6]) * sc, __uint_as_float(orow[8 * u + 7]) * sc));
      } else {
        float4* dst = reinterpret_cast<float4*>(a.part_o + (static_cast<int64_t>(seg.partial) * a.heads + h) * kDv + 256 * c + 32 * cc);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          dst[u] = make_float4(__uint_as_float(orow[4 * u]) * inv, __uint_as_float(orow[4 * u + 1]) * inv,
                               __uint_as_float(orow[4 * u + 2]) * inv, __uint_as_float(orow[4 * u + 3]) * inv);
      }
    }
    tc::tc_fence_before();
    if (c == 0 && h < a.heads) {
      if (seg.partial < 0) { if (a.lse) a.lse[row] = lse2 * 0.69314718055994531f; }
      else a.part_lse[static_cast<int64_t>(seg.partial) * a.heads + h] = lse2;
    }
  }
}

template <int KV>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) decode_tc_kernel(const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int c = static_cast<int>(tc::cluster_ctarank());
  const int worker = blockIdx.x >> 1;
  const int seg_b = a.worker_ptr[worker], seg_e = a.worker_ptr[worker + 1];
  Sync sy;
  sy.bars = base + OFF_BAR;
  sy.abort = reinterpret_cast<volatile int*>(sbase + OFF_ABORT);
  sy.status = a.status;

  if (tid == 0) {
    for (int i = 0; i < kKSlots; ++i) { tc::mbar_init(sy.bar(B_K_FULL + i), kDQ); tc::mbar_init(sy.bar(B_K_EMPTY + i), 1); }
    for (int i = 0; i < kVSlots; ++i) { tc::mbar_init(sy.bar(B_V_FULL + i), kDQ); tc::mbar_init(sy.bar(B_V_EMPTY + i), 1); }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(sy.bar(B_S_FULL + i), 1);
      tc::mbar_init(sy.bar(B_S_FREE + i), 128);
      tc::mbar_init(sy.bar(B_P_LOCAL + i), 128);
      tc::mbar_init(sy.bar(B_P_FULL + i), 4);        // one per softmax warp, plus the peer's 8 KB of P in bytes
      tc::mbar_init(sy.bar(B_P_FREE + i), 2);        // P.V of the page in both CTAs
      tc::mbar_init(sy.bar(B_O_DONE + i), 1);
      tc::mbar_init(sy.bar(B_RM_FULL + i), 1);       // plus the peer's 128 x 4 bytes, counted in bytes
      tc::mbar_init(sy.bar(B_LX_FULL + i), 1);
    }
    tc::mbar_init(sy.bar(B_Q_READY), 128);
    tc::mbar_init(sy.bar(B_FINAL), 3);             // one commit per MMA-issuing thread
    *sy.abort = 0;
    *reinterpret_cast<volatile uint32_t*>(sbase + OFF_QVER) = 0;
    tc::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(base + OFF_TSLOT, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();          // the peer's barriers are initialised before any remote arrive
  tc::tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(sbase + OFF_TSLOT);

  if (warp < 4) {
    role_softmax<KV>(a, sy, seg_b, seg_e, c, tid, tbase, base + OFF_P, base + OFF_Q, base + OFF_RM, base + OFF_LX,
                     base + OFF_QVER, reinterpret_cast<float*>(sbase + OFF_SIG));
  } else if (warp < kQkWarpOdd) {
    role_dequant<KV>(a, sy, seg_b, seg_e, c, tid - 128, base + OFF_K, base + OFF_V, base + OFF_SIG);
  } else if (warp == kPvWarp) {
    if ((tid & 31) == 0) role_pv(a, sy, seg_b, seg_e, c, tbase, base + OFF_V, base + OFF_P);
  } else if ((tid & 31) == 0) {
    role_qk(a, sy, seg_b, seg_e, c, warp == kQkWarpOdd ? 1 : 0, tbase, base + OFF_K, base + OFF_V, base + OFF_Q,
            base + OFF_QVER);
  }
  // every MMA of the three issuing threads has completed before TMEM is released
  if (warp >= kQkWarpOdd && (tid & 31) == 0) sy.wait(B_FINAL, 0, false, 64);
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tbase, 512);
  }
  // After a timeout a bulk copy into the peer may still be in flight: give it time to land before
  // either CTA of the pair releases its shared memory. Normal runs consume every copy they issue.
  if (tid == 0) {
    const int peer_abort = tc::ld_cluster_u32(tc::mapa(base + OFF_ABORT, static_cast<uint32_t>(c ^ 1)));
    if (*sy.abort || peer_abort) {
      const long long t0 = clock64();
      while (clock64() - t0 < 200000) {}
    }
  }
  tc::cluster_sync();          // no CTA leaves while its peer may still touch its shared memory
}

template <int KV>
cudaError_t launch_kv(const DecodeArgs& a, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  decode_tc_kernel<KV><<<static_cast<unsigned>(a.num_workers * 2), kThreads, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int tc_max_active_clusters() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaFuncSetAttribute(decode_tc_kernel<KV_FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return -1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<KV_FP8>, &cfg) != cudaSuccess) return -1;
  return n;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  if (a.num_segments == 0) return cudaSuccess;
  if (a.heads < 16 || a.heads > 128 || a.heads % 16 || a.ctas_per_worker != 2) return cudaErrorInvalidValue;
  switch (a.kv_dtype) {
    case KV_FP8: return launch_kv<KV_FP8>(a, s);
    case KV_NVFP4: return launch_kv<KV_NVFP4>(a, s);
    case KV_BF16: return launch_kv<KV_BF16>(a, s);
    case KV_FP8PT: return launch_kv<KV_FP8PT>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qkvp
