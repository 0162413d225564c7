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
// work item runs on a pair of CTAs (a cluster of two). CTA c owns latent dims [256c, 256c + 256) of
// the 512 "nope" dims and [512 + 32c, 512 + 32c + 32) of the rope dims: it computes the partial
// logits over its 288 dims, trades them with its peer through distributed shared memory, and both
// CTAs add the two partials in the same order, so they hold bit-identical logits, maxima and
// probabilities. Each then accumulates its own 256 output dims. Dequantization is never duplicated.
//
// Per CTA (256 threads, two warps per SM sub-partition):
//   warps 0-3 (softmax): thread h owns head h = TMEM lane h. Loads Q once per request (the nope half
//     into TMEM as the A operand of Q.K^T, the rope half into shared memory), then per page: reads
//     its 64 partial logits from TMEM, exchanges them, runs the FP32 online softmax (base 2, with a
//     lazy rescale of O when the running maximum grows by more than 2^8), and writes its row of
//     P (FP16) to shared memory. At the end of a segment it reads O from TMEM and writes the output.
//   warps 4-6 (dequant): per page, load this CTA's half of the raw page from global memory (the next
//     page's loads are in flight while the current one is converted), convert to FP16 and write the
//     swizzled operand tile (three tiles in a ring).
//   warp 7 (MMA): one thread issues S = Q.K^T (M 128 heads x N 64 tokens x K 288) into one of two
//     TMEM logit buffers and O += P.V (M 128 x N 256 x K 64) into the TMEM accumulator; tcgen05.commit
//     signals the other roles through mbarriers.
// TMEM: O [0, 256), Q nope [256, 384), logits [384, 448) and [448, 512).
// Barrier phases: every barrier is waited on by parity, which is only sound while the barrier is at
// most one phase away from the phase waited for. Buffers indexed by the global page counter g keep
// that true; the PV-completion barrier is split by the parity of g because the softmax warps wait on
// it only now and then (lazy rescales, segment ends), and QK(g) completing implies PV(g - 2) has.
// Every wait is bounded; a timeout sets bits in the status word and the CTA drains and exits.
#include <cstdint>

#include "qkvp_device.cuh"
#include "qkvp_internal.h"
#include "tc_ptx.cuh"

namespace qkvp {
namespace {

constexpr int kThreads = 256;
constexpr int kDQ = 96;                     // dequant threads (warps 4-6)
constexpr int kTiles = 3;
constexpr uint32_t kTileBytes = 36864;      // nope 64 tokens x 256 dims (32 KB) + rope 64 x 32 (4 KB)
constexpr uint32_t kRopeOff = 32768;
constexpr uint32_t kPBytes = 16384;         // 128 heads x 64 tokens FP16
constexpr uint32_t kQRBytes = 8192;         // 128 heads x 32 rope dims FP16
constexpr uint32_t kXBytes = 32768;         // 128 heads x 64 FP32 logits, [16-byte chunk][head]

constexpr uint32_t OFF_TILE = 0;
constexpr uint32_t OFF_P = OFF_TILE + kTiles * kTileBytes;
constexpr uint32_t OFF_QR = OFF_P + 2 * kPBytes;
constexpr uint32_t OFF_X = OFF_QR + kQRBytes;
constexpr uint32_t OFF_BAR = OFF_X + 2 * kXBytes;
enum : uint32_t {
  B_TILE_FULL = 0, B_TILE_EMPTY = 3, B_S_FULL = 6, B_S_FREE = 8, B_P_FULL = 10, B_P_FREE = 12,
  B_X_FULL = 14, B_O_DONE = 16, B_Q_READY = 18, B_FINAL = 19, B_X_FREE = 20, NUM_BARS = 22
};
constexpr uint32_t OFF_TSLOT = OFF_BAR + 8 * NUM_BARS;
constexpr uint32_t OFF_QMAX = OFF_TSLOT + 4;
constexpr uint32_t OFF_ABORT = OFF_QMAX + 4;
constexpr uint32_t kSmemUsed = OFF_ABORT + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;   // slack to align the base to 1024 bytes

constexpr uint32_t TM_O = 0, TM_QN = 256, TM_S = 384;

constexpr uint32_t kIdescQK = tc::idesc_f16(128, 64, 0, 0);
constexpr uint32_t kIdescPV = tc::idesc_f16(128, 256, 0, 1);

// Walks a worker's (segment, page) sequence.
struct Cursor {
  int si, se, j;
  Segment seg;
  __device__ void begin(const DecodeArgs& a, int s0, int s1) {
    si = s0; se = s1; j = 0;
    if (si < se) seg = a.segs[si];
  }
  __device__ bool done() const { return si >= se; }
  __device__ void next(const DecodeArgs& a) {
    if (++j >= seg.num_pages) { j = 0; if (++si < se) seg = a.segs[si]; }
  }
  __device__ int valid() const { return min(kPage, seg.num_tokens - j * kPage); }
  __device__ int64_t page(const DecodeArgs& a) const { return a.kv_indices[seg.page_begin + j]; }
};

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

// ---- dequantization of one page half into an operand tile --------------------------------------
// Tile layout: nope dims [256c, 256c + 256) as 4 atoms of 64 dims (8 KB each, 128-byte swizzle,
// rows = tokens); rope dims [512 + 32c, +32) as one 64-byte-swizzle region (rows = tokens).
template <int KV> struct Dequant;

template <> struct Dequant<KV_FP8> {
  static constexpr int kIters = 12;         // 64 tokens x 18 chunks of 16 bytes / 96 threads
  struct Raw { uint4 v[kIters]; };
  __device__ static void load(Raw& r, const DecodeArgs& a, int64_t page, int valid, int c, int t) {
    const uint8_t* base = a.kv + page * (kPage * kLatent);
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + kDQ * i, tok = q / 18, k = q % 18;
      if (tok < valid) r.v[i] = ldg_nc(base + tok * kLatent + (k < 16 ? 256 * c + 16 * k : 512 + 32 * c + 16 * (k - 16)));
    }
  }
  __device__ static void store(const Raw& r, const DecodeArgs&, int64_t, int valid, int, int t, uint32_t tile) {
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + kDQ * i, tok = q / 18, k = q % 18;
      uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
      if (tok < valid) {
        const uint4 v = r.v[i];
        lo = make_uint4(dev::e4m3x2_to_f16x2(v.x & 0xFFFF), dev::e4m3x2_to_f16x2(v.x >> 16),
                        dev::e4m3x2_to_f16x2(v.y & 0xFFFF), dev::e4m3x2_to_f16x2(v.y >> 16));
        hi = make_uint4(dev::e4m3x2_to_f16x2(v.z & 0xFFFF), dev::e4m3x2_to_f16x2(v.z >> 16),
                        dev::e4m3x2_to_f16x2(v.w & 0xFFFF), dev::e4m3x2_to_f16x2(v.w >> 16));
      }
      if (k < 16) {
        const uint32_t at = tile + (k >> 2) * 8192, ch = (k & 3) * 2;
        sts128(at + tc::sw128_offset(tok, ch), lo);
        sts128(at + tc::sw128_offset(tok, ch + 1), hi);
      } else {
        const uint32_t ch = (k - 16) * 2;
        sts128(tile + kRopeOff + tc::sw64_offset(tok, ch), lo);
        sts128(tile + kRopeOff + tc::sw64_offset(tok, ch + 1), hi);
      }
    }
  }
};

template <> struct Dequant<KV_NVFP4> {
  static constexpr int kIters = 6;          // 64 tokens x 9 chunks (8 nope + 1 rope) = 576 / 96
  struct Raw { uint4 v[kIters]; uint32_t s[kIters]; };
  __device__ static void load(Raw& r, const DecodeArgs& a, int64_t page, int valid, int c, int t) {
    const uint8_t* base = a.kv + page * (kPage * kPacked);
    const uint8_t* sbase = a.kv_scale + page * (kPage * kScales);
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + kDQ * i, tok = q / 9, k = q % 9;
      if (tok < valid) {
        r.v[i] = ldg_nc(base + tok * kPacked + (k < 8 ? 128 * c + 16 * k : 256 + 16 * c));
        r.s[i] = *reinterpret_cast<const uint16_t*>(sbase + tok * kScales + (k < 8 ? 16 * c + 2 * k : 32 + 2 * c));
      }
    }
  }
  __device__ static void store(const Raw& r, const DecodeArgs&, int64_t, int valid, int, int t, uint32_t tile) {
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int q = t + kDQ * i, tok = q / 9, k = q % 9;
      uint32_t o[16];
      if (tok < valid) {
        const uint32_t sa = r.s[i] & 0xFFu, sb = (r.s[i] >> 8) & 0xFFu;
        const uint32_t ha = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(sa | (sa << 8)));
        const uint32_t hb = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(sb | (sb << 8)));
        const uint32_t w[4] = {r.v[i].x, r.v[i].y, r.v[i].z, r.v[i].w};
#pragma unroll
        for (int b = 0; b < 16; ++b) o[b] = dev::nvfp4x2_to_f16x2((w[b >> 2] >> (8 * (b & 3))) & 0xFFu, b < 8 ? ha : hb);
      } else {
#pragma unroll
        for (int b = 0; b < 16; ++b) o[b] = 0;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 v = make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
        if (k < 8) sts128(tile + (k >> 1) * 8192 + tc::sw128_offset(tok, (k & 1) * 4 + u), v);
        else sts128(tile + kRopeOff + tc::sw64_offset(tok, u), v);
      }
    }
  }
};

template <> struct Dequant<KV_BF16> {      // the cast-then-attend baseline: BF16 pages
  struct Raw {};
  __device__ static void load(Raw&, const DecodeArgs&, int64_t, int, int, int) {}
  __device__ static void store(const Raw&, const DecodeArgs& a, int64_t page, int valid, int c, int t, uint32_t tile) {
    const uint8_t* base = a.kv + page * (kPage * kLatent * 2);
    // 64 tokens x 36 chunks of 8 BF16 (32 nope + 4 rope) = 2304 chunks / 96 threads, in two halves
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      uint4 v[12];
#pragma unroll
      for (int i = 0; i < 12; ++i) {
        const int q = t + kDQ * (12 * h2 + i), tok = q / 36, k = q % 36;
        if (tok < valid) v[i] = ldg_nc(base + tok * kLatent * 2 + (k < 32 ? (256 * c + 8 * k) : (512 + 32 * c + 8 * (k - 32))) * 2);
      }
#pragma unroll
      for (int i = 0; i < 12; ++i) {
        const int q = t + kDQ * (12 * h2 + i), tok = q / 36, k = q % 36;
        uint4 o = make_uint4(0, 0, 0, 0);
        if (tok < valid) o = make_uint4(dev::bf16x2_to_f16x2(v[i].x), dev::bf16x2_to_f16x2(v[i].y),
                                        dev::bf16x2_to_f16x2(v[i].z), dev::bf16x2_to_f16x2(v[i].w));
        if (k < 32) sts128(tile + (k >> 3) * 8192 + tc::sw128_offset(tok, k & 7), o);
        else sts128(tile + kRopeOff + tc::sw64_offset(tok, k - 32), o);
      }
    }
  }
};

__device__ __forceinline__ bool page_ok(const DecodeArgs& a, int64_t page) { return page >= 0 && page < a.num_pages; }

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

struct Sync {
  uint32_t bars;
  volatile int* abort;
  int* status;
  __device__ uint32_t bar(uint32_t i) const { return bars + 8 * i; }
  __device__ bool wait(uint32_t i, uint32_t parity, bool cluster = false, int code = 1) const {
    const uint32_t b = bar(i);
    if (cluster ? tc::mbar_try_wait_cluster(b, parity) : tc::mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    for (int n = 0;; ++n) {
      if (cluster ? tc::mbar_try_wait_cluster(b, parity) : tc::mbar_try_wait(b, parity)) return true;
      if ((n & 255) == 0) {
        if (*abort) return false;
        if (clock64() - t0 > (1ll << 31)) {
          *abort = 1;
          atomicOr(status, code);
          return false;
        }
      }
    }
  }
};

// ---- roles -------------------------------------------------------------------------------------------
template <int KV>
__device__ void role_dequant(const DecodeArgs& a, const Sync& sy, int seg_b, int seg_e, int c, int t, uint32_t tiles) {
  using D = Dequant<KV>;
  Cursor cur;
  cur.begin(a, seg_b, seg_e);
  typename D::Raw raw_cur, raw_nxt;
  if (cur.done()) return;
  int64_t pg = cur.page(a);
  int valid = page_ok(a, pg) ? cur.valid() : 0;
  D::load(raw_cur, a, pg, valid, c, t);
  for (int g = 0; !cur.done(); ++g) {
    Cursor nx = cur;
    nx.next(a);
    int64_t npg = 0;
    int nvalid = 0;
    if (!nx.done()) {
      npg = nx.page(a);
      nvalid = page_ok(a, npg) ? nx.valid() : 0;
      D::load(raw_nxt, a, npg, nvalid, c, t);
    }
    const int buf = g % kTiles;
    if (g >= kTiles && !sy.wait(B_TILE_EMPTY + buf, ((g / kTiles) - 1) & 1, false, 2)) return;
    D::store(raw_cur, a, pg, valid, c, t, tiles + buf * kTileBytes);
    tc::fence_proxy_async_smem();
    tc::mbar_arrive(sy.bar(B_TILE_FULL + buf));
    raw_cur = raw_nxt;
    cur = nx;
    pg = npg;
    valid = nvalid;
  }
}

// MMA role (one thread). QK^T of page g and P.V of page g are issued in page order, each as soon as
// its inputs are ready: QK(g) needs its operand tile, a free logit buffer (page g - 2 read out) and,
// at a new request, the new Q; PV(g) needs P(g). Issuing whichever is ready keeps QK running ahead
// while the softmax works, and cannot deadlock at segment boundaries.
__device__ void role_mma(const DecodeArgs& a, const Sync& sy, int seg_b, int seg_e, uint32_t tbase, uint32_t tiles,
                         uint32_t pbuf, uint32_t qr) {
  int total = 0;
  for (int si = seg_b; si < seg_e; ++si) total += a.segs[si].num_pages;
  Cursor cq, cp;
  cq.begin(a, seg_b, seg_e);
  cp.begin(a, seg_b, seg_e);
  int gq = 0, gp = 0, qcount = 0, q_req = -1;
  long long t_last = clock64();
  while (gp < total) {
    bool did = false;
    if (gp < gq && mbar_test(sy.bar(B_P_FULL + (gp & 1)), (gp >> 1) & 1)) {
      tc::tc_fence_after();
      const int s = gp & 1, buf = gp % kTiles;
      const uint32_t pa = pbuf + s * kPBytes, tv = tiles + buf * kTileBytes;
      const bool first = cp.j == 0;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = tc::smem_desc(pa + 32 * kk, 16, 1024, tc::kSwizzle128);
        const uint64_t bd = tc::smem_desc(tv + 2048 * kk, 8192, 1024, tc::kSwizzle128);
        tc::mma_ss(tbase + TM_O, ad, bd, kIdescPV, (first && kk == 0) ? 0u : 1u);
      }
      tc::mma_commit(sy.bar(B_TILE_EMPTY + buf));
      tc::mma_commit(sy.bar(B_P_FREE + s));
      tc::mma_commit(sy.bar(B_O_DONE + s));
      cp.next(a);
      ++gp;
      did = true;
    } else if (gq < total) {
      const bool newq = cq.j == 0 && cq.seg.req != q_req;
      const int buf = gq % kTiles, s = gq & 1;
      if (mbar_test(sy.bar(B_TILE_FULL + buf), (gq / kTiles) & 1) &&
          (gq < 2 || mbar_test(sy.bar(B_S_FREE + s), ((gq >> 1) - 1) & 1)) &&
          (!newq || mbar_test(sy.bar(B_Q_READY), qcount & 1))) {
        tc::tc_fence_after();
        const uint32_t td = tbase + TM_S + 64 * s, tk = tiles + buf * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const uint64_t bd = tc::smem_desc(tk + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, tc::kSwizzle128);
          tc::mma_ts(td, tbase + TM_QN + 8 * ks, bd, kIdescQK, ks > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const uint64_t ad = tc::smem_desc(qr + 32 * ks, 16, 512, tc::kSwizzle64);
          const uint64_t bd = tc::smem_desc(tk + kRopeOff + 32 * ks, 16, 512, tc::kSwizzle64);
          tc::mma_ss(td, ad, bd, kIdescQK, 1u);
        }
        tc::mma_commit(sy.bar(B_S_FULL + s));
        if (newq) { q_req = cq.seg.req; ++qcount; }
        cq.next(a);
        ++gq;
        did = true;
      }
    }
    if (did) {
      t_last = clock64();
    } else if (((clock64() - t_last) & 0xFF) == 0 || clock64() - t_last > (1ll << 31)) {
      if (*sy.abort) break;
      if (clock64() - t_last > (1ll << 31)) {
        *sy.abort = 1;
        atomicOr(sy.status, 4);
        break;
      }
    }
  }
  // drain: every MMA issued so far has completed before TMEM is released
  tc::mma_commit(sy.bar(B_FINAL));
  sy.wait(B_FINAL, 0, false, 64);
}

// Softmax role, software-pipelined over pages: at page g it reads its partial logits S(g) from TMEM
// and stores them straight into the peer's exchange buffer (stage 1), then finishes page g - 1
// (stage 2): waits for the peer's partial of g - 1, adds the two in a fixed order, runs the online
// softmax and writes P(g - 1). The remote stores of page g drain while stage 2 computes: the arrive
// that frees the peer's buffer is relaxed (the values it guards have been used), and the
// release-arrive that publishes page g comes last. Buffers are [16-byte chunk][head], so a warp's
// remote store covers 512 contiguous bytes. Every wait is followed by a warp vote, so the warps stay
// converged for the warp-collective tcgen05.ld / tcgen05.st and continue or give up as a whole.
struct PendingPage {
  int g, valid, j, last, partial, req;
  float q_scale;
};

template <int KV>
__device__ void role_softmax(const DecodeArgs& a, const Sync& sy, int seg_b, int seg_e, int c, int h,
                             uint32_t tbase, uint32_t pbuf, uint32_t qr, uint32_t xbuf) {
  const uint32_t peer = c ^ 1u;
  const uint32_t tl = tbase + (static_cast<uint32_t>(h & ~31) << 16);   // this warp's TMEM lane quarter
  auto wait = [&](uint32_t bar, uint32_t parity, bool cluster, int code) -> bool {
    const bool ok = sy.wait(bar, parity, cluster, code);
    return __all_sync(0xffffffffu, ok);
  };
  float m_used = -INFINITY, l = 0.0f;          // running softmax state of the segment in stage 2

  // stage 2: finish page pp (own partial logits in `own`, the peer's in the local exchange buffer)
  auto finish = [&](const PendingPage& pp, const uint32_t (&own)[64]) -> bool {
    const int b = pp.g, s = b & 1;
    if (pp.j == 0) { m_used = -INFINITY; l = 0.0f; }
    if (!wait(B_X_FULL + s, (b >> 1) & 1, true, 256)) return false;
    const uint32_t xb = xbuf + s * kXBytes + h * 16;
    float x[64];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint4 pv = lds128(xb + i * 2048);
      const uint32_t p4[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float mine = __uint_as_float(own[4 * i + u]), theirs = __uint_as_float(p4[u]);
        x[4 * i + u] = c == 0 ? (mine + theirs) : (theirs + mine);
      }
    }
    tc::mbar_arrive_cluster_relaxed(sy.bar(B_X_FREE + s), peer);   // the peer may refill this buffer
    // row maximum of the raw logit sums (the scale is positive), as a tree for ILP
    float mx8[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      if (i >= pp.valid) x[i] = -INFINITY;
      mx8[i & 7] = fmaxf(mx8[i & 7], x[i]);
    }
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
      for (int u = 0; u < w; ++u) mx8[u] = fmaxf(mx8[u], mx8[u + w]);
    const float rmax = mx8[0] * pp.q_scale;
    const bool renew = rmax > -INFINITY && (m_used == -INFINITY || rmax > m_used + 8.0f);
    const float alpha = renew ? dev::fast_exp2(m_used - rmax) : 1.0f;   // 0 when m_used is -inf
    // O holds earlier pages of this segment scaled to the old maximum: rescale the rows that renew
    // (the whole warp takes part in the TMEM traffic) once PV(b - 1) has completed
    const bool rescale_row = renew && pp.j > 0 && m_used != -INFINITY;
    if (__any_sync(0xffffffffu, rescale_row)) {
      if (!wait(B_O_DONE + ((b - 1) & 1), ((b - 1) >> 1) & 1, false, 512)) return false;
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
    const float mref = m_used == -INFINITY ? 0.0f : m_used;
    uint32_t pk[32];
    float l4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 32; ++i) {   // p = 2^(x * scale - m): one FMA and one exp2 per logit
      const float p0 = dev::fast_exp2(fmaf(x[2 * i], pp.q_scale, -mref));
      const float p1 = dev::fast_exp2(fmaf(x[2 * i + 1], pp.q_scale, -mref));
      l4[i & 3] += p0 + p1;
      pk[i] = dev::pack_f16x2(p0, p1);
    }
    l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
    if (b >= 2 && !wait(B_P_FREE + s, ((b >> 1) - 1) & 1, false, 1024)) return false;
    const uint32_t prow = pbuf + s * kPBytes;
#pragma unroll
    for (int i = 0; i < 8; ++i) sts128(prow + tc::sw128_offset(h, i), make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]));
    tc::fence_proxy_async_smem();
    tc::mbar_arrive(sy.bar(B_P_FULL + s));
    if (!pp.last) return true;
    // ---- segment epilogue: O / l for this CTA's 256 output dims ----
    if (!wait(B_O_DONE + s, (b >> 1) & 1, false, 2048)) return false;
    tc::tc_fence_after();
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    const float lse2 = l > 0.0f ? m_used + __log2f(l) : -INFINITY;
    const int64_t row = static_cast<int64_t>(pp.req) * a.heads + h;
#pragma unroll 1
    for (int cc = 0; cc < 8; ++cc) {
      uint32_t orow[32];
      tc::tmem_ld32(tl + TM_O + 32 * cc, orow);
      tc::tmem_wait_ld();
      if (pp.partial < 0) {
        const float sc = inv * a.out_scale;
        uint4* dst = reinterpret_cast<uint4*>(a.out + row * kDv + 256 * c + 32 * cc);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          dst[u] = make_uint4(dev::pack_bf16x2(__uint_as_float(orow[8 * u]) * sc, __uint_as_float(orow[8 * u + 1]) * sc),
                              dev::pack_bf16x2(__uint_as_float(orow[8 * u + 2]) * sc, __uint_as_float(orow[8 * u + 3]) * sc),
                              dev::pack_bf16x2(__uint_as_float(orow[8 * u + 4]) * sc, __uint_as_float(orow[8 * u + 5]) * sc),
                              dev::pack_bf16x2(__uint_as_float(orow[8 * u + 6]) * sc, __uint_as_float(orow[8 * u + 7]) * sc));
      } else {
        float4* dst = reinterpret_cast<float4*>(a.part_o + (static_cast<int64_t>(pp.partial) * a.heads + h) * kDv + 256 * c + 32 * cc);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          dst[u] = make_float4(__uint_as_float(orow[4 * u]) * inv, __uint_as_float(orow[4 * u + 1]) * inv,
                               __uint_as_float(orow[4 * u + 2]) * inv, __uint_as_float(orow[4 * u + 3]) * inv);
      }
    }
    tc::tc_fence_before();
    if (c == 0) {
      if (pp.partial < 0) { if (a.lse) a.lse[row] = lse2 * 0.69314718055994531f; }
      else a.part_lse[static_cast<int64_t>(pp.partial) * a.heads + h] = lse2;
    }
    return true;
  };

  Cursor cur;
  cur.begin(a, seg_b, seg_e);
  int cur_req = -1;
  float q_scale = a.scale_log2;
  PendingPage pend{};
  bool have = false;
  uint32_t own_prev[64];
  for (int g = 0; !cur.done(); ++g) {
    const Segment seg = cur.seg;
    if (cur.j == 0 && seg.req != cur_req) {
      // ---- Q row of head h (QK of the previous page has completed: its logits were read). A
      // power of two 2^-sh from the row's largest |q| (the same in both CTAs) keeps every value
      // inside FP16; 2^sh joins this row's logit scale ----
      const uint8_t* qrow = reinterpret_cast<const uint8_t*>(a.q) + (static_cast<int64_t>(seg.req) * 128 + h) * (kLatent * 2);
      uint32_t mx = 0;
      for (int i = 0; i < kLatent * 2 / 16; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + 16 * i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
      }
      int sh = 0;
      if (mx != 0u && mx < 0x7F80u) sh = max(-100, min(113, static_cast<int>(mx >> 7) - 127 - 14));
      const float down = __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
      q_scale = a.scale_log2 * __uint_as_float(static_cast<uint32_t>(127 + sh) << 23);
#pragma unroll
      for (int part = 0; part < 4; ++part) {          // 4 x 64 nope dims -> 4 x 32 TMEM columns
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = *reinterpret_cast<const uint4*>(qrow + (256 * c + 64 * part + 8 * i) * 2);
          r[4 * i] = dev::bf16x2_to_f16x2(v.x, down);
          r[4 * i + 1] = dev::bf16x2_to_f16x2(v.y, down);
          r[4 * i + 2] = dev::bf16x2_to_f16x2(v.z, down);
          r[4 * i + 3] = dev::bf16x2_to_f16x2(v.w, down);
        }
        __syncwarp();
        tc::tmem_st32(tl + TM_QN + 32 * part, r);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {                   // 32 rope dims -> one 64-byte row
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + (512 + 32 * c + 8 * i) * 2);
        sts128(qr + tc::sw64_offset(h, i), make_uint4(dev::bf16x2_to_f16x2(v.x, down), dev::bf16x2_to_f16x2(v.y, down),
                                                     dev::bf16x2_to_f16x2(v.z, down), dev::bf16x2_to_f16x2(v.w, down)));
      }
      tc::tmem_wait_st();
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(sy.bar(B_Q_READY));
      cur_req = seg.req;
    }
    const int64_t pg = cur.page(a);
    PendingPage now;
    now.g = g;
    now.valid = page_ok(a, pg) ? cur.valid() : 0;
    now.j = cur.j;
    now.last = cur.j == seg.num_pages - 1;
    now.partial = seg.partial;
    now.req = seg.req;
    now.q_scale = q_scale;
    // ---- stage 1: this page's partial logits into the local exchange buffer ----
    const int s = g & 1;
    if (!wait(B_S_FULL + s, (g >> 1) & 1, false, 128)) return;
    tc::tc_fence_after();
    uint32_t sr[64];
    tc::tmem_ld32(tl + TM_S + 64 * s, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
    tc::tmem_ld32(tl + TM_S + 64 * s + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
    tc::tmem_wait_ld();
    tc::tc_fence_before();
    tc::mbar_arrive(sy.bar(B_S_FREE + s));
    if (g >= 2 && !wait(B_X_FREE + s, ((g >> 1) - 1) & 1, true, 4096)) return;
    const uint32_t xremote = tc::mapa(xbuf + s * kXBytes + h * 16, peer);
#pragma unroll
    for (int i = 0; i < 16; ++i) tc::st_cluster_v4(xremote + i * 2048, sr[4 * i], sr[4 * i + 1], sr[4 * i + 2], sr[4 * i + 3]);
    // ---- stage 2: the previous page, while the remote stores drain ----
    if (have && !finish(pend, own_prev)) return;
    tc::mbar_arrive_cluster(sy.bar(B_X_FULL + s), peer);   // release: publishes this page's logits
#pragma unroll
    for (int i = 0; i < 64; ++i) own_prev[i] = sr[i];
    pend = now;
    have = true;
    cur.next(a);
  }
  if (have) finish(pend, own_prev);
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
    for (int i = 0; i < 3; ++i) { tc::mbar_init(sy.bar(B_TILE_FULL + i), kDQ); tc::mbar_init(sy.bar(B_TILE_EMPTY + i), 1); }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(sy.bar(B_S_FULL + i), 1);
      tc::mbar_init(sy.bar(B_S_FREE + i), 128);
      tc::mbar_init(sy.bar(B_P_FULL + i), 128);
      tc::mbar_init(sy.bar(B_P_FREE + i), 1);
      tc::mbar_init(sy.bar(B_X_FULL + i), 128);
    }
    tc::mbar_init(sy.bar(B_O_DONE), 1);
    tc::mbar_init(sy.bar(B_O_DONE + 1), 1);
    tc::mbar_init(sy.bar(B_Q_READY), 128);
    tc::mbar_init(sy.bar(B_X_FREE), 128);
    tc::mbar_init(sy.bar(B_X_FREE + 1), 128);
    tc::mbar_init(sy.bar(B_FINAL), 1);
    *sy.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 7) {
    tc::tmem_alloc(base + OFF_TSLOT, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();          // the peer's barriers are initialised before any remote arrive
  tc::tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(sbase + OFF_TSLOT);

  if (warp < 4) {
    role_softmax<KV>(a, sy, seg_b, seg_e, c, tid, tbase, base + OFF_P, base + OFF_QR, base + OFF_X);
  } else if (warp < 7) {
    role_dequant<KV>(a, sy, seg_b, seg_e, c, tid - 128, base + OFF_TILE);
  } else if ((tid & 31) == 0) {
    role_mma(a, sy, seg_b, seg_e, tbase, base + OFF_TILE, base + OFF_P, base + OFF_QR);
  }
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 7) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tbase, 512);
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
  if (a.heads != 128 || a.ctas_per_worker != 2) return cudaErrorInvalidValue;
  switch (a.kv_dtype) {
    case KV_FP8: return launch_kv<KV_FP8>(a, s);
    case KV_NVFP4: return launch_kv<KV_NVFP4>(a, s);
    case KV_BF16: return launch_kv<KV_BF16>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qkvp
