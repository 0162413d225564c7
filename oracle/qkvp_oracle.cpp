// Oracle for paged MLA decode over a quantized (FP8 E4M3 / NVFP4) latent KV cache.
//
// TEST INFRASTRUCTURE. This file is the plain, slow CPU statement of what the GPU path computes.
// Only the tests, the package's smoke check and the benchmark's CPU-baseline leg may load it. The
// product path never does. It shares no code, header, table or constant generator with the CUDA
// library; it is built with plain g++ (-O2 -ffp-contract=off, no fast-math), so every FP32 step
// below is one IEEE-754 operation rounded to nearest-even, and every FP64 step is plain double
// arithmetic.
//
// Sources (pages as extracted; see the module notes for readings where the pages are silent):
//  * FP8 KV storage as float8_e4m3fn: "The FP8 KV Cache Wall", section "Context and Motivation".
//  * The 576-wide latent (512 + 64) and the pool [495552, 1, 576]: "The Smoking Gun", section
//    "The Investigation Leading to This Message".
//  * NVFP4: 4-bit E2M1 values (1 sign, 2 exponent, 1 mantissa bit), one E4M3 scale per block of 16
//    values, one FP32 global scale per tensor; 8 packed bytes + 1 scale byte per 16 values:
//    "SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "NVFP4 format: two-level scaling".
//  * Quantize-on-write and in-kernel dequant for decode: same page, section "SGLang
//    implementation", items 1-3.
//  * Per-token-scaled FP8 pages (c9): each token's E4M3 elements with 4 scale bytes of their own,
//    64 tokens per page: "The Precision Frontier: Implementing bf16 Index Keys ...", section "The
//    Message: Planning the bf16-K Implementation".
//  * Attention is softmax(sm_scale * q . k) v with K = the whole latent and V = its first 512 dims,
//    the paged CSR page table of the pages' plan() call: "The Smoking Gun", section "What Message
//    1408 Actually Reveals".
//
// Parity status per function is stated in its comment. Every function here is pinned by a
// `-m "not gpu"` test (closed forms, library routines, brute force, invariants).

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr int kLatent = 576;   // kv_lora_rank 512 + rope 64
constexpr int kDv = 512;       // V = first 512 latent dims
constexpr int kBlock = 16;     // NVFP4 values per E4M3 block scale
constexpr int kBlocksPerToken = kLatent / kBlock;      // 36
constexpr int kPackedPerToken = kLatent / 2;           // 288 bytes of E2M1 pairs

enum { KV_FP8 = 1, KV_NVFP4 = 2, KV_BF16 = 3, KV_FP8_PT = 4 };

// Per-token-scaled FP8 pages (c9): page p holds kPagePT token rows of 576 E4M3 codes, then the
// kPagePT FP32 token scales (little-endian), kPagePT * (576 + 4) = 37,120 bytes in all.
constexpr int kPagePT = 64;
constexpr int64_t kPageBytesPT = static_cast<int64_t>(kPagePT) * (kLatent + 4);
enum { SRC_FP8 = 1, SRC_BF16 = 2 };

// ---- c1: code -> value tables, from the bit layouts ------------------------------------------

// E4M3 (float8_e4m3fn): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 is
// subnormal (m * 2^-9); the all-ones pattern S.1111.111 is NaN; there is no infinity.
double e4m3_value(uint32_t code) {
  code &= 0xFF;
  const double sign = (code & 0x80) ? -1.0 : 1.0;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  if (e == 0xF && m == 0x7) return std::nan("");
  if (e == 0) return sign * std::ldexp(static_cast<double>(m), -9);
  return sign * std::ldexp(1.0 + m / 8.0, e - 7);
}

// E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent field 0 is subnormal (m * 0.5).
// No NaN and no infinity. Codes 0x0-0x7 are +{0, 0.5, 1, 1.5, 2, 3, 4, 6}; bit 3 is the sign.
double e2m1_value(uint32_t code) {
  code &= 0xF;
  const double sign = (code & 0x8) ? -1.0 : 1.0;
  const int e = (code >> 1) & 0x3;
  const int m = code & 0x1;
  if (e == 0) return sign * 0.5 * m;
  return sign * std::ldexp(1.0 + m / 2.0, e - 1);
}

// Round-half-to-even of a non-negative double that is exactly representable (q < 2^52).
double rne(double q) {
  double f = std::floor(q);
  double r = q - f;  // exact
  if (r > 0.5) return f + 1.0;
  if (r < 0.5) return f;
  return (std::fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

// ---- c2: FP32 -> E4M3, round to nearest even, saturate to +-448 ------------------------------
// NaN -> 0x7F. Signed zero and values that round to zero keep their sign (0x80 for negatives).
uint8_t e4m3_encode(float xf) {
  if (std::isnan(xf)) return 0x7F;
  const uint8_t sign = std::signbit(xf) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(xf));
  if (a >= 448.0) return sign | 0x7E;  // satfinite: 448 and everything above (inf included)
  if (a < std::ldexp(1.0, -6)) {       // below the smallest normal: multiples of 2^-9
    const double m = rne(std::ldexp(a, 9));    // 0..8; 8 is the smallest normal, code 0x08
    return sign | static_cast<uint8_t>(m);
  }
  int e2;
  std::frexp(a, &e2);                  // a = f * 2^e2, f in [0.5, 1)  ->  a in [2^(e2-1), 2^e2)
  int e = e2 - 1;                      // unbiased exponent of a
  double m = rne(std::ldexp(a, 3 - e));  // in [8, 16]
  if (m == 16.0) { m = 8.0; e += 1; }
  const int code = ((e + 7) << 3) | (static_cast<int>(m) - 8);
  return sign | static_cast<uint8_t>(code);  // a < 448 keeps code <= 0x7E
}

// ---- c3 step 5: FP32 -> E2M1, round to nearest even, saturate to +-6 -------------------------
// Thresholds are the midpoints between neighbouring E2M1 values; a value exactly on a midpoint
// goes to the neighbour whose code is even. NaN -> 0x0. Negatives that round to zero give 0x8.
uint8_t e2m1_encode(float xf) {
  if (std::isnan(xf)) return 0x0;
  const uint8_t sign = std::signbit(xf) ? 0x8 : 0x0;
  const double a = std::fabs(static_cast<double>(xf));
  uint8_t c;
  if (a <= 0.25) c = 0;        // 0   | 0.5 : tie -> 0 (even)
  else if (a < 0.75) c = 1;    // 0.5 | 1   : tie -> 1.0 (code 2)
  else if (a <= 1.25) c = 2;   // 1   | 1.5 : tie -> 1.0
  else if (a < 1.75) c = 3;    // 1.5 | 2   : tie -> 2.0 (code 4)
  else if (a <= 2.5) c = 4;    // 2   | 3   : tie -> 2.0
  else if (a < 3.5) c = 5;     // 3   | 4   : tie -> 4.0 (code 6)
  else if (a <= 5.0) c = 6;    // 4   | 6   : tie -> 4.0
  else c = 7;                  // 6 and above (saturate)
  return sign | c;
}

// ---- c3: NVFP4 quantisation of one 16-value block --------------------------------------------
// FP32 throughout, one rounding per operation, in this order:
//   amax = max |x_i| (NaN if any x_i is NaN)
//   s    = amax / (6 * g)                 (6 * g rounded first)
//   s8   = E4M3(s)                        (c2)
//   sd   = value(s8) * g
//   c_i  = 0 if sd == 0, else E2M1(x_i / sd)
// byte k of the packed pair holds c_{2k} in its low nibble and c_{2k+1} in its high nibble.
void nvfp4_block(const float* x, float g, uint8_t* packed, uint8_t* scale) {
  float amax = 0.0f;
  bool nan = false;
  for (int i = 0; i < kBlock; ++i) {
    if (std::isnan(x[i])) nan = true;
    else if (std::fabs(x[i]) > amax) amax = std::fabs(x[i]);
  }
  if (nan) amax = std::nanf("");
  volatile float denom = 6.0f * g;
  volatile float s = amax / denom;
  const uint8_t s8 = e4m3_encode(s);
  volatile float sd = static_cast<float>(e4m3_value(s8)) * g;
  uint8_t c[kBlock];
  for (int i = 0; i < kBlock; ++i) {
    if (sd == 0.0f) { c[i] = 0; continue; }
    volatile float v = x[i] / sd;
    c[i] = e2m1_encode(v);
  }
  for (int k = 0; k < kBlock / 2; ++k) packed[k] = static_cast<uint8_t>(c[2 * k] | (c[2 * k + 1] << 4));
  *scale = s8;
}

// ---- c9: per-token-scaled FP8 of one token ---------------------------------------------------
// The pages' indexer key cache stores each token's FP8 elements with 4 scale bytes of their own, in
// a paged uint8 buffer [npages, page_bytes] with 64 tokens per page ("The Precision Frontier:
// Implementing bf16 Index Keys ...", section "The Message: Planning the bf16-K Implementation":
// 128 elements + 4 scale bytes = 132 bytes per token). Here the layout carries the 576-wide latent:
// 576 + 4 bytes per token. The pages give no formula for the scale; the one here maps the token's
// largest magnitude onto E4M3's largest finite value (448, c1). FP32 throughout, one rounding per
// operation:
//   amax  = max |x_i|
//   sigma = amax / 448, or the NaN 0x7FC00000 if any x_i is NaN (one fixed pattern for the stored
//           bytes: a division's NaN result carries no portable payload)
//   c_i   = E4M3(x_i / sigma)             (c2; 0x7F for every element of a NaN token), or
//           E4M3(x_i) (a signed zero) when sigma == 0
// The value of element i is sigma * value(c_i).
void pt_token(const float* x, uint8_t* codes, float* sigma) {
  float amax = 0.0f;
  bool nan = false;
  for (int i = 0; i < kLatent; ++i) {
    if (x[i] != x[i]) nan = true;
    const float a = std::fabs(x[i]);
    if (a > amax) amax = a;
  }
  float s = amax / 448.0f;
  if (nan) {
    const uint32_t qnan = 0x7FC00000u;
    std::memcpy(&s, &qnan, 4);
  }
  for (int i = 0; i < kLatent; ++i) codes[i] = (s == 0.0f) ? e4m3_encode(x[i]) : e4m3_encode(x[i] / s);
  *sigma = s;
}

float bf16_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Source element i of token n as FP32 (FP8 bytes decode exactly; BF16 widens exactly).
float src_value(const void* src, int src_dtype, int64_t n, int i) {
  if (src_dtype == SRC_FP8) return static_cast<float>(e4m3_value(static_cast<const uint8_t*>(src)[n * kLatent + i]));
  return bf16_to_float(static_cast<const uint16_t*>(src)[n * kLatent + i]);
}

template <class F>
void parallel_for(int64_t n, int threads, F f) {
  if (threads <= 1 || n <= 1) { for (int64_t i = 0; i < n; ++i) f(i); return; }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t)
    pool.emplace_back([&] { for (int64_t i; (i = next.fetch_add(1)) < n;) f(i); });
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

double qo_e4m3_value(uint32_t code) { return e4m3_value(code); }
double qo_e2m1_value(uint32_t code) { return e2m1_value(code); }
uint8_t qo_e4m3_encode(float x) { return e4m3_encode(x); }
uint8_t qo_e2m1_encode(float x) { return e2m1_encode(x); }

// Encode n FP32 values (c2 when fmt == 1, E2M1 of c3 step 5 when fmt == 2), one byte per value.
void qo_encode_array(const float* x, int64_t n, int fmt, uint8_t* out, int threads) {
  const int64_t chunk = 1 << 20;
  parallel_for((n + chunk - 1) / chunk, threads, [&](int64_t c) {
    const int64_t a = c * chunk, b = std::min(n, a + chunk);
    for (int64_t i = a; i < b; ++i) out[i] = (fmt == 1) ? e4m3_encode(x[i]) : e2m1_encode(x[i]);
  });
}

// Encode every FP32 bit pattern in [lo, hi) and return how many codes differ from `codes`
// (indexed from lo); the first mismatching pattern goes to *first_bad. For the exhaustive check.
int64_t qo_encode_range_compare(uint64_t lo, uint64_t hi, int fmt, const uint8_t* codes,
                                uint64_t* first_bad, int threads) {
  const int64_t n = static_cast<int64_t>(hi - lo);
  const int64_t chunk = 1 << 22;
  const int64_t nchunks = (n + chunk - 1) / chunk;
  std::vector<int64_t> bad(nchunks, 0);
  std::vector<uint64_t> first(nchunks, ~0ull);
  parallel_for(nchunks, threads, [&](int64_t c) {
    const int64_t a = c * chunk, b = std::min(n, a + chunk);
    for (int64_t i = a; i < b; ++i) {
      const uint32_t bits = static_cast<uint32_t>(lo + i);
      float f;
      std::memcpy(&f, &bits, 4);
      const uint8_t want = (fmt == 1) ? e4m3_encode(f) : e2m1_encode(f);
      if (want != codes[i]) { if (!bad[c]) first[c] = lo + i; ++bad[c]; }
    }
  });
  int64_t total = 0;
  uint64_t fb = ~0ull;
  for (int64_t c = 0; c < nchunks; ++c) { total += bad[c]; if (bad[c] && first[c] < fb) fb = first[c]; }
  if (first_bad) *first_bad = fb;
  return total;
}

// c3 on one block of 16 FP32 values.
void qo_nvfp4_block(const float* x16, float g, uint8_t* packed8, uint8_t* scale1) {
  nvfp4_block(x16, g, packed8, scale1);
}

// Quantise n tokens token-major. kv_dtype FP8: out_data [n][576] E4M3 bytes (FP8 sources are
// copied; BF16 sources go through c2). kv_dtype NVFP4: out_data [n][288] packed E2M1 pairs and
// out_scale [n][36] E4M3 block scales (c3 per block of 16 consecutive channels). kv_dtype FP8_PT:
// out_data [n][576] E4M3 codes and out_scale [n] FP32 token scales as 4 little-endian bytes (c9).
int qo_quant_tokens(const void* src, int src_dtype, int64_t n, int kv_dtype, float g,
                    uint8_t* out_data, uint8_t* out_scale, int threads) {
  if (src_dtype != SRC_FP8 && src_dtype != SRC_BF16) return -2;
  if (kv_dtype != KV_FP8 && kv_dtype != KV_NVFP4 && kv_dtype != KV_FP8_PT) return -2;
  parallel_for(n, threads, [&](int64_t t) {
    if (kv_dtype == KV_FP8_PT) {
      float x[kLatent], sigma;
      for (int i = 0; i < kLatent; ++i) x[i] = src_value(src, src_dtype, t, i);
      pt_token(x, out_data + t * kLatent, &sigma);
      std::memcpy(out_scale + 4 * t, &sigma, 4);
      return;
    }
    if (kv_dtype == KV_FP8) {
      for (int i = 0; i < kLatent; ++i) {
        out_data[t * kLatent + i] = (src_dtype == SRC_FP8)
            ? static_cast<const uint8_t*>(src)[t * kLatent + i]
            : e4m3_encode(src_value(src, src_dtype, t, i));
      }
      return;
    }
    float x[kBlock];
    for (int j = 0; j < kBlocksPerToken; ++j) {
      for (int i = 0; i < kBlock; ++i) x[i] = src_value(src, src_dtype, t, j * kBlock + i);
      nvfp4_block(x, g, out_data + t * kPackedPerToken + j * (kBlock / 2), out_scale + t * kBlocksPerToken + j);
    }
  });
  return 0;
}

// The paged write of quantize-on-append: token n goes to slot slots[n] (page * page_size +
// offset) of the pool; negative slots are skipped. Pools: FP8 [pages][page_size][576];
// NVFP4 data [pages][page_size][288] and scales [pages][page_size][36]; FP8_PT [pages][37,120]
// (c9 layout, page_size 64).
int qo_append(const void* src, int src_dtype, int64_t n, const int64_t* slots, int kv_dtype,
              float g, int page_size, int64_t num_pages, uint8_t* pool_data, uint8_t* pool_scale) {
  const int64_t nslots = num_pages * page_size;
  if (kv_dtype == KV_FP8_PT && page_size != kPagePT) return -2;
  const int row = (kv_dtype == KV_NVFP4) ? kPackedPerToken : kLatent;
  std::vector<uint8_t> d(row), s(kBlocksPerToken);
  for (int64_t t = 0; t < n; ++t) {
    const int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= nslots) return -1;
    const uint8_t* one = nullptr;
    if (src_dtype == SRC_FP8) one = static_cast<const uint8_t*>(src) + t * kLatent;
    else one = reinterpret_cast<const uint8_t*>(static_cast<const uint16_t*>(src) + t * kLatent);
    int rc = qo_quant_tokens(one, src_dtype, 1, kv_dtype, g, d.data(), s.data(), 1);
    if (rc) return rc;
    if (kv_dtype == KV_FP8_PT) {
      uint8_t* page = pool_data + (slot / kPagePT) * kPageBytesPT;
      std::memcpy(page + (slot % kPagePT) * kLatent, d.data(), kLatent);
      std::memcpy(page + kPagePT * kLatent + (slot % kPagePT) * 4, s.data(), 4);
      continue;
    }
    std::memcpy(pool_data + slot * row, d.data(), row);
    if (kv_dtype == KV_NVFP4) std::memcpy(pool_scale + slot * kBlocksPerToken, s.data(), kBlocksPerToken);
  }
  return 0;
}

// c4: the dequantised latent of one pool slot, in FP64.
//   FP8:   x_i = value(byte_i)
//   NVFP4: x_i = g * value(s8_{i/16}) * value(c_i)
//   BF16:  x_i = the BF16 value
//   FP8_PT: x_i = sigma * value(c_i), slot = page * 64 + offset in the c9 page layout
void qo_dequant_slot(const void* kv_data, const uint8_t* kv_scale, int kv_dtype, double g,
                     int64_t slot, double* x) {
  if (kv_dtype == KV_FP8_PT) {
    const uint8_t* page = static_cast<const uint8_t*>(kv_data) + (slot / kPagePT) * kPageBytesPT;
    float sigma;
    std::memcpy(&sigma, page + kPagePT * kLatent + (slot % kPagePT) * 4, 4);
    for (int i = 0; i < kLatent; ++i) x[i] = static_cast<double>(sigma) * e4m3_value(page[(slot % kPagePT) * kLatent + i]);
    return;
  }
  for (int i = 0; i < kLatent; ++i) {
    if (kv_dtype == KV_FP8) {
      x[i] = e4m3_value(static_cast<const uint8_t*>(kv_data)[slot * kLatent + i]);
    } else if (kv_dtype == KV_BF16) {
      x[i] = bf16_to_float(static_cast<const uint16_t*>(kv_data)[slot * kLatent + i]);
    } else {
      const uint8_t byte = static_cast<const uint8_t*>(kv_data)[slot * kPackedPerToken + i / 2];
      const uint8_t code = (i & 1) ? (byte >> 4) : (byte & 0xF);
      x[i] = g * e4m3_value(kv_scale[slot * kBlocksPerToken + i / kBlock]) * e2m1_value(code);
    }
  }
}

// c5: decode attention for a list of (request, head) pairs, in FP64.
// For request r of length L and head h, token t (< L) is slot
// kv_indices[kv_indptr[r] + t / page_size] * page_size + t % page_size, and
//   z_t  = sm_scale * sum_{d<576} q[r,h,d] * x_t[d]
//   lse  = m + ln sum_t exp(z_t - m),  m = max_t z_t
//   o[v] = sum_t exp(z_t - lse) * x_t[v],  v < 512
// L == 0 gives o = 0 and lse = -inf. Returns -1 if a page id is outside the pool.
int qo_mla_decode(const uint16_t* q_bf16, int batch, int heads, const void* kv_data,
                  const uint8_t* kv_scale, int kv_dtype, int page_size, int64_t num_pages,
                  const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* kv_len,
                  double sm_scale, double g, const int32_t* pairs, int64_t npairs,
                  double* out_o, double* out_lse, int threads) {
  std::atomic<int> err{0};
  if (kv_dtype == KV_FP8_PT && page_size != kPagePT) return -2;
  const int64_t n = pairs ? npairs : static_cast<int64_t>(batch) * heads;
  parallel_for(n, threads, [&](int64_t p) {
    const int r = pairs ? pairs[2 * p] : static_cast<int>(p / heads);
    const int h = pairs ? pairs[2 * p + 1] : static_cast<int>(p % heads);
    const int64_t L = kv_len[r];
    double* o = out_o + p * kDv;
    for (int v = 0; v < kDv; ++v) o[v] = 0.0;
    if (L == 0) { out_lse[p] = -INFINITY; return; }
    const uint16_t* q = q_bf16 + (static_cast<int64_t>(r) * heads + h) * kLatent;
    std::vector<double> qd(kLatent), x(kLatent), z(L);
    for (int d = 0; d < kLatent; ++d) qd[d] = bf16_to_float(q[d]);
    std::vector<int64_t> slot(L);
    for (int64_t t = 0; t < L; ++t) {
      const int64_t page = kv_indices[kv_indptr[r] + t / page_size];
      if (page < 0 || page >= num_pages) { err = -1; return; }
      slot[t] = page * page_size + t % page_size;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < L; ++t) {
      qo_dequant_slot(kv_data, kv_scale, kv_dtype, g, slot[t], x.data());
      double dot = 0.0;
      for (int d = 0; d < kLatent; ++d) dot += qd[d] * x[d];
      z[t] = sm_scale * dot;
      if (z[t] > m) m = z[t];
    }
    double sum = 0.0;
    for (int64_t t = 0; t < L; ++t) sum += std::exp(z[t] - m);
    const double lse = m + std::log(sum);
    for (int64_t t = 0; t < L; ++t) {
      qo_dequant_slot(kv_data, kv_scale, kv_dtype, g, slot[t], x.data());
      const double p_t = std::exp(z[t] - lse);
      for (int v = 0; v < kDv; ++v) o[v] += p_t * x[v];
    }
    out_lse[p] = lse;
  });
  return err.load();
}

// c6: merge n partial results (o_i normalised within its part, lse_i its log-sum-exp):
//   lse = M + ln sum_i exp(lse_i - M),  o = sum_i exp(lse_i - lse) o_i,  M = max_i lse_i.
// Parts with lse_i = -inf (empty) carry no weight; all parts empty gives o = 0, lse = -inf.
void qo_lse_merge(int n, int dv, const double* o_parts, const double* lse_parts, double* o, double* lse) {
  double M = -INFINITY;
  for (int i = 0; i < n; ++i) if (lse_parts[i] > M) M = lse_parts[i];
  for (int v = 0; v < dv; ++v) o[v] = 0.0;
  if (M == -INFINITY) { *lse = -INFINITY; return; }
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += std::exp(lse_parts[i] - M);
  const double L = M + std::log(s);
  for (int i = 0; i < n; ++i) {
    const double w = std::exp(lse_parts[i] - L);
    for (int v = 0; v < dv; ++v) o[v] += w * o_parts[static_cast<int64_t>(i) * dv + v];
  }
  *lse = L;
}

// The pool-wide cast of the pages' baseline: every FP8 byte to its BF16 value (exact).
// NaN bytes (0x7F, 0xFF) become the canonical BF16 quiet NaN 0x7FC0.
void qo_cast_fp8_to_bf16(const uint8_t* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    if ((in[i] & 0x7F) == 0x7F) { out[i] = 0x7FC0; continue; }
    const float f = static_cast<float>(e4m3_value(in[i]));
    uint32_t u;
    std::memcpy(&u, &f, 4);
    out[i] = static_cast<uint16_t>(u >> 16);
  }
}

// c7: the extend path's gather ("SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "SGLang
// implementation", item 2: the cached prefix is gathered and dequantized into an FP8 workspace shared
// by all layers). Row tok_indptr[r] + t of `out` ([tok_indptr[batch]][576] E4M3 bytes) holds token t
// of request r, read from slot kv_indices[p] * page_size + t % page_size with
// p = kv_indptr[r] + t / page_size. FP8 pools are copied byte for byte. NVFP4 elements become
//   v = fp32(value(s8) * value(c)) * g   (the first product is exact, at most 4 + 2 significant
//                                           bits; the multiply by g is one FP32 rounding)
//   byte = E4M3_RNE_satfinite(v)         (c2)
// which reads "dequantize into FP8" as a return to the E4M3 domain the NVFP4 data was quantized from
// (the page gives no other scale for the workspace). A row whose page-table entry lies outside the
// request's pages, the table (nnz entries) or the pool is written as zeros. Returns the number of
// such rows.
int64_t qo_gather_fp8(const void* kv_data, const uint8_t* kv_scale, int kv_dtype, float g, int page_size,
                      int64_t num_pages, const int32_t* kv_indptr, const int32_t* kv_indices, int64_t nnz,
                      const int64_t* tok_indptr, int batch, uint8_t* out) {
  int64_t bad = 0;
  for (int r = 0; r < batch; ++r) {
    for (int64_t t = 0; t < tok_indptr[r + 1] - tok_indptr[r]; ++t) {
      uint8_t* row = out + (tok_indptr[r] + t) * kLatent;
      const int64_t p = kv_indptr[r] + t / page_size;
      const bool ok_p = p < kv_indptr[r + 1] && p >= 0 && p < nnz;
      const int64_t page = ok_p ? kv_indices[p] : -1;
      if (page < 0 || page >= num_pages) {
        std::memset(row, 0, kLatent);
        ++bad;
        continue;
      }
      const int64_t slot = page * page_size + t % page_size;
      for (int i = 0; i < kLatent; ++i) {
        if (kv_dtype == KV_FP8) {
          row[i] = static_cast<const uint8_t*>(kv_data)[slot * kLatent + i];
        } else {
          const uint8_t byte = static_cast<const uint8_t*>(kv_data)[slot * kPackedPerToken + i / 2];
          const uint8_t code = (i & 1) ? (byte >> 4) : (byte & 0xF);
          const float se = static_cast<float>(e4m3_value(kv_scale[slot * kBlocksPerToken + i / kBlock]) *
                                              e2m1_value(code));
          const float v = se * g;
          row[i] = e4m3_encode(v);
        }
      }
    }
  }
  return bad;
}

// c8: the gather-then-cast baseline ("The FP8 KV Cache Wall", sections "The Message" and
// "Aftermath": Option B, cast only the active tokens instead of the whole pool): page i of `out`
// ([n][page_size][576] BF16 bits) is pool page page_ids[i] cast
// exactly as in the pool-wide cast (NaN bytes become 0x7FC0). Page ids outside the pool give zeros.
void qo_gather_pages_bf16(const uint8_t* pool, int page_size, int64_t num_pages, const int32_t* page_ids,
                          int64_t n, uint16_t* out) {
  const int64_t per = static_cast<int64_t>(page_size) * kLatent;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t page = page_ids[i];
    if (page < 0 || page >= num_pages) {
      std::memset(out + i * per, 0, per * sizeof(uint16_t));
      continue;
    }
    qo_cast_fp8_to_bf16(pool + page * per, per, out + i * per);
  }
}

int qo_hardware_threads() { return static_cast<int>(std::thread::hardware_concurrency()); }

}  // extern "C"
