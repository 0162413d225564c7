// Gathers of a paged pool into dense buffers:
//  * the extend path's FP8 workspace ("SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "SGLang
//    implementation", item 2: a chunked-prefill step gathers each request's cached prefix and
//    dequantizes it into one FP8 workspace that all layers share). FP8 pools are copied; NVFP4
//    elements become E4M3(fp32(scale * e2m1) * g), i.e. the E4M3 domain the cache was quantized from.
//  * the gather-then-cast baseline ("The FP8 KV Cache Wall", sections "The Message" and "Aftermath":
//    Option B casts only the pages a batch reads to BF16, not the whole pool).
// Both are streaming kernels bound by HBM: 16-byte loads and stores, one thread per 16 latent
// elements, every page-table entry bounds-checked (an entry outside the request's pages, the table
// or the pool gives a zero row).
#include <cstdint>

#include "qkvp_device.cuh"
#include "qkvp_internal.h"

namespace qkvp {
namespace {

constexpr int kRowsPerPass = 8;                 // 8 rows x 36 blocks of 16 elements = 288 threads
constexpr int kGatherThreads = kRowsPerPass * (kLatent / 16);

// Request owning workspace row `row`: the largest r < batch with tok_indptr[r] <= row.
__device__ __forceinline__ int find_request(const int64_t* tok_indptr, int batch, int64_t row) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tok_indptr[mid] <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float f16_low(uint32_t h2) { return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu))); }
__device__ __forceinline__ float f16_high(uint32_t h2) { return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16))); }

// Two E4M3 pairs (16-bit results of the pair conversions) -> one word, first pair in the low half.
__device__ __forceinline__ uint32_t pack_b16x2(uint32_t lo, uint32_t hi) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, h;\n\tcvt.u16.u32 l, %1;\n\tcvt.u16.u32 h, %2;\n\tmov.b32 %0, {l, h};\n\t}"
      : "=r"(r) : "r"(lo), "r"(hi));
  return r;
}

// One NVFP4 block (16 elements: 8 packed bytes, one scale byte) -> 16 E4M3 bytes.
__device__ __forceinline__ uint4 nvfp4_block_to_e4m3(uint2 d, uint32_t s8, float g) {
  if ((s8 & 0x7Fu) == 0x7Fu)                  // NaN block scale: every element is NaN -> 0x7F
    return make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  const uint32_t s2 = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(s8 | (s8 << 8)));
  uint32_t c[8];                              // code pairs from byte registers; pair k = elements 2k, 2k + 1
  dev::e2m1x8_to_f16x2x4(d.x, *reinterpret_cast<uint32_t(*)[4]>(c));
  dev::e2m1x8_to_f16x2x4(d.y, *reinterpret_cast<uint32_t(*)[4]>(c + 4));
  uint32_t e[8];
  if (g == 1.0f) {
    // s * e has at most 6 significant bits within [2^-10, 2688]: exact in FP16, so one FP16x2
    // multiply and one FP16x2 -> E4M3x2 conversion (RNE, satfinite) per pair
#pragma unroll
    for (int k = 0; k < 8; ++k) e[k] = dev::f16x2_to_e4m3x2(dev::hmul2_f16(c[k], s2));
  } else {
    // the exact product in FP16x2, widened to FP32, one FP32 multiply by g per element, one
    // conversion per pair (RNE, satfinite; no NaN can reach it: NaN scales were handled above)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t v2 = dev::hmul2_f16(c[k], s2);
      e[k] = dev::f32x2_to_e4m3x2(__fmul_rn(f16_low(v2), g), __fmul_rn(f16_high(v2), g));
    }
  }
  return make_uint4(pack_b16x2(e[0], e[1]), pack_b16x2(e[2], e[3]), pack_b16x2(e[4], e[5]), pack_b16x2(e[6], e[7]));
}

// Each CTA pass covers 64 workspace rows. The 64 rows' pool slots are resolved once per pass (one
// thread per row: the request by binary search over tok_indptr, then the page-table entry, every
// entry bounds-checked) into shared memory; thread (sub, blk) then handles block blk of rows
// base + sub + 8k, k = 0..7, with its eight loads in flight together before any conversion.
template <int KV>
__global__ void __launch_bounds__(kGatherThreads) gather_fp8_kernel(const GatherArgs a) {
  constexpr int kRows = 8;
  constexpr int kPassRows = kRowsPerPass * kRows;
  __shared__ int64_t s_slot[kPassRows];
  const int sub = threadIdx.x / 36, blk = threadIdx.x % 36;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kPassRows; base < a.total_tokens;
       base += static_cast<int64_t>(gridDim.x) * kPassRows) {
    if (threadIdx.x < kPassRows) {
      const int64_t row = base + threadIdx.x;
      int64_t slot = -1;
      if (row < a.total_tokens) {
        const int r = find_request(a.tok_indptr, a.batch, row);
        const int64_t t = row - a.tok_indptr[r];
        const int64_t p = a.kv_indptr[r] + t / kPage;
        if (t >= 0 && p >= 0 && p < a.kv_indptr[r + 1] && p < a.nnz) {
          const int64_t page = a.kv_indices[p];
          if (page >= 0 && page < a.num_pages) slot = page * kPage + t % kPage;
        }
      }
      s_slot[threadIdx.x] = slot;
    }
    __syncthreads();
    int64_t slot[kRows];
    uint4 raw[kRows];
    uint32_t s8[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      slot[k] = s_slot[sub + kRowsPerPass * k];
      raw[k] = make_uint4(0, 0, 0, 0);
      s8[k] = 0;
      if (slot[k] < 0) continue;
      if (KV == KV_FP8) {
        raw[k] = __ldcs(reinterpret_cast<const uint4*>(a.kv + slot[k] * kLatent) + blk);
      } else {
        const uint2 d = __ldcs(reinterpret_cast<const uint2*>(a.kv + slot[k] * kPacked) + blk);
        raw[k].x = d.x;
        raw[k].y = d.y;
        s8[k] = a.kv_scale[slot[k] * kScales + blk];
      }
    }
    __syncthreads();                          // s_slot is rewritten by the next pass
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      const int64_t row = base + sub + kRowsPerPass * k;
      if (row >= a.total_tokens) continue;
      uint4 o = make_uint4(0, 0, 0, 0);
      if (slot[k] >= 0) o = KV == KV_FP8 ? raw[k] : nvfp4_block_to_e4m3(make_uint2(raw[k].x, raw[k].y), s8[k], a.g);
      __stcs(reinterpret_cast<uint4*>(a.out + row * kLatent) + blk, o);
    }
  }
}

// Page i of `out` (BF16) = pool page ids[i], 9 CTAs of 256 threads per page, 16 bytes in / 32 out.
__global__ void __launch_bounds__(256) gather_pages_bf16_kernel(const uint8_t* __restrict__ pool, int64_t num_pages,
                                                                const int32_t* __restrict__ ids,
                                                                uint4* __restrict__ out) {
  constexpr int kChunks = kPage * kLatent / 16;     // 2304 chunks of 16 FP8 bytes per page
  const int64_t i = blockIdx.x / 9;
  const int c = (blockIdx.x % 9) * 256 + threadIdx.x;
  const int64_t page = ids[i];
  uint32_t o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (page >= 0 && page < num_pages) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(pool + page * (kPage * kLatent)) + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t two = (w[k] >> (16 * h)) & 0xFFFFu;
        uint32_t b = dev::fp8x2_to_bf16x2(two);
        if ((two & 0x7Fu) == 0x7Fu) b = (b & 0xFFFF0000u) | 0x7FC0u;          // NaN -> canonical BF16 NaN
        if ((two & 0x7F00u) == 0x7F00u) b = (b & 0x0000FFFFu) | 0x7FC00000u;
        o[2 * k + h] = b;
      }
    }
  }
  uint4* dst = out + (i * kChunks + c) * 2;
  __stcs(dst, make_uint4(o[0], o[1], o[2], o[3]));
  __stcs(dst + 1, make_uint4(o[4], o[5], o[6], o[7]));
}

}  // namespace

cudaError_t launch_gather_fp8(const GatherArgs& a, cudaStream_t s) {
  if (a.total_tokens == 0 || a.batch == 0) return cudaSuccess;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (a.total_tokens + kRowsPerPass * 8 - 1) / (kRowsPerPass * 8);   // passes of 64 rows
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * 8;      // 8 CTAs of 288 threads per SM
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (a.kv_dtype == KV_FP8) gather_fp8_kernel<KV_FP8><<<grid, kGatherThreads, 0, s>>>(a);
  else gather_fp8_kernel<KV_NVFP4><<<grid, kGatherThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gather_pages_bf16(const uint8_t* pool, int64_t num_pages, const int32_t* ids, int64_t n,
                                     void* out, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  gather_pages_bf16_kernel<<<static_cast<unsigned>(n * 9), 256, 0, s>>>(pool, num_pages, ids, reinterpret_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace qkvp
