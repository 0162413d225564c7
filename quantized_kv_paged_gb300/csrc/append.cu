// Quantize-on-append (FP8 E4M3 and NVFP4 pools), the device rounding check and the pool cast.
//
// NVFP4 block quantisation follows "SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "NVFP4
// format: two-level scaling" (E2M1 values, an E4M3 scale per 16 values, an FP32 global scale)
// and section "SGLang implementation", items 1-2 (quantize FP8 KV into NVFP4 on write). The
// pages give no arithmetic for the block scale; the one used here, and by the CPU oracle, is:
// amax / (6 g) rounded to nearest-even E4M3, element codes E2M1(x / (scale * g)).
//
// The per-token-scaled FP8 pool carries the pages' indexer key layout ("The Precision Frontier:
// Implementing bf16 Index Keys", section "The Message: Planning the bf16-K Implementation": FP8
// elements + 4 scale bytes per token, 64-token pages) for the latent: one FP32 scale per token,
// amax / 448, and codes E4M3(x / scale).
//
// One thread quantises one block of 16 consecutive latent elements of one token (36 blocks per
// token; one warp per token for the per-token-scaled pool, whose scale needs the whole token); the
// append of a decode step touches a handful of tokens, a bulk fill touches millions, and both are
// bound by reading the source.
#include <cstdint>

#include "qkvp_device.cuh"
#include "qkvp_internal.h"

namespace qkvp {
namespace {

constexpr int kBlocks = kLatent / 16;   // 36 blocks of 16 elements per token

__device__ __forceinline__ void load16(const void* src, int src_dtype, int64_t tok, int blk, float (&x)[16]) {
  if (src_dtype == SRC_FP8) {
    const uint4 v = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(src) + tok * kLatent + blk * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j) x[4 * i + j] = dev::e4m3_to_float((w[i] >> (8 * j)) & 0xFFu);
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + tok * kLatent + blk * 16);
    const uint4 a = p[0], b = p[1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

__global__ void append_fp8_kernel(const void* __restrict__ src, int src_dtype, int64_t n,
                                  const int64_t* __restrict__ slots, uint8_t* __restrict__ pool,
                                  int64_t num_slots) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= n * kBlocks) return;
  const int64_t tok = gid / kBlocks;
  const int blk = static_cast<int>(gid % kBlocks);
  const int64_t slot = slots[tok];
  if (slot < 0 || slot >= num_slots) return;
  uint8_t* dst = pool + slot * kLatent + blk * 16;
  if (src_dtype == SRC_FP8) {
    *reinterpret_cast<uint4*>(dst) =
        *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(src) + tok * kLatent + blk * 16);
    return;
  }
  float x[16];
  load16(src, src_dtype, tok, blk, x);
  uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i / 4] |= dev::encode_e4m3(x[i]) << (8 * (i % 4));
  *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void append_nvfp4_kernel(const void* __restrict__ src, int src_dtype, int64_t n,
                                    const int64_t* __restrict__ slots, uint8_t* __restrict__ data,
                                    uint8_t* __restrict__ scale, float g, int64_t num_slots) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= n * kBlocks) return;
  const int64_t tok = gid / kBlocks;
  const int blk = static_cast<int>(gid % kBlocks);
  const int64_t slot = slots[tok];
  if (slot < 0 || slot >= num_slots) return;
  float x[16];
  load16(src, src_dtype, tok, blk, x);
  // amax over the block; any NaN makes it NaN
  float amax = 0.0f;
  bool nan = false;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    nan |= (x[i] != x[i]);
    amax = fmaxf(amax, fabsf(x[i]));
  }
  if (nan) amax = __uint_as_float(0x7FC00000u);
  const float s = __fdiv_rn(amax, __fmul_rn(6.0f, g));
  const uint32_t s8 = dev::encode_e4m3(s);
  const float sd = __fmul_rn(dev::e4m3_to_float(s8), g);
  uint32_t w[2] = {0, 0};
  if (sd != 0.0f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t c = dev::encode_e2m1(__fdiv_rn(x[i], sd));
      w[i / 8] |= c << (4 * (i % 8));     // element 2k -> low nibble of byte k
    }
  }
  *reinterpret_cast<uint2*>(data + slot * kPacked + blk * 8) = make_uint2(w[0], w[1]);
  scale[slot * kScales + blk] = static_cast<uint8_t>(s8);
}

__global__ void append_fp8pt_kernel(const void* __restrict__ src, int src_dtype, int64_t n,
                                    const int64_t* __restrict__ slots, uint8_t* __restrict__ pool,
                                    int64_t num_slots) {
  const int64_t tok = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (tok >= n) return;                       // tok and slot are the same for the whole warp
  const int64_t slot = slots[tok];
  if (slot < 0 || slot >= num_slots) return;
  constexpr int kExtra = kBlocks - 32;        // lanes 0..3 hold a second block (blocks 32..35)
  float x0[16], x1[16];
  load16(src, src_dtype, tok, lane, x0);
  if (lane < kExtra) load16(src, src_dtype, tok, 32 + lane, x1);
  float amax = 0.0f;
  bool nan = false;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    nan |= (x0[i] != x0[i]);
    amax = fmaxf(amax, fabsf(x0[i]));
    if (lane < kExtra) {
      nan |= (x1[i] != x1[i]);
      amax = fmaxf(amax, fabsf(x1[i]));
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // a token holding a NaN gets the scale 0x7FC00000 (one fixed NaN pattern for the stored bytes)
  const bool any_nan = __any_sync(0xffffffffu, nan);
  const float sc = any_nan ? __uint_as_float(0x7FC00000u) : __fdiv_rn(amax, 448.0f);
  uint8_t* page = pool + (slot / kPage) * kPtPageBytes;
  uint8_t* row = page + (slot % kPage) * kLatent;
  auto encode16 = [&](const float (&x)[16], int blk) {
    uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i / 4] |= dev::encode_e4m3(sc == 0.0f ? x[i] : __fdiv_rn(x[i], sc)) << (8 * (i % 4));
    *reinterpret_cast<uint4*>(row + blk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  };
  encode16(x0, lane);
  if (lane < kExtra) encode16(x1, 32 + lane);
  if (lane == 0) *reinterpret_cast<float*>(page + kPtScaleOff + (slot % kPage) * 4) = sc;
}

__global__ void encode_kernel(const float* __restrict__ x, int64_t n, int fmt, uint8_t* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float v = x[i];
    out[i] = static_cast<uint8_t>(fmt == 1 ? dev::encode_e4m3(v) : dev::encode_e2m1(v));
  }
}

// Pool-wide FP8 -> BF16 cast (the baseline the pages trace): one 16-byte chunk in and 32 bytes out
// per thread, one chunk per thread and a grid over the whole pool, streaming loads and stores. A
// grid-stride loop over 8 CTAs per SM (one chunk in flight per thread) reached only 68 % of the
// measured copy bandwidth; with every chunk its own thread the loads of many CTAs per SM are in
// flight together, as in the gather-then-cast kernel on the same byte pattern.
__global__ void __launch_bounds__(256) cast_kernel(const uint4* __restrict__ in, int64_t n16, uint4* __restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const uint4 v = __ldcs(in + i);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t two = (w[k] >> (16 * h)) & 0xFFFFu;
      uint32_t b = dev::fp8x2_to_bf16x2(two);
      if ((two & 0x7Fu) == 0x7Fu) b = (b & 0xFFFF0000u) | 0x7FC0u;            // NaN -> canonical BF16 NaN
      if ((two & 0x7F00u) == 0x7F00u) b = (b & 0x0000FFFFu) | 0x7FC00000u;
      o[2 * k + h] = b;
    }
  }
  __stcs(out + 2 * i, make_uint4(o[0], o[1], o[2], o[3]));
  __stcs(out + 2 * i + 1, make_uint4(o[4], o[5], o[6], o[7]));
}

}  // namespace

cudaError_t launch_append(const void* src, int src_dtype, int64_t n, const int64_t* slots,
                          void* kv_data, uint8_t* kv_scale, int kv_dtype, float g,
                          int64_t num_slots, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (n * kBlocks + threads - 1) / threads;
  if (kv_dtype == KV_FP8) {
    append_fp8_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
        src, src_dtype, n, slots, static_cast<uint8_t*>(kv_data), num_slots);
  } else if (kv_dtype == KV_FP8PT) {
    append_fp8pt_kernel<<<static_cast<unsigned>((n + threads / 32 - 1) / (threads / 32)), threads, 0, s>>>(
        src, src_dtype, n, slots, static_cast<uint8_t*>(kv_data), num_slots);
  } else {
    append_nvfp4_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
        src, src_dtype, n, slots, static_cast<uint8_t*>(kv_data), kv_scale, g, num_slots);
  }
  return cudaGetLastError();
}

cudaError_t launch_encode(const float* x, int64_t n, int fmt, uint8_t* codes, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int64_t want = (n + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(want < 152 * 64 ? want : 152 * 64);
  encode_kernel<<<blocks, 256, 0, s>>>(x, n, fmt, codes);
  return cudaGetLastError();
}

cudaError_t launch_cast(const uint8_t* in, int64_t n, uint16_t* out, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int64_t n16 = n / 16;
  const int64_t blocks = (n16 + 255) / 256;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  cast_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(reinterpret_cast<const uint4*>(in), n16,
                                                            reinterpret_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace qkvp
