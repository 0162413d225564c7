// Log-sum-exp combine of split-KV partials.
//
// Each segment of a request that spans several segments left a normalised FP32 partial o_i and its
// base-2 log-sum-exp L_i. With M = max_i L_i and w_i = 2^(L_i - M):
//   out = g * sum_i w_i o_i / sum_i w_i,   lse = (M + log2 sum_i w_i) * ln 2.
// Requests with one segment were written by the decode kernel; requests with no tokens get zeros
// and lse = -inf. One CTA per (request, head, quarter of the 512 output dims).
#include <cstdint>

#include "qkvp_device.cuh"
#include "qkvp_internal.h"

namespace qkvp {
namespace {

__global__ void __launch_bounds__(128) combine_kernel(const DecodeArgs a) {
  const int r = blockIdx.x, h = blockIdx.y, quarter = blockIdx.z;
  const int s0 = a.req_seg_ptr[r], ns = a.req_seg_ptr[r + 1] - s0;
  if (ns == 1) return;
  const int v = quarter * 128 + threadIdx.x;
  const int64_t orow = (static_cast<int64_t>(r) * a.heads + h) * kDv;
  if (ns == 0) {
    a.out[orow + v] = 0;
    if (a.lse && quarter == 0 && threadIdx.x == 0) a.lse[static_cast<int64_t>(r) * a.heads + h] = -INFINITY;
    return;
  }
  float M = -INFINITY;
  for (int i = 0; i < ns; ++i) M = fmaxf(M, a.part_lse[static_cast<int64_t>(a.segs[s0 + i].partial) * a.heads + h]);
  float wsum = 0.0f, acc = 0.0f;
  if (M != -INFINITY) {
    for (int i = 0; i < ns; ++i) {
      const int64_t p = a.segs[s0 + i].partial;
      const float w = exp2f(a.part_lse[p * a.heads + h] - M);
      wsum += w;
      if (w > 0.0f) acc += w * a.part_o[(p * a.heads + h) * kDv + v];
    }
  }
  const float o = wsum > 0.0f ? acc / wsum * a.out_scale : 0.0f;
  a.out[orow + v] = static_cast<uint16_t>(dev::pack_bf16x2(o, 0.0f) & 0xFFFFu);
  if (a.lse && quarter == 0 && threadIdx.x == 0)
    a.lse[static_cast<int64_t>(r) * a.heads + h] = wsum > 0.0f ? (M + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s) {
  if (a.batch == 0) return cudaSuccess;
  combine_kernel<<<dim3(a.batch, a.heads, kDv / 128), 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace qkvp
