// Log-sum-exp combine of split-KV partials.
//
// Each segment of a request that spans several segments left a normalised FP32 partial o_i and its
// base-2 log-sum-exp L_i. With M = max_i L_i and w_i = 2^(L_i - M):
//   out = g * sum_i w_i o_i / sum_i w_i,   lse = (M + log2 sum_i w_i) * ln 2.
// Requests with one segment were written by the decode kernel; requests with no tokens get zeros
// and lse = -inf.
//
// The kernel is a pure stream over the partials (each FP32 value read once) and the BF16 output. A
// thread owns 8 consecutive output dims and walks its segments in chunks of four: the chunk's L_i
// and both 16-byte halves of each o_i are loaded before any is used, and a running maximum
// rescales what was summed so far when a later chunk raises it, so the partials are read in one
// pass. One launch holds two kinds of 128-thread CTA:
//  - narrow: one (request, pair of heads), 64 threads per head; for requests with at most
//    kCombineWideSegs segments, i.e. at most two chunks per thread;
//  - wide: one (wide request, head, quarter of the 512 dims), 16 threads per segment group and 8
//    groups, group k taking chunks k, k + 8, ...; the groups' sums are merged in shared memory. A
//    request cut into ~150 segments (a long context alone on the GPU) then has ~5 chunks per thread
//    in turn instead of ~40.
#include <cstdint>

#include "qkvp_device.cuh"
#include "qkvp_internal.h"

namespace qkvp {
namespace {

constexpr int kThreads = 128;
constexpr int kDimsPerThread = 8;
constexpr int kChunk = 4;                               // segments loaded together
constexpr int kNarrowLanes = kDv / kDimsPerThread;      // 64 threads per head
constexpr int kNarrowHeads = kThreads / kNarrowLanes;   // 2 heads per narrow CTA
constexpr int kWideParts = 4;                           // a wide CTA covers 128 of the 512 dims
constexpr int kWideLanes = kDv / kWideParts / kDimsPerThread;  // 16 threads per group
constexpr int kWideGroups = kThreads / kWideLanes;             // 8 segment groups

// Running state of one thread: max m of the L_i seen, sum of 2^(L_i - m) and of 2^(L_i - m) o_i.
struct Run {
  float m = -INFINITY, wsum = 0.0f, acc[kDimsPerThread] = {};
};

// Merges segments i0 .. i0 + 3 (those below ns) of the request starting at segment s0 into s, for
// head h and output dims v .. v + 7.
__device__ __forceinline__ void merge_chunk(Run& s, const DecodeArgs& a, int s0, int i0, int ns, int h, int v) {
  float l[kChunk];
  float4 x[kChunk][2];
#pragma unroll
  for (int j = 0; j < kChunk; ++j) {
    l[j] = -INFINITY;
    x[j][0] = x[j][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (i0 + j < ns) {
      const int64_t p = static_cast<int64_t>(a.segs[s0 + i0 + j].partial) * a.heads + h;
      l[j] = a.part_lse[p];
      const float4* src = reinterpret_cast<const float4*>(a.part_o + p * kDv + v);
      x[j][0] = __ldcs(src);
      x[j][1] = __ldcs(src + 1);
    }
  }
  float mn = s.m;
#pragma unroll
  for (int j = 0; j < kChunk; ++j) mn = fmaxf(mn, l[j]);
  if (mn == -INFINITY) return;  // nothing with weight yet
  const float c = exp2f(s.m - mn);  // 0 when s.m is -inf
  s.wsum *= c;
#pragma unroll
  for (int d = 0; d < kDimsPerThread; ++d) s.acc[d] *= c;
  s.m = mn;
#pragma unroll
  for (int j = 0; j < kChunk; ++j) {
    const float w = exp2f(l[j] - mn);
    s.wsum += w;
    if (w > 0.0f) {  // a partial whose weight underflows contributes nothing
      s.acc[0] += w * x[j][0].x;
      s.acc[1] += w * x[j][0].y;
      s.acc[2] += w * x[j][0].z;
      s.acc[3] += w * x[j][0].w;
      s.acc[4] += w * x[j][1].x;
      s.acc[5] += w * x[j][1].y;
      s.acc[6] += w * x[j][1].z;
      s.acc[7] += w * x[j][1].w;
    }
  }
}

__device__ __forceinline__ void write_out(const Run& s, const DecodeArgs& a, int64_t row, int v, bool write_lse) {
  const float k = s.wsum > 0.0f ? a.out_scale / s.wsum : 0.0f;
  uint4 o;
  o.x = dev::pack_bf16x2(s.acc[0] * k, s.acc[1] * k);
  o.y = dev::pack_bf16x2(s.acc[2] * k, s.acc[3] * k);
  o.z = dev::pack_bf16x2(s.acc[4] * k, s.acc[5] * k);
  o.w = dev::pack_bf16x2(s.acc[6] * k, s.acc[7] * k);
  *reinterpret_cast<uint4*>(a.out + row * kDv + v) = o;
  if (a.lse && write_lse) a.lse[row] = s.wsum > 0.0f ? (s.m + log2f(s.wsum)) * 0.69314718055994531f : -INFINITY;
}

__global__ void __launch_bounds__(kThreads) combine_kernel(const DecodeArgs a, int narrow_ctas) {
  const int t = threadIdx.x;
  if (static_cast<int>(blockIdx.x) < narrow_ctas) {
    const int per_req = a.heads / kNarrowHeads;
    const int r = blockIdx.x / per_req;
    const int h = (blockIdx.x % per_req) * kNarrowHeads + t / kNarrowLanes;
    const int v = (t % kNarrowLanes) * kDimsPerThread;
    const int s0 = a.req_seg_ptr[r], ns = a.req_seg_ptr[r + 1] - s0;
    if (ns == 1 || ns > kCombineWideSegs) return;  // written by the decode kernel / by wide CTAs
    Run s;
    for (int i0 = 0; i0 < ns; i0 += kChunk) merge_chunk(s, a, s0, i0, ns, h, v);
    write_out(s, a, static_cast<int64_t>(r) * a.heads + h, v, v == 0);
    return;
  }
  const int b = blockIdx.x - narrow_ctas;
  const int per_req = a.heads * kWideParts;
  const int r = a.wide_req[b / per_req];
  const int h = (b % per_req) / kWideParts;
  const int grp = t / kWideLanes, lane = t % kWideLanes;
  const int v = (b % kWideParts) * (kDv / kWideParts) + lane * kDimsPerThread;
  const int s0 = a.req_seg_ptr[r], ns = a.req_seg_ptr[r + 1] - s0;
  if (ns == 1) return;  // the same for the whole CTA
  Run s;
  for (int i0 = grp * kChunk; i0 < ns; i0 += kWideGroups * kChunk) merge_chunk(s, a, s0, i0, ns, h, v);
  __shared__ float sm_m[kWideGroups], sm_w[kWideGroups];
  __shared__ float4 sm_acc[kWideGroups][kWideLanes][2];
  if (lane == 0) sm_m[grp] = s.m;
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kWideGroups; ++k) M = fmaxf(M, sm_m[k]);
  const float c = M == -INFINITY ? 0.0f : exp2f(s.m - M);
  if (lane == 0) sm_w[grp] = s.wsum * c;
  sm_acc[grp][lane][0] = make_float4(s.acc[0] * c, s.acc[1] * c, s.acc[2] * c, s.acc[3] * c);
  sm_acc[grp][lane][1] = make_float4(s.acc[4] * c, s.acc[5] * c, s.acc[6] * c, s.acc[7] * c);
  __syncthreads();
  if (grp != 0) return;
  Run f;
  f.m = M;
#pragma unroll
  for (int k = 0; k < kWideGroups; ++k) {
    f.wsum += sm_w[k];
    const float4 u = sm_acc[k][lane][0], w = sm_acc[k][lane][1];
    f.acc[0] += u.x;
    f.acc[1] += u.y;
    f.acc[2] += u.z;
    f.acc[3] += u.w;
    f.acc[4] += w.x;
    f.acc[5] += w.y;
    f.acc[6] += w.z;
    f.acc[7] += w.w;
  }
  write_out(f, a, static_cast<int64_t>(r) * a.heads + h, v, v == 0);
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, int num_wide, cudaStream_t s) {
  if (a.batch == 0) return cudaSuccess;
  const int64_t narrow = static_cast<int64_t>(a.batch) * (a.heads / kNarrowHeads);
  const int64_t ctas = narrow + static_cast<int64_t>(num_wide) * a.heads * kWideParts;
  if (ctas > INT32_MAX) return cudaErrorInvalidValue;
  combine_kernel<<<static_cast<unsigned>(ctas), kThreads, 0, s>>>(a, static_cast<int>(narrow));
  return cudaGetLastError();
}

}  // namespace qkvp
